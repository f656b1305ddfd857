"""FP8 (e4m3) block quantization with incoherent processing, in plain numpy fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources: "已有的几种大模型上下文支持情况" (cicada blog) §4.4 (FA-3's FP8 path):
  - §4.4.1 block-wise quantization: each tile that enters a tensor-core product
    carries its own scale factor instead of one scale per matrix;
  - §4.4.2 incoherent processing: Q and K are multiplied by a random orthogonal
    matrix R, a Hadamard matrix with random signs, before quantization; the
    scores do not change, S = (QR)(KR)^T = Q R R^T K^T = Q K^T, while outliers
    of single feature dimensions are spread over all of them.

The e4m3 format (the "fn" variant without infinities: 1 sign bit, 4 exponent
bits with bias 7, 3 mantissa bits; largest finite value 448, smallest normal
2^-6, subnormals k * 2^-9) is rounded to nearest, ties to even, with values
beyond 448 saturated to 448 (the kernels convert with saturation as well).

Readings (the page leaves them open):
  - R = diag(signs) H_d / sqrt(d) with H_d the Sylvester-Hadamard matrix; a row
    x is rotated as x R. V is not rotated (it does not enter the scores).
  - A tile is 128 consecutive rows of one (batch, head); its scale is
    amax / 448 over the tile's rotated values (1 for an all-zero tile), so the
    largest magnitude maps to 448.
  - V takes one scale per (batch, head): the output accumulates over all V
    tiles in one fp32 accumulator, and per-tile V scales would not factor out.
"""
from __future__ import annotations

import math

import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_NORMAL_EXP = -6
E4M3_MANTISSA_BITS = 3
TILE_ROWS = 128


def e4m3_round(x):
    """Nearest e4m3 value (ties to even), saturating at +-448. Returns fp64."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    out = np.zeros_like(a)
    nz = a > 0
    # exponent of the binade; below the smallest normal the spacing is fixed
    e = np.floor(np.log2(np.where(nz, a, 1.0)))
    e = np.maximum(e, E4M3_MIN_NORMAL_EXP)
    quantum = np.exp2(e - E4M3_MANTISSA_BITS)
    q = a / quantum
    # round half to even: np.rint rounds halves to even
    r = np.rint(q) * quantum
    # log2 of a value just below a power of two can land in the binade above;
    # either way r is the nearest representable value of that binade grid
    out[nz] = r[nz]
    out = np.minimum(out, E4M3_MAX)
    return np.copysign(out, x)


def e4m3_encode(v):
    """Bit codes (uint8) of values already on the e4m3 grid."""
    v = np.asarray(v, dtype=np.float64)
    sign = (np.signbit(v)).astype(np.uint8) << 7
    a = np.abs(v)
    code = np.zeros(a.shape, dtype=np.uint8)
    sub = (a > 0) & (a < 2.0 ** E4M3_MIN_NORMAL_EXP)
    code[sub] = np.round(a[sub] / 2.0 ** -9).astype(np.uint8)
    nrm = a >= 2.0 ** E4M3_MIN_NORMAL_EXP
    e = np.floor(np.log2(np.where(nrm, a, 1.0))).astype(np.int64)
    m = np.round((a / np.exp2(e) - 1.0) * 8).astype(np.int64)
    code[nrm] = (((e[nrm] + 7) << 3) | m[nrm]).astype(np.uint8)
    return code | sign


def e4m3_decode(code):
    """Values of e4m3 codes (uint8), fp64; 0x7f / 0xff decode to NaN."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7))
    val = np.where((c & 0x7F) == 0x7F, np.nan, val)
    return s * val


def hadamard(d: int, signs=None):
    """R = diag(signs) H_d / sqrt(d), H_d by Sylvester's construction (d a power of 2)."""
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    r = h / math.sqrt(d)
    if signs is not None:
        r = np.asarray(signs, dtype=np.float64).reshape(d, 1) * r
    return r


def quantize(x, signs=None, per_head: bool = False, transpose: bool = False):
    """Block-quantize x [B, H, N, d] to e4m3.

    signs: length-d +-1 vector for the incoherent rotation x -> x R (None: no
    rotation). per_head: one scale per (b, h) instead of one per 128-row tile.
    transpose: return codes as [B, H, d, N] (the layout of V^T).
    Returns (codes uint8, scales fp64 [B, H, T] or [B, H]).
    """
    x = np.asarray(x, dtype=np.float64)
    B, H, N, d = x.shape
    y = x @ hadamard(d, signs) if signs is not None else x.copy()
    T = (N + TILE_ROWS - 1) // TILE_ROWS
    if per_head:
        amax = np.abs(y).reshape(B, H, -1).max(axis=2)
        scales = np.where(amax > 0, amax / E4M3_MAX, 1.0)
        q = e4m3_round(y / scales[:, :, None, None])
    else:
        scales = np.ones((B, H, T))
        q = np.empty_like(y)
        for t in range(T):
            blk = y[:, :, t * TILE_ROWS:(t + 1) * TILE_ROWS]
            amax = np.abs(blk).reshape(B, H, -1).max(axis=2)
            s = np.where(amax > 0, amax / E4M3_MAX, 1.0)
            scales[:, :, t] = s
            q[:, :, t * TILE_ROWS:(t + 1) * TILE_ROWS] = e4m3_round(blk / s[:, :, None, None])
    codes = e4m3_encode(q)
    if transpose:
        codes = np.ascontiguousarray(np.swapaxes(codes, 2, 3))
    return codes, scales


def dequantize(codes, scales, transpose: bool = False):
    """Inverse of quantize (without undoing the rotation): fp64 [B, H, N, d]."""
    v = e4m3_decode(codes)
    if transpose:
        v = np.swapaxes(v, 2, 3)
    B, H, N, d = v.shape
    scales = np.asarray(scales, dtype=np.float64)
    if scales.ndim == 2:
        return v * scales[:, :, None, None]
    per_row = np.repeat(scales, TILE_ROWS, axis=2)[:, :, :N]
    return v * per_row[:, :, :, None]
