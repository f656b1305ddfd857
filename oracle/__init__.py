"""fp64 CPU oracle for exact attention and Flash-Decoding.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The product path
(``exact_attention_29_gb300`` and its CUDA library) never imports it, and the
two share no code: this package does its arithmetic in plain C
(``attention.c``, fp64, S and P materialised) and in plain Python
(``combine.py``, the (m, l, o) summaries and their combine operator).

Public functions
----------------
attention(q, k, v, causal, scale)            -> (o, lse), [B,H,N,d] inputs
attention_rows(q_rows, q_pos, k, v, ...)     -> (o, lse, s, p) for one head
decode(q, k_cache, v_cache, seqlens)         -> (o, lse), one query per (b, h)
attention_bwd(q, k, v, dout, causal, scale)  -> (dq, dk, dv), [B,H,N,d] inputs
set_threads(n)                               -> OpenMP thread count (timing only)

Inputs may be numpy arrays or torch CPU tensors of any float dtype; they are
widened to fp64 exactly (bf16 and fp32 values are representable in fp64), so
the oracle sees the very values handed to the GPU.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, invariants, a 50-digit brute force and page-printed numbers).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_SRC = os.path.join(_HERE, "attention.c")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``attention.c`` into ``liboracle.so`` with gcc (OpenMP, no fast-math).

    ``-ffp-contract=off`` keeps the arithmetic identical on x86_64 and aarch64.
    """
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-std=c11",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int)
            lib.oracle_attention_rows.argtypes = [dp, ip, dp, dp, ctypes.c_int, ctypes.c_int,
                                                  ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                                  dp, dp, dp, dp]
            lib.oracle_attention_rows.restype = ctypes.c_int
            lib.oracle_attention.argtypes = [dp, dp, dp, dp, dp] + [ctypes.c_int] * 5 + [ctypes.c_double]
            lib.oracle_attention.restype = ctypes.c_int
            lib.oracle_decode.argtypes = [dp, dp, dp, ip, dp, dp] + [ctypes.c_int] * 4
            lib.oracle_decode.restype = ctypes.c_int
            lib.oracle_attention_block_mask.argtypes = [dp, dp, dp, ctypes.POINTER(ctypes.c_ubyte), ctypes.c_int,
                                                         ctypes.c_int, dp, dp] + [ctypes.c_int] * 5 + [ctypes.c_double]
            lib.oracle_attention_block_mask.restype = ctypes.c_int
            lib.oracle_decode_gqa.argtypes = [dp, dp, dp, ip, dp, dp] + [ctypes.c_int] * 5
            lib.oracle_decode_gqa.restype = ctypes.c_int
            lib.oracle_attention_bwd.argtypes = [dp] * 7 + [ctypes.c_int] * 5 + [ctypes.c_double]
            lib.oracle_attention_bwd.restype = ctypes.c_int
            lib.oracle_set_threads.argtypes = [ctypes.c_int]
            lib.oracle_set_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def set_threads(n: int) -> int:
    """Thread count of the oracle's OpenMP loops for later calls from this
    thread (timing only: results do not depend on it); returns the count in
    effect. set_threads(0) leaves it unchanged and only reports it."""
    return _load().oracle_set_threads(int(n))


def _f64(x) -> np.ndarray:
    """Widen to a C-contiguous fp64 numpy array (torch tensors are converted on the CPU)."""
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu")
        import torch

        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray, ctype=ctypes.c_double):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def attention_rows(q_rows, q_pos, k, v, causal: bool, scale: float, want_sp: bool = False):
    """Standard attention for one head and a list of query rows.

    q_rows [n, d]; q_pos [n] int (positions, needed when causal); k, v [N, d].
    Returns (o [n, d], lse [n], s [n, N] or None, p [n, N] or None), where s is
    the scaled and masked score matrix and p the softmax probabilities.
    """
    lib = _load()
    q = _f64(q_rows)
    kk = _f64(k)
    vv = _f64(v)
    n, d = q.shape
    nk = kk.shape[0]
    if kk.shape != (nk, d) or vv.shape != (nk, d):
        raise ValueError("k and v must be [N, d] with the same d as q")
    pos = None
    if q_pos is not None:
        pos = np.ascontiguousarray(np.asarray(q_pos, dtype=np.int32))
        if pos.shape != (n,):
            raise ValueError("q_pos must have one entry per query row")
    elif causal:
        raise ValueError("causal attention needs query positions")
    o = np.empty((n, d), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    s = np.empty((n, nk), dtype=np.float64) if want_sp else None
    p = np.empty((n, nk), dtype=np.float64) if want_sp else None
    rc = lib.oracle_attention_rows(
        _ptr(q), _ptr(pos, ctypes.c_int) if pos is not None else None, _ptr(kk), _ptr(vv),
        n, nk, d, int(bool(causal)), float(scale), _ptr(o), _ptr(lse),
        _ptr(s) if s is not None else None, _ptr(p) if p is not None else None)
    _check(rc, "attention_rows")
    return o, lse, s, p


def attention(q, k, v, causal: bool, scale: float):
    """Standard attention over [B, H, N, d] tensors. Returns (o [B,H,N,d], lse [B,H,N])."""
    lib = _load()
    qq, kk, vv = _f64(q), _f64(k), _f64(v)
    if qq.ndim != 4 or qq.shape != kk.shape or qq.shape != vv.shape:
        raise ValueError("q, k, v must all be [B, H, N, d]")
    B, H, N, d = qq.shape
    o = np.empty_like(qq)
    lse = np.empty((B, H, N), dtype=np.float64)
    rc = lib.oracle_attention(_ptr(qq), _ptr(kk), _ptr(vv), _ptr(o), _ptr(lse),
                              B, H, N, d, int(bool(causal)), float(scale))
    _check(rc, "attention")
    return o, lse


def decode(q, k_cache, v_cache, seqlens):
    """One query token per (b, h) against the first seqlens[b] cache entries.

    q [B,H,d]; k_cache, v_cache [B,H,L,d]; seqlens [B]. Scale is 1/sqrt(d).
    Returns (o [B,H,d], lse [B,H]).
    """
    lib = _load()
    qq, kk, vv = _f64(q), _f64(k_cache), _f64(v_cache)
    B, H, L, d = kk.shape
    if qq.shape != (B, H, d) or vv.shape != kk.shape:
        raise ValueError("q must be [B,H,d] and the caches [B,H,L,d]")
    if hasattr(seqlens, "detach"):
        seqlens = seqlens.detach().cpu().numpy()
    sl = np.ascontiguousarray(np.asarray(seqlens, dtype=np.int32))
    o = np.empty((B, H, d), dtype=np.float64)
    lse = np.empty((B, H), dtype=np.float64)
    rc = lib.oracle_decode(_ptr(qq), _ptr(kk), _ptr(vv), _ptr(sl, ctypes.c_int), _ptr(o), _ptr(lse),
                           B, H, L, d)
    _check(rc, "decode")
    return o, lse


def attention_block_mask(q, k, v, mask, causal: bool, scale: float, block: int = 128):
    """Attention of [B, H, N, d] tensors under a block mask [T, T] or
    [H, T, T] (T = ceil(N / block)); returns (o, lse) as fp64 arrays."""
    lib = _load()
    qq, kk, vv = _f64(q), _f64(k), _f64(v)
    B, H, N, d = qq.shape
    if hasattr(mask, "detach"):
        mask = mask.detach().cpu().numpy()
    mk = np.ascontiguousarray(np.asarray(mask) != 0, dtype=np.uint8)
    T = (N + block - 1) // block
    if mk.ndim == 2:
        mk = mk[None]
    if mk.shape[1:] != (T, T) or mk.shape[0] not in (1, H):
        raise ValueError("mask must be [T, T] or [H, T, T]")
    o = np.empty((B, H, N, d), dtype=np.float64)
    lse = np.empty((B, H, N), dtype=np.float64)
    rc = lib.oracle_attention_block_mask(_ptr(qq), _ptr(kk), _ptr(vv), mk.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte)),
                                         mk.shape[0], block, _ptr(o), _ptr(lse), B, H, N, d, int(bool(causal)),
                                         float(scale))
    _check(rc, "attention_block_mask")
    return o, lse


def decode_gqa(q, k_cache, v_cache, seqlens):
    """Decode with grouped K/V heads: q [B,Hq,d], caches [B,Hkv,L,d], Hq a
    multiple of Hkv; query head h uses K/V head h // (Hq // Hkv).

    Returns (o [B,Hq,d], lse [B,Hq]).
    """
    lib = _load()
    qq, kk, vv = _f64(q), _f64(k_cache), _f64(v_cache)
    B, Hkv, L, d = kk.shape
    if qq.ndim != 3 or qq.shape[0] != B or qq.shape[2] != d or vv.shape != kk.shape:
        raise ValueError("q must be [B,Hq,d] and the caches [B,Hkv,L,d]")
    Hq = qq.shape[1]
    if hasattr(seqlens, "detach"):
        seqlens = seqlens.detach().cpu().numpy()
    sl = np.ascontiguousarray(np.asarray(seqlens, dtype=np.int32))
    o = np.empty((B, Hq, d), dtype=np.float64)
    lse = np.empty((B, Hq), dtype=np.float64)
    rc = lib.oracle_decode_gqa(_ptr(qq), _ptr(kk), _ptr(vv), _ptr(sl, ctypes.c_int), _ptr(o), _ptr(lse),
                               B, Hq, Hkv, L, d)
    _check(rc, "decode_gqa")
    return o, lse


def attention_bwd(q, k, v, dout, causal: bool, scale: float):
    """Backward of standard attention over [B, H, N, d] tensors.

    Returns (dq, dk, dv) for the upstream gradient dout of O, as fp64 arrays.
    """
    lib = _load()
    qq, kk, vv, gg = _f64(q), _f64(k), _f64(v), _f64(dout)
    if qq.ndim != 4 or not (qq.shape == kk.shape == vv.shape == gg.shape):
        raise ValueError("q, k, v, dout must all be [B, H, N, d]")
    B, H, N, d = qq.shape
    dq, dk, dv = np.empty_like(qq), np.empty_like(qq), np.empty_like(qq)
    rc = lib.oracle_attention_bwd(_ptr(qq), _ptr(kk), _ptr(vv), _ptr(gg), _ptr(dq), _ptr(dk), _ptr(dv),
                                  B, H, N, d, int(bool(causal)), float(scale))
    _check(rc, "attention_bwd")
    return dq, dk, dv
