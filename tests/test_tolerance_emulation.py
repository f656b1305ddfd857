"""Where the GPU tolerances come from.

The bf16 forward, the e4m3 forward and the backward round intermediates that
the fp64 oracle keeps exact. These CPU tests redo the kernels' roundings (and
only those) on the GPU tests' own inputs, in numpy next to the oracle, and
check that the bounds the GPU tests use leave the margin their docstrings state
over the error those roundings alone produce. Nothing here runs the CUDA path.

bf16 forward (cicada blog §5 and CMU 15-779 Lecture 5 notes §5.1): S in fp32,
the stale running maximum of the conditional rescale (threshold 8 in log2
units), P = 2^(x - m) in fp32 with l summing the fp32 values, P rounded to
bf16 for the P V product, O rounded to bf16 at the end.

e4m3 forward ("已有的几种大模型上下文支持情况" §4.4, FA-3's FP8 path): S from
the e4m3 codes, keys in 128-key tiles with the kernel's stale running maximum
(rescale only when a tile's maximum exceeds it by more than 8 in log2 units,
the cicada blog §5 rule), P = 2^(x - m) in fp32 with l summing the fp32
values, P rounded to e4m3 for the P V product, O rounded to bf16 at the end.

Backward (CMU 15-779 Lecture 5 notes §7.2-7.4): P recomputed from the LSE in
fp32 and rounded to bf16, that bf16 P both in the dV product and in
dS = P (dP - D); D = rowsum(dO * O) from the bf16 O, dS rounded to bf16 before
its products, fp32 accumulation, every gradient rounded to bf16.
"""
import numpy as np
import pytest

import oracle
from oracle import fp8 as ofp8
from exact_attention_29_gb300 import workloads as wl
from parity import GRAD_ATOL, GRAD_MAX_REL, GRAD_MEAN_REL, MAX_ABS_LSE, MAX_ABS_O, MEAN_ABS_O
from test_gpu_fp8 import FP8_MAX_ABS_LSE, FP8_MAX_ABS_O, FP8_MEAN_ABS_O, _oracle_inputs, _signs

LOG2E = 1.4426950408889634
LN2 = 0.6931471805599453


def bf16(x):
    """Round to the nearest bf16 (ties to even), returned as fp64."""
    b = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    return r.view(np.float32).astype(np.float64)


def _bf16_forward_emulated(q, k, v, causal, scale, round_p=True):
    """One head, fp64 [N, d] inputs (bf16 values): the kernel's roundings
    (round_p=False keeps P in fp32, to show what its rounding adds)."""
    N = q.shape[0]
    s_all = (q @ k.T).astype(np.float32)
    sl2 = np.float32(scale * LOG2E)
    o = np.zeros_like(q)
    lse = np.zeros(N)
    for i in range(N):
        vis = i + 1 if causal else N
        m_used, l, acc = -np.inf, np.float32(0.0), np.zeros(q.shape[1])
        for j0 in range(0, vis, 128):
            s = s_all[i, j0:min(j0 + 128, vis)]
            m_tile = float(np.float32(s.max()) * sl2)  # the maximum of the raw scores, then scaled
            if m_used != -np.inf and m_tile > m_used + 8.0:
                alpha = np.float32(2.0 ** (m_used - m_tile))
                l, acc, m_used = np.float32(l * alpha), acc * float(alpha), m_tile
            if m_used == -np.inf:
                m_used = m_tile
            p = np.exp2((s * sl2 - np.float32(m_used)).astype(np.float32), dtype=np.float32)
            l = np.float32(l + p.sum(dtype=np.float32))
            acc += (bf16(p) if round_p else p.astype(np.float64)) @ v[j0:j0 + p.size]
        o[i] = acc / float(l)
        lse[i] = (m_used + np.log2(float(l))) * LN2
    return bf16(o), lse


def test_bf16_forward_bounds_cover_the_roundings():
    """The forward tests' shapes and criterion (max and mean of |dO| over the
    whole output, max |dLSE|): the bounds over the rounding-only error. Measured
    here: max |dO| up to 8.5e-3 (d = 64, 128 keys, causal) and mean |dO| up to
    7.3e-4 (7 keys per row), so the max bound is 2.35x and the mean bound 2.74x
    the rounding-only error at their worst; the LSE sums fp32 values and its
    error stays near 3e-7, thousands of times below its bound. The maximum is
    set mostly by the bf16 rounding of O itself (7.8e-3 with P in fp32: half a
    bf16 step at |o| in [4, 8)); rounding P raises the mean by about a sixth."""
    worst_max = worst_mean = worst_lse = worst_mean_fp32_p = 0.0
    for d in (64, 128):
        for N in (1, 7, 128, 129, 300, 1000):
            for causal in (False, True):
                B, H = (2, 2) if N <= 300 else (1, 2)
                q, k, v = wl.prefill_inputs(B, H, N, d, seed=N + d)
                o_ref, lse_ref = oracle.attention(q, k, v, causal, d ** -0.5)
                qq, kk, vv = (t.double().numpy() for t in (q, k, v))
                o, lse = np.zeros_like(o_ref), np.zeros_like(lse_ref)
                o32 = np.zeros_like(o_ref)
                for b in range(B):
                    for h in range(H):
                        o[b, h], lse[b, h] = _bf16_forward_emulated(qq[b, h], kk[b, h], vv[b, h], causal, d ** -0.5)
                        o32[b, h] = _bf16_forward_emulated(qq[b, h], kk[b, h], vv[b, h], causal, d ** -0.5,
                                                           round_p=False)[0]
                worst_mean_fp32_p = max(worst_mean_fp32_p, np.abs(o32 - o_ref).mean())
                do = np.abs(o - o_ref)
                worst_max = max(worst_max, do.max())
                worst_mean = max(worst_mean, do.mean())
                worst_lse = max(worst_lse, np.abs(lse - lse_ref).max())
    assert MAX_ABS_O / worst_max >= 2.2, worst_max
    assert MEAN_ABS_O / worst_mean >= 2.5, worst_mean
    assert MAX_ABS_LSE / worst_lse >= 100, worst_lse
    # the emulation rounds P: its bf16 rounding adds to the error of the bf16 output alone
    assert worst_mean > 1.1 * worst_mean_fp32_p, (worst_mean, worst_mean_fp32_p)


def _fp8_forward_emulated(qd, kd, vd, causal, scale):
    """One head: qd, kd, vd fp64 [N, d] (the dequantized e4m3 inputs)."""
    N = qd.shape[0]
    x_all = (qd @ kd.T) * (scale * LOG2E)  # log2 units
    o = np.zeros_like(qd)
    lse = np.zeros(N)
    for i in range(N):
        vis = i + 1 if causal else N
        m_used, l, acc = -np.inf, np.float32(0.0), np.zeros(qd.shape[1])
        for j0 in range(0, vis, 128):
            x = x_all[i, j0:min(j0 + 128, vis)].astype(np.float32)
            m_tile = float(x.max())
            if m_used != -np.inf and m_tile > m_used + 8.0:
                alpha = np.float32(2.0 ** (m_used - m_tile))
                l, acc, m_used = np.float32(l * alpha), acc * float(alpha), m_tile
            if m_used == -np.inf:
                m_used = m_tile
            p = np.exp2(x - np.float32(m_used), dtype=np.float32)
            l = np.float32(l + p.sum(dtype=np.float32))
            acc += ofp8.e4m3_round(p.astype(np.float64)) @ vd[j0:j0 + p.size]
        o[i] = acc / float(l)
        lse[i] = (m_used + np.log2(float(l))) * LN2
    return bf16(o), lse


def test_fp8_forward_bounds_cover_the_e4m3_rounding_of_p():
    """Per case (the GPU test's shapes and criterion: max and mean of |dO| over
    the whole output): the bounds over the rounding-only error. Measured here:
    max |dO| 4.8e-2 (128 keys, causal: short rows) and mean |dO| 6.2e-3 (7 keys
    per row: few keys average the rounding); so the max bound is 3.1x and the
    mean bound 1.3x the rounding-only error at their worst, and 2.2x or more on
    the mean of every case with 128 keys or more."""
    margins_max, margins_mean, worst_lse, worst_max = [], {}, 0.0, 0.0
    for N in (1, 7, 128, 129, 300, 1000):
        for causal in (False, True):
            q, k, v = wl.prefill_inputs(2, 2, N, 128, seed=N + 3)
            qi, ki, vi = _oracle_inputs(q, k, v, _signs(N))
            qd, kd = ofp8.dequantize(*qi), ofp8.dequantize(*ki)
            vd = ofp8.dequantize(*vi, transpose=True)
            o_ref, lse_ref = oracle.attention(qd, kd, vd, causal, 128 ** -0.5)
            o, lse = np.zeros_like(o_ref), np.zeros_like(lse_ref)
            for b in range(2):
                for h in range(2):
                    o[b, h], lse[b, h] = _fp8_forward_emulated(qd[b, h], kd[b, h], vd[b, h], causal, 128 ** -0.5)
            do = np.abs(o - o_ref)
            worst_max = max(worst_max, do.max())
            margins_max.append(FP8_MAX_ABS_O / do.max())
            margins_mean[N] = min(margins_mean.get(N, np.inf), FP8_MEAN_ABS_O / do.mean())
            worst_lse = max(worst_lse, np.abs(lse - lse_ref).max())
    assert min(margins_max) >= 3.0, margins_max
    assert min(margins_mean.values()) >= 1.25, margins_mean
    assert min(m for n, m in margins_mean.items() if n >= 128) >= 2.2, margins_mean
    # the LSE sums fp32 values: the rounding of P does not reach it, and its bound is the bf16 path's
    assert worst_lse * 100 <= FP8_MAX_ABS_LSE, worst_lse
    # the emulation rounds: P in e4m3 moves O well beyond the bf16 rounding of the output (7.8e-3 here)
    assert worst_max > 3e-2, worst_max


def _bwd_emulated(q, k, v, do, causal, scale):
    """One head, fp64 [N, d] inputs (bf16 values): the kernel's roundings."""
    N = q.shape[0]
    o_ref, lse_ref = oracle.attention(q[None, None], k[None, None], v[None, None], causal, scale)
    o16, lse = bf16(o_ref[0, 0]), lse_ref[0, 0].astype(np.float32)
    dd = (do * o16).sum(axis=1).astype(np.float32)  # D from the bf16 O
    s = (q @ k.T).astype(np.float32)
    p = np.exp2(s * np.float32(scale * LOG2E) - (lse * np.float32(LOG2E))[:, None], dtype=np.float32)
    if causal:
        p = np.tril(p)
    p = bf16(p)
    dv = bf16(p.T @ do)
    dp = (do @ v.T).astype(np.float32)
    ds = bf16(p * (dp - dd[:, None]))
    dk = bf16(scale * (ds.T @ q))
    dq = bf16(scale * (ds @ k))
    return dq, dk, dv


@pytest.mark.parametrize("d", [64, 128])
def test_backward_bounds_cover_the_bf16_roundings(d):
    """Per case and gradient, with the GPU test's criterion (max and mean of
    |err| against GRAD_MAX_REL * max|ref| and GRAD_MEAN_REL * mean|ref|, plus
    GRAD_ATOL): the bounds are 2.7x or more the rounding-only error. Measured
    here: max |err| up to 0.60 % of max|ref| and mean |err| up to 0.36 % of
    mean|ref| (7 keys, causal)."""
    margins, worst_rel = [], 0.0
    for N in (1, 7, 128, 129, 255, 256, 300, 384):
        for causal in (False, True):
            B, H = (2, 2) if N <= 256 else (1, 2)
            q, k, v = wl.prefill_inputs(B, H, N, d, seed=N + d)
            do = wl.backward_inputs(B, H, N, d, seed=N + d)
            ref = oracle.attention_bwd(q, k, v, do, causal, d ** -0.5)
            f = lambda t: t.double().numpy()
            qq, kk, vv, dd = f(q), f(k), f(v), f(do)
            got = [np.zeros_like(r) for r in ref]
            for b in range(B):
                for h in range(H):
                    for i, g in enumerate(_bwd_emulated(qq[b, h], kk[b, h], vv[b, h], dd[b, h], causal, d ** -0.5)):
                        got[i][b, h] = g
            for g, r in zip(got, ref):
                err = np.abs(g - r)
                worst_rel = max(worst_rel, err.max() / max(np.abs(r).max(), 1e-30))
                margins.append((GRAD_MAX_REL * np.abs(r).max() + GRAD_ATOL) / max(err.max(), 1e-30))
                margins.append((GRAD_MEAN_REL * np.abs(r).mean() + GRAD_ATOL) / max(err.mean(), 1e-30))
    assert min(margins) >= 2.7, min(margins)
    # the emulation rounds: bf16 P and dS leave errors far above fp32 arithmetic
    assert worst_rel > 2e-3, worst_rel
