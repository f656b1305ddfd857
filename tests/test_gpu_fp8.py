"""FP8 (e4m3) path on the GPU: the quantizer against the fp64 quantization
oracle, and the e4m3 forward against the fp64 attention oracle run on the
dequantized inputs (the inputs handed to the GPU forward are the oracle's codes
and scales).

Tolerances for the forward: beyond the inputs' quantization the kernel rounds
P to e4m3 (3 mantissa bits) for the P V product while l sums the fp32 values.
A CPU emulation of exactly that rounding against the fp64 oracle
(test_tolerance_emulation.py, on these tests' inputs) gives max |dO| <= 4.8e-2
(128 keys, causal: short rows, where few keys average the rounding) and mean
|dO| <= 6.2e-3 (7 keys per row), 3.5e-3 or less from 128 keys on. The max bound
is 3.1x the emulated error; the mean bound 1.3x at 7 keys and 2.2x or more
from 128 keys on. The LSE uses the fp32 sums, so it stays at the bf16 path's
bound.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8 as ofp8
from exact_attention_29_gb300 import workloads as wl
from parity import record, require_gpu

pytestmark = pytest.mark.gpu

FP8_MAX_ABS_O = 0.15
FP8_MEAN_ABS_O = 8e-3
FP8_MAX_ABS_LSE = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    oracle.build()


def _signs(seed, d=128):
    return np.random.default_rng(seed).choice([-1.0, 1.0], size=d)


def _oracle_inputs(q, k, v, signs):
    """Oracle quantization (rotated Q, K with tile scales; V^T with a head scale)."""
    qc, qs = ofp8.quantize(q.double().numpy(), signs)
    kc, ks = ofp8.quantize(k.double().numpy(), signs)
    vc, vs = ofp8.quantize(v.double().numpy(), per_head=True, transpose=True)
    return (qc, qs), (kc, ks), (vc, vs)


def _to_gpu(q, k, v):
    (qc, qs), (kc, ks), (vc, vs) = q, k, v
    B, H, d, N = vc.shape
    pitch = (N + 15) // 16 * 16
    vt = np.zeros((B, H, d, pitch), dtype=np.uint8)
    vt[..., :N] = vc
    f = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dt).cuda()
    return (f(qc, torch.uint8), f(kc, torch.uint8), f(vt, torch.uint8), f(qs, torch.float32), f(ks, torch.float32),
            f(vs, torch.float32))


def _compare(o, lse, o_ref, lse_ref, what):
    o = o.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), what
    do, dl = np.abs(o - o_ref), np.abs(lse - lse_ref)
    msg = f"{what}: max|dO|={do.max():.3e} mean|dO|={do.mean():.3e} max|dLSE|={dl.max():.3e}"
    ok = do.max() <= FP8_MAX_ABS_O and do.mean() <= FP8_MEAN_ABS_O and dl.max() <= FP8_MAX_ABS_LSE
    record("forward e4m3", what, ok, max_abs_dO=do.max(), mean_abs_dO=do.mean(), max_abs_dLSE=dl.max(), elements=o.size)
    assert ok, msg


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 7, 128, 129, 300, 1000])
def test_fwd_fp8_against_oracle_on_dequantized_inputs(N, causal):
    import exact_attention_29_gb300 as fa

    q, k, v = wl.prefill_inputs(2, 2, N, 128, seed=N + 3)
    qi, ki, vi = _oracle_inputs(q, k, v, _signs(N))
    args = _to_gpu(qi, ki, vi)
    o, lse = fa.fa_fwd_fp8(*args, causal=causal)
    fa.fa_check_device_error()
    qd, kd = ofp8.dequantize(*qi), ofp8.dequantize(*ki)
    vd = ofp8.dequantize(*vi, transpose=True)
    o_ref, lse_ref = oracle.attention(qd, kd, vd, causal, 128 ** -0.5)
    _compare(o, lse, o_ref, lse_ref, f"N={N} causal={causal}")


def _codes_agree(gpu_codes, ref_codes, ref_values, what):
    """Codes equal, or the exact value sits on a rounding tie (within fp32
    error) that the kernel's fp32 arithmetic decided the other way."""
    g = gpu_codes.cpu().numpy()
    diff = g != ref_codes
    frac = diff.mean()
    assert frac <= 1e-3, f"{what}: {frac:.2e} of the codes differ"
    if diff.any():
        gv = ofp8.e4m3_decode(g[diff])
        rv = ofp8.e4m3_decode(ref_codes[diff])
        x = ref_values[diff]
        mid = (gv + rv) / 2
        assert np.all(np.abs(x - mid) <= 1e-5 * np.abs(x) + 1e-12), f"{what}: a code differs away from a tie"


@pytest.mark.parametrize("rotate", [False, True])
def test_quantizer_matches_oracle(rotate):
    import exact_attention_29_gb300 as fa

    q, _, v = wl.prefill_inputs(2, 3, 300, 128, seed=9)
    signs = _signs(4) if rotate else None
    sg = torch.tensor(signs, dtype=torch.float32).cuda() if rotate else None
    codes, scales = fa.fa_quantize_fp8(q.cuda(), sg)
    fa.fa_check_device_error()
    rc, rs = ofp8.quantize(q.double().numpy(), signs)
    np.testing.assert_allclose(scales.cpu().numpy(), rs, rtol=1e-5)
    y = q.double().numpy() @ ofp8.hadamard(128, signs) if rotate else q.double().numpy()
    scaled = y / np.repeat(rs, 128, axis=2)[:, :, :300, None]
    _codes_agree(codes, rc, scaled, f"Q rotate={rotate}")
    # V: one scale per head, transposed
    vcodes, vscales = fa.fa_quantize_fp8(v.cuda(), None, per_head=True, transpose=True)
    fa.fa_check_device_error()
    rvc, rvs = ofp8.quantize(v.double().numpy(), per_head=True, transpose=True)
    np.testing.assert_allclose(vscales.cpu().numpy(), rvs, rtol=1e-5)
    vscaled = np.swapaxes(v.double().numpy(), 2, 3) / rvs[:, :, None, None]
    _codes_agree(vcodes[..., :300].contiguous(), rvc, vscaled, "V^T")


def test_rotation_reduces_the_error_with_outlier_dimensions():
    """[CTX] §4.4.2: with a few feature dimensions of Q and K 40x larger than the
    rest, quantizing the rotated Q and K gives attention much closer to the
    exact (bf16-input) result than quantizing them as they are."""
    import exact_attention_29_gb300 as fa

    q, k, v = wl.prefill_inputs(1, 4, 1024, 128, seed=17)
    q, k = q.float(), k.float()
    for c in (3, 77):
        q[..., c] *= 40.0
        k[..., c] *= 40.0
    q, k = q.bfloat16(), k.bfloat16()
    scale = 128 ** -0.5 / 8  # keeps the scores in a softmax-friendly range despite the outliers
    o_true, _ = oracle.attention(q, k, v, False, scale)
    errs = {}
    for rotate in (False, True):
        sg = torch.tensor(_signs(23), dtype=torch.float32).cuda() if rotate else None
        q8, qs = fa.fa_quantize_fp8(q.cuda(), sg)
        k8, ks = fa.fa_quantize_fp8(k.cuda(), sg)
        vt8, vs = fa.fa_quantize_fp8(v.cuda(), None, per_head=True, transpose=True)
        o, _ = fa.fa_fwd_fp8(q8, k8, vt8, qs, ks, vs, causal=False, scale=scale)
        fa.fa_check_device_error()
        errs[rotate] = np.abs(o.float().cpu().numpy() - o_true).mean()
    assert errs[True] < 0.7 * errs[False], errs


@pytest.mark.parametrize("causal", [True, False])
def test_llama3_8b_full_size_sampled_rows(causal):
    """Full size (B2 H32 N4096 d128): oracle-quantized inputs, the GPU result on
    seeded rows of four heads against the oracle on the dequantized inputs."""
    import exact_attention_29_gb300 as fa

    c = wl.PREFILL["llama3_8b_prefill"]
    q, k, v = wl.prefill_inputs(c.B, c.H, c.N, c.d, seed=0)
    qi, ki, vi = _oracle_inputs(q, k, v, _signs(0))
    o, lse = fa.fa_fwd_fp8(*_to_gpu(qi, ki, vi), causal=causal)
    fa.fa_check_device_error()
    rows = wl.row_subsets(c.B, c.H, c.N, 48, seed=0)
    qd, kd = ofp8.dequantize(*qi), ofp8.dequantize(*ki)
    vd = ofp8.dequantize(*vi, transpose=True)
    og, lg, orf, lrf = [], [], [], []
    for b, h in ((0, 0), (0, 31), (1, 5), (1, 30)):
        r = torch.unique(torch.cat([rows[b, h], torch.tensor([0, c.N - 1])])).numpy()
        ro, rl, _, _ = oracle.attention_rows(qd[b, h, r], r, kd[b, h], vd[b, h], causal, c.scale)
        og.append(o[b, h, r].cpu())
        lg.append(lse[b, h, r].cpu())
        orf.append(ro)
        lrf.append(rl)
    _compare(torch.cat(og), torch.cat(lg), np.concatenate(orf), np.concatenate(lrf), f"llama causal={causal}")
