"""Backward pass on the GPU (through the C ABI) against the fp64 backward oracle."""
import pytest
import torch

import oracle
from exact_attention_29_gb300 import workloads as wl
from parity import compare_grads, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    oracle.build()


def _grads(q, k, v, do, causal, scale=None):
    import exact_attention_29_gb300 as fa

    q, k, v, do = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.fa_fwd(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, lse, do, causal=causal, scale=scale)
    fa.fa_check_device_error()
    return dq, dk, dv


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 7, 128, 129, 255, 256, 300, 384])
def test_small_shapes_full_oracle(N, d, causal):
    """Fewer work items (K/V tiles of a head) than SMs, one per CTA: a single
    row, partial tiles, ragged tails, and several K/V tiles whose dQ shares
    meet in the atomic accumulation."""
    B, H = (2, 2) if N <= 256 else (1, 2)
    q, k, v = wl.prefill_inputs(B, H, N, d, seed=N + d)
    do = wl.backward_inputs(B, H, N, d, seed=N + d)
    got = _grads(q, k, v, do, causal)
    ref = oracle.attention_bwd(q, k, v, do, causal, d ** -0.5)
    compare_grads(got, ref, f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_several_waves_full_oracle(d, causal):
    """60 heads x 6 K/V tiles = 360 CTAs, more than two waves of the 152 SMs,
    every gradient element against the oracle: under the causal mask the CTAs
    of a wave walk very different numbers of Q tiles, and the last tile is
    ragged."""
    B, H, N = 3, 20, 700
    q, k, v = wl.prefill_inputs(B, H, N, d, seed=d + 1)
    do = wl.backward_inputs(B, H, N, d, seed=d + 1)
    got = _grads(q, k, v, do, causal)
    ref = oracle.attention_bwd(q, k, v, do, causal, d ** -0.5)
    compare_grads(got, ref, f"B={B} H={H} N={N} d={d} causal={causal}")


def test_non_default_scale():
    q, k, v = wl.prefill_inputs(1, 2, 200, 64, seed=5)
    do = wl.backward_inputs(1, 2, 200, 64, seed=5)
    got = _grads(q, k, v, do, True, scale=0.3)
    compare_grads(got, oracle.attention_bwd(q, k, v, do, True, 0.3), "scale=0.3")


def test_gpt2_small_causal_full_oracle():
    c = wl.PREFILL["gpt2_small_causal"]
    q, k, v = wl.prefill_inputs(c.B, c.H, c.N, c.d, seed=0)
    do = wl.backward_inputs(c.B, c.H, c.N, c.d, seed=0)
    got = _grads(q, k, v, do, c.causal)
    compare_grads(got, oracle.attention_bwd(q, k, v, do, c.causal, c.scale), c.name)


@pytest.mark.parametrize("name", ["llama3_8b_prefill", "llama3_8b_prefill_noncausal"])
def test_llama3_8b_full_size_sampled_heads(name):
    """Full-size launch; every head's gradients depend only on that head, so
    the oracle checks two whole heads of the result (the first and the last)."""
    c = wl.PREFILL[name]
    q, k, v = wl.prefill_inputs(c.B, c.H, c.N, c.d, seed=0, device="cuda")
    do = wl.backward_inputs(c.B, c.H, c.N, c.d, seed=0, device="cuda")
    dq, dk, dv = _grads(q, k, v, do, c.causal)
    for b, h in ((0, 0), (c.B - 1, c.H - 1)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref = oracle.attention_bwd(q[sl].cpu(), k[sl].cpu(), v[sl].cpu(), do[sl].cpu(), c.causal, c.scale)
        compare_grads((dq[sl], dk[sl], dv[sl]), ref, f"{name} head ({b},{h})")


def test_repeat_calls_are_deterministic_up_to_atomics():
    """Two calls on the same inputs: dK and dV are written once per key and are
    bitwise identical; dQ is summed by atomics in varying order and agrees to
    fp32 reassociation before its bf16 rounding."""
    q, k, v = wl.prefill_inputs(1, 4, 640, 128, seed=11)
    do = wl.backward_inputs(1, 4, 640, 128, seed=11)
    a = _grads(q, k, v, do, True)
    b = _grads(q, k, v, do, True)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert (a[0].float() - b[0].float()).abs().max().item() <= 2 ** -7 * a[0].float().abs().max().item()
