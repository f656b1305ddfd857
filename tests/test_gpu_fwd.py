"""Prefill attention on the GPU (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_29_gb300 import workloads as wl
from parity import Accumulator, compare, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    oracle.build()


def _run(q, k, v, causal, scale=None):
    import exact_attention_29_gb300 as fa

    o, lse = fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    fa.fa_check_device_error()
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 7, 128, 129, 200, 255, 256, 257, 384, 1000])
def test_small_shapes_full_oracle(N, d, causal):
    """Tiles are 128 rows, CTAs take 256 query rows: these sizes cover a single
    row, partial tiles, an inactive second Q tile, ragged key tails and several
    K/V tiles."""
    B, H = (2, 2) if N <= 256 else (1, 2)
    q, k, v = wl.prefill_inputs(B, H, N, d, seed=N + d)
    o, lse = _run(q, k, v, causal)
    o_ref, lse_ref = oracle.attention(q, k, v, causal, d ** -0.5)
    compare(o, lse, o_ref, lse_ref, f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_item_count_just_over_the_grid(causal):
    """B=7, H=11, N=700: 77 heads x 2 Q-tile pairs = 154 work items for 152
    persistent CTAs, so two CTAs take a second item (dealt in reverse), and the
    last pair of every head has a ragged second tile."""
    q, k, v = wl.prefill_inputs(7, 11, 700, 64, seed=77)
    o, lse = _run(q, k, v, causal)
    o_ref, lse_ref = oracle.attention(q, k, v, causal, 64 ** -0.5)
    compare(o, lse, o_ref, lse_ref, f"7x11x700 causal={causal}")


def test_pr1_config():
    """B=1, H=1, N=128, d=64, non-causal, seed 0 — the smallest named workload."""
    c = wl.PREFILL["pr1"]
    q, k, v = wl.prefill_inputs(c.B, c.H, c.N, c.d, seed=0)
    o, lse = _run(q, k, v, c.causal)
    o_ref, lse_ref = oracle.attention(q, k, v, c.causal, c.scale)
    compare(o, lse, o_ref, lse_ref, "pr1")


@pytest.mark.parametrize("name", ["gpt2_small", "gpt2_small_causal"])
def test_gpt2_small_full_oracle(name):
    c = wl.PREFILL[name]
    q, k, v = wl.prefill_inputs(c.B, c.H, c.N, c.d, seed=0)
    o, lse = _run(q, k, v, c.causal)
    o_ref, lse_ref = oracle.attention(q, k, v, c.causal, c.scale)
    compare(o, lse, o_ref, lse_ref, name)


def _sampled_check(c, rows_per_head, heads=None, seed=0):
    """Full-size run on the GPU; the oracle evaluates a seeded subset of rows of
    each checked head (each a full row over its visible keys)."""
    q, k, v = wl.prefill_inputs(c.B, c.H, c.N, c.d, seed=seed, device="cuda")
    o, lse = _run(q, k, v, c.causal)
    rows = wl.row_subsets(c.B, c.H, c.N, rows_per_head, seed=seed)
    heads = heads or [(b, h) for b in range(c.B) for h in range(c.H)]
    o_all, l_all, or_all, lr_all = [], [], [], []
    for b, h in heads:
        r = rows[b, h]
        # always include the last row (the longest causal row) and row 0
        r = torch.unique(torch.cat([r, torch.tensor([0, c.N - 1])]))
        kk, vv = k[b, h].cpu(), v[b, h].cpu()
        o_ref, lse_ref, _, _ = oracle.attention_rows(q[b, h, r.cuda()].cpu(), r.numpy(), kk, vv, c.causal, c.scale)
        o_all.append(o[b, h, r.cuda()].cpu())
        l_all.append(lse[b, h, r.cuda()].cpu())
        or_all.append(o_ref)
        lr_all.append(lse_ref)
    compare(torch.cat(o_all), torch.cat(l_all), np.concatenate(or_all), np.concatenate(lr_all), c.name)
    return o, lse


def _full_check(c, seed=0):
    """Full-size run on the GPU, then every row of every head against the oracle,
    one head at a time (each head's S and P are N x N in fp64)."""
    q, k, v = wl.prefill_inputs(c.B, c.H, c.N, c.d, seed=seed, device="cuda")
    o, lse = _run(q, k, v, c.causal)
    acc = Accumulator(f"{c.name} (all {c.B * c.H} heads, every row)")
    pos = np.arange(c.N)
    for b in range(c.B):
        qb, kb, vb, ob, lb = q[b].cpu(), k[b].cpu(), v[b].cpu(), o[b].cpu(), lse[b].cpu()
        for h in range(c.H):
            o_ref, lse_ref, _, _ = oracle.attention_rows(qb[h], pos, kb[h], vb[h], c.causal, c.scale)
            acc.add(ob[h], lb[h], o_ref, lse_ref)
    acc.finish()
    assert acc.n_o == c.B * c.H * c.N * c.d


def test_llama3_8b_prefill_full_oracle():
    """B2 H32 N4096 d128 causal: the whole output (33.5 M values of O, 262,144 of LSE)."""
    _full_check(wl.PREFILL["llama3_8b_prefill"])


def test_llama3_8b_prefill_noncausal_full_oracle():
    _full_check(wl.PREFILL["llama3_8b_prefill_noncausal"])


def test_long_16k_sampled():
    _sampled_check(wl.PREFILL["long_16k"], rows_per_head=256)


def test_long_64k_sampled():
    _sampled_check(wl.PREFILL["long_64k"], rows_per_head=256)


def test_deterministic():
    """No atomics in the forward: two runs are bitwise identical."""
    q, k, v = wl.prefill_inputs(2, 4, 777, 128, seed=5)
    o1, l1 = _run(q, k, v, True)
    o2, l2 = _run(q, k, v, True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_causal_row0_is_v0():
    """Row 0 sees only key 0: O_0 = V_0 (exactly, after bf16 rounding) and LSE_0 = scale q0.k0."""
    q, k, v = wl.prefill_inputs(1, 3, 300, 64, seed=6)
    o, lse = _run(q, k, v, True)
    assert torch.equal(o[0, :, 0].cpu(), v[0, :, 0])
    ref = (q[0, :, 0].double() * k[0, :, 0].double()).sum(-1) / 8.0
    assert (lse[0, :, 0].double().cpu() - ref).abs().max().item() <= 1e-4


def test_large_scores_rescale_path():
    """Scores far beyond exp range (scale 1, inputs x4): the running max and the
    conditional rescale of O must keep everything finite and exact."""
    q, k, v = wl.prefill_inputs(1, 2, 640, 128, seed=7)
    q = (q.float() * 4).to(torch.bfloat16)
    # growing keys so the row max keeps rising tile after tile
    ramp = torch.linspace(0.5, 3.0, 640).view(1, 1, 640, 1)
    k = (k.float() * ramp).to(torch.bfloat16)
    for causal in (False, True):
        o, lse = _run(q, k, v, causal, scale=1.0)
        o_ref, lse_ref = oracle.attention(q, k, v, causal, 1.0)
        compare(o, lse, o_ref, lse_ref, f"large scores causal={causal}")


def test_one_hot_dominant_rows():
    """A key equal to 8x its query dominates the row: O row = that V row."""
    q, k, v = wl.prefill_inputs(1, 1, 256, 64, seed=8)
    for i, j in ((3, 200), (130, 10), (255, 255)):
        k[0, 0, j] = (q[0, 0, i].float() * 8).to(torch.bfloat16)
    o, lse = _run(q, k, v, False)
    o_ref, lse_ref = oracle.attention(q, k, v, False, 0.125)
    compare(o, lse, o_ref, lse_ref, "one-hot")
    for i, j in ((3, 200), (130, 10), (255, 255)):
        assert (o[0, 0, i].float().cpu() - v[0, 0, j].float()).abs().max().item() <= 2e-2


def test_output_buffers_and_stream():
    """Caller-provided outputs on a side stream are filled in place."""
    import exact_attention_29_gb300 as fa

    q, k, v = wl.prefill_inputs(1, 2, 300, 64, seed=9)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o = torch.full_like(q, float("nan"))
    lse = torch.full((1, 2, 300), float("nan"), device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fa.fa_fwd(q, k, v, causal=True, o=o, lse=lse, stream=s)
    s.synchronize()
    fa.fa_check_device_error(s)
    o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), True, 0.125)
    compare(o, lse, o_ref, lse_ref, "side stream")


@pytest.mark.parametrize("d", [64, 128])
def test_output_16_byte_aligned_only(d):
    """An output that is 16- but not 32-byte aligned takes the 16-byte store
    path of the epilogue; both paths write the same bits."""
    import exact_attention_29_gb300 as fa

    q, k, v = wl.prefill_inputs(2, 3, 333, d, seed=10)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o_a = torch.empty_like(q)
    flat = torch.empty(q.numel() + 8, dtype=q.dtype, device="cuda")
    o_b = flat[8:].view(q.shape)  # 16 bytes past a 256-byte boundary
    assert o_a.data_ptr() % 32 == 0 and o_b.data_ptr() % 32 == 16
    lse = torch.empty((2, 3, 333), device="cuda")
    fa.fa_fwd(q, k, v, causal=True, o=o_a, lse=lse)
    fa.fa_fwd(q, k, v, causal=True, o=o_b, lse=lse)
    fa.fa_check_device_error()
    assert torch.equal(o_a, o_b)
    o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), True, d ** -0.5)
    compare(o_b, lse, o_ref, lse_ref, "16-byte aligned output")


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("causal", [False, True])
def test_host_buffer_call_matches_device_call(pinned, causal):
    """fa_fwd_host (host inputs and outputs, copies inside the call) gives the
    same bits as fa_fwd on device copies of the same inputs, from pinned and
    from pageable host memory, and matches the oracle."""
    import exact_attention_29_gb300 as fa

    q, k, v = wl.prefill_inputs(2, 3, 517, 128, seed=21 + int(causal))
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
        o_h = lse_h = None
    else:
        o_h = torch.full(q.shape, float("nan"), dtype=torch.bfloat16)
        lse_h = torch.full((2, 3, 517), float("nan"))
    s = torch.cuda.Stream()
    o_h, lse_h = fa.fa_fwd_host(q, k, v, causal=causal, o=o_h, lse=lse_h, stream=s)
    s.synchronize()
    fa.fa_check_device_error(s)
    assert o_h.device.type == "cpu" and o_h.is_pinned() == pinned
    o_d, lse_d = _run(q, k, v, causal)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_d.cpu())
    assert torch.equal(lse_h, lse_d.cpu())
    o_ref, lse_ref = oracle.attention(q, k, v, causal, 128 ** -0.5)
    compare(o_h, lse_h, o_ref, lse_ref, f"host buffers pinned={pinned} causal={causal}")


def test_host_buffer_calls_pipelined_over_streams():
    """Six fa_fwd_host calls issued round-robin over three streams without waiting
    in between (each stream reuses its own workspace while the others' copies and
    kernels are in flight): every call's outputs equal fa_fwd's on the same inputs."""
    import exact_attention_29_gb300 as fa

    streams = [torch.cuda.Stream() for _ in range(3)]
    cases = []
    for c in range(6):
        q, k, v = (t.pin_memory() for t in wl.prefill_inputs(1, 4, 640, 128, seed=40 + c))
        cases.append((q, k, v))
    outs = []
    for c, (q, k, v) in enumerate(cases):
        o = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
        lse = torch.empty((1, 4, 640)).pin_memory()
        fa.fa_fwd_host(q, k, v, causal=bool(c & 1), o=o, lse=lse, stream=streams[c % 3])
        outs.append((o, lse))
    torch.cuda.synchronize()
    for st in streams:
        fa.fa_check_device_error(st)
    for c, ((q, k, v), (o, lse)) in enumerate(zip(cases, outs)):
        o_d, lse_d = _run(q, k, v, bool(c & 1))
        torch.cuda.synchronize()
        assert torch.equal(o, o_d.cpu()), c
        assert torch.equal(lse, lse_d.cpu()), c


def test_host_buffer_call_refuses_device_memory():
    import exact_attention_29_gb300 as fa

    lib = fa.load_library()
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device="cuda")
    h = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16).pin_memory()
    lse = torch.zeros(1, 1, 128).pin_memory()
    st = lib.fa_fwd_host(h.data_ptr(), q.data_ptr(), h.data_ptr(), h.data_ptr(), lse.data_ptr(), 1, 1, 128, 64, 0,
                         0.125, None)
    assert st == fa.FA_ERR_INVALID_ARG
    assert b"device memory" in lib.fa_last_error_string()
    o = torch.full_like(h, float("nan")).pin_memory()
    st = lib.fa_fwd_host(h.data_ptr(), h.data_ptr(), h.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 1, 128, 64, 0,
                         0.125, None)
    assert st == fa.FA_OK
    torch.cuda.synchronize()
    fa.fa_check_device_error()
    assert torch.equal(o, h)  # zero V gives zero O


def test_bindings_reject_wrong_shapes_before_any_launch():
    """The library takes raw pointers; the binding refuses tensors whose extent
    or device does not match (caller-provided outputs and scales included)."""
    import exact_attention_29_gb300 as fa

    q = torch.zeros((1, 2, 200, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        fa.fa_fwd(q, q, q, o=torch.empty((1, 2, 100, 64), dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError):
        fa.fa_fwd(q, q, q, lse=torch.empty((1, 2, 100), device="cuda"))
    mask = torch.ones((2, 2), dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        fa.fa_fwd_sparse(q, q[:, :, :128].contiguous(), q, mask)
    with pytest.raises(ValueError):
        fa.fa_fwd_sparse(q, q, q, mask, o=torch.empty((1, 2, 200, 32), dtype=torch.bfloat16, device="cuda"))
    dq = torch.zeros((2, 4, 64), dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros((2, 4, 300, 64), dtype=torch.bfloat16, device="cuda")
    sl = torch.full((2,), 300, dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        fa.fa_decode(dq, cache, cache, sl, 2, o=torch.empty((2, 4, 32), dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError):
        fa.fa_decode(dq, cache, cache, sl, 2, lse=torch.empty((2, 3), device="cuda"))
    with pytest.raises(ValueError):
        fa.fa_decode_gqa(dq, cache[:, :2].contiguous(), cache[:, :2].contiguous(), sl, 2,
                         lse=torch.empty((2, 2), device="cuda"))
    q8 = torch.zeros((1, 2, 200, 128), dtype=torch.uint8, device="cuda")
    vt8 = torch.zeros((1, 2, 128, 208), dtype=torch.uint8, device="cuda")
    good = torch.ones((1, 2, 2), device="cuda")
    with pytest.raises(ValueError):
        fa.fa_fwd_fp8(q8, q8, vt8, torch.ones((1, 2, 1), device="cuda"), good, torch.ones((1, 2), device="cuda"))
    with pytest.raises(ValueError):
        fa.fa_fwd_fp8(q8, q8, vt8, good, good, torch.ones((1, 2, 2), device="cuda"))
    torch.cuda.synchronize()
    fa.fa_check_device_error()


def test_python_binding_rejects_bad_tensors():
    import exact_attention_29_gb300 as fa

    q = torch.zeros((1, 1, 8, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        fa.fa_fwd(q.float(), q, q)
    with pytest.raises(ValueError):
        fa.fa_fwd(q.cpu(), q, q)
    with pytest.raises(ValueError):
        fa.fa_fwd(q, q[:, :, :4], q)
    qq = torch.zeros((1, 1, 8, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd(qq, qq, qq)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED
