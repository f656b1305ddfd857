"""fa_decode_noalloc: decode attention for callers that cannot allocate device
memory while they decode (for example a serving engine whose KV-cache pool owns
nearly all of HBM, or a latency-critical decode loop). Its split partials live
in a fixed 16 MiB array inside libfa.so instead of a per-call allocation.

This file is collected last on purpose. Each check calls the new entry point
through the C ABI and compares it with fa_decode and with the fp64 oracle on
the same inputs, twice in a row, since all calls share one workspace that keeps
the previous contents.
"""

import gc

import pytest
import torch

import oracle
from exact_attention_29_gb300 import workloads as wl
from parity import MAX_ABS_LSE, MAX_ABS_O, MEAN_ABS_O, compare, require_gpu

pytestmark = pytest.mark.gpu

WORKSPACE_FLOATS = 1 << 22


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    oracle.build()


def _c_noalloc(lib, q, kc, vc, sl, splits, o, lse):
    B, H, L, d = kc.shape
    stream = torch.cuda.current_stream().cuda_stream
    return lib.fa_decode_noalloc(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), sl.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), B, H, L, d, splits, stream)


def _close(o_a, lse_a, o_b, lse_b):
    do = (o_a.float() - o_b.float()).abs()
    dl = (lse_a - lse_b).abs()
    assert do.max().item() <= MAX_ABS_O and do.mean().item() <= MEAN_ABS_O and dl.max().item() <= MAX_ABS_LSE


def test_noalloc_matches_decode_on_two_calls_in_a_row():
    import exact_attention_29_gb300 as fa

    lib = fa.load_library()
    cases = [
        # (B, H, L, d, splits, seqlens, seed): the second call reuses the workspace
        # with fewer splits and shorter sequences than the first left in it
        (4, 8, 2048, 128, 16, [2048, 1, 700, 1999], 21),
        (3, 4, 1024, 64, 3, [5, 1024, 333], 22),
    ]
    for B, H, L, d, splits, lens, seed in cases:
        q, kc, vc, _ = wl.decode_inputs(B, H, L, d, seed=seed, device="cuda")
        sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
        o_ref, lse_ref = fa.fa_decode(q, kc, vc, sl, splits)
        o = torch.empty_like(q)
        lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
        st = _c_noalloc(lib, q, kc, vc, sl, splits, o, lse)
        assert st == fa.FA_OK, lib.fa_last_error_string()
        torch.cuda.synchronize()
        fa.fa_check_device_error()
        _close(o, lse, o_ref, lse_ref)
        ro, rl = oracle.decode(q.cpu(), kc.cpu(), vc.cpu(), sl.cpu())
        compare(o, lse, ro, rl, f"fa_decode_noalloc B{B} H{H} L{L} d{d} S{splits}")


def test_noalloc_allocates_nothing():
    """After the first call on the device (which looks up the workspace address),
    further calls leave the device's free memory and torch's allocator unchanged."""
    import exact_attention_29_gb300 as fa

    lib = fa.load_library()
    q, kc, vc, _ = wl.decode_inputs(2, 4, 4096, 128, seed=23, device="cuda")
    sl = torch.tensor([4096, 1234], dtype=torch.int32, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((2, 4), dtype=torch.float32, device="cuda")
    assert _c_noalloc(lib, q, kc, vc, sl, 32, o, lse) == fa.FA_OK
    torch.cuda.synchronize()
    gc.collect()  # earlier tests' tensors are freed now, not during the calls below
    free_before = torch.cuda.mem_get_info()[0]
    allocated, reserved = torch.cuda.memory_allocated(), torch.cuda.memory_reserved()
    for _ in range(2):
        assert _c_noalloc(lib, q, kc, vc, sl, 32, o, lse) == fa.FA_OK
    torch.cuda.synchronize()
    # neither torch's allocator nor the device as a whole gave out memory
    assert torch.cuda.memory_allocated() <= allocated and torch.cuda.memory_reserved() <= reserved
    assert torch.cuda.mem_get_info()[0] >= free_before
    ro, rl = oracle.decode(q.cpu(), kc.cpu(), vc.cpu(), sl.cpu())
    compare(o, lse, ro, rl, "fa_decode_noalloc after repeated calls")
    o_ref, lse_ref = fa.fa_decode(q, kc, vc, sl, 32)
    _close(o, lse, o_ref, lse_ref)


def test_noalloc_rejects_requests_beyond_the_workspace():
    import exact_attention_29_gb300 as fa

    lib = fa.load_library()
    # 16 * 32 * 64 * 129 = 4,227,072 > 4,194,304 fp32 values
    B, H, L, d, splits = 16, 32, 64, 128, 64
    assert B * H * splits * (d + 1) > WORKSPACE_FLOATS
    q = torch.zeros((B, H, d), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((B, H, L, d), dtype=torch.bfloat16, device="cuda")
    sl = torch.full((B,), L, dtype=torch.int32, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    assert _c_noalloc(lib, q, kc, kc, sl, splits, o, lse) == fa.FA_ERR_INVALID_ARG
    assert b"static workspace" in lib.fa_last_error_string()
    # one split fewer fits
    assert B * H * 32 * (d + 1) <= WORKSPACE_FLOATS
    assert _c_noalloc(lib, q, kc, kc, sl, 32, o, lse) == fa.FA_OK
    torch.cuda.synchronize()
