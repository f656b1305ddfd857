"""Calls that allocate nothing (fa_fwd, fa_decode_noalloc) captured in a CUDA
graph and replayed: every replay computes exactly what eager calls compute,
and it reads the input buffers at replay time, not values frozen at capture."""
import pytest
import torch

import oracle
from exact_attention_29_gb300 import workloads as wl
from parity import compare, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    oracle.build()


def _eager(fa, q, k, v, dq, kc, vc, sl):
    o, lse = fa.fa_fwd(q, k, v, causal=True)
    od, lsed = fa.fa_decode_noalloc(dq, kc, vc, sl, num_splits=8)
    torch.cuda.synchronize()
    fa.fa_check_device_error()
    return o, lse, od, lsed


def test_prefill_and_decode_replayed_from_a_graph():
    import exact_attention_29_gb300 as fa

    q, k, v = (t.cuda() for t in wl.prefill_inputs(2, 4, 700, 128, seed=31))
    dq, kc, vc, _ = wl.decode_inputs(4, 8, 3000, 128, seed=32)
    dq, kc, vc = dq.cuda(), kc.cuda(), vc.cuda()
    sl = torch.tensor([3000, 1, 1777, 64], dtype=torch.int32, device="cuda")
    ref = _eager(fa, q, k, v, dq, kc, vc, sl)  # also initialises the library's per-device state

    o, lse = torch.empty_like(q), torch.empty((2, 4, 700), device="cuda")
    od, lsed = torch.empty_like(dq), torch.empty((4, 8), device="cuda")
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        fa.fa_fwd(q, k, v, causal=True, o=o, lse=lse, stream=s)
        fa.fa_decode_noalloc(dq, kc, vc, sl, num_splits=8, o=od, lse=lsed, stream=s)
    for _ in range(3):
        for t in (o, lse, od, lsed):
            t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        fa.fa_check_device_error()
        for got, want in zip((o, lse, od, lsed), ref):
            assert torch.equal(got, want)

    # new values in the same buffers: the replay computes on them
    q.copy_(wl.prefill_inputs(2, 4, 700, 128, seed=33)[0].cuda())
    dq.copy_(wl.decode_inputs(4, 8, 3000, 128, seed=34)[0].cuda())
    sl.copy_(torch.tensor([5, 3000, 129, 2048], dtype=torch.int32))
    g.replay()
    torch.cuda.synchronize()
    fa.fa_check_device_error()
    ref2 = _eager(fa, q, k, v, dq, kc, vc, sl)
    for got, want in zip((o, lse, od, lsed), ref2):
        assert torch.equal(got, want)
    o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), True, 128 ** -0.5)
    compare(o, lse, o_ref, lse_ref, "graph replay, prefill")
    od_ref, lsed_ref = oracle.decode(dq.cpu(), kc.cpu(), vc.cpu(), sl.cpu())
    compare(od, lsed, od_ref, lsed_ref, "graph replay, decode")
    del g
