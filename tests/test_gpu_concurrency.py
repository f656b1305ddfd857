"""The library under concurrent use: several streams and host threads at once,
and many calls through the workspace pool (memory stays flat)."""
import threading

import numpy as np
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


def test_two_streams_at_once():
    """Prefill on one stream and decode on another, enqueued back to back, each
    equal to the oracle."""
    import exact_attention_29_gb300 as fa

    q, k, v = wl.prefill_inputs(2, 4, 700, 128, seed=31)
    dq, kc, vc, _ = wl.decode_inputs(3, 4, 900, 128, seed=32)
    sl = torch.tensor([900, 333, 5], dtype=torch.int32)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    dqd, kcd, vcd, sld = dq.cuda(), kc.cuda(), vc.cuda(), sl.cuda()
    torch.cuda.synchronize()
    for _ in range(5):
        o1, l1 = fa.fa_fwd(qd, kd, vd, causal=True, stream=s1)
        o2, l2 = fa.fa_decode(dqd, kcd, vcd, sld, 4, stream=s2)
    torch.cuda.synchronize()
    fa.fa_check_device_error()
    compare(o1, l1, *oracle.attention(q, k, v, True, 128 ** -0.5), "prefill on stream 1")
    compare(o2, l2, *oracle.decode(dq, kc, vc, sl), "decode on stream 2")


def test_host_threads_share_the_library():
    """Four host threads, each with its own stream, call every allocating entry
    point (workspaces come from the library's pool)."""
    import exact_attention_29_gb300 as fa

    q, kc, vc, _ = wl.decode_gqa_inputs(2, 8, 2, 600, 128, seed=33)
    sl = torch.tensor([600, 200], dtype=torch.int32)
    ref = oracle.decode_gqa(q, kc, vc, sl)
    qd, kcd, vcd, sld = q.cuda(), kc.cuda(), vc.cuda(), sl.cuda()
    pq, pk, pv = (t.cuda() for t in wl.prefill_inputs(1, 2, 300, 64, seed=34))
    dout = wl.backward_inputs(1, 2, 300, 64, seed=34).cuda()
    torch.cuda.synchronize()
    results, errors = {}, []

    def work(i):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(10):
                    o, lse = fa.fa_decode_gqa(qd, kcd, vcd, sld, 2 + i, stream=s)
                    po, plse = fa.fa_fwd(pq, pk, pv, causal=True, stream=s)
                    grads = fa.fa_bwd(pq, pk, pv, po, plse, dout, causal=True, stream=s)
                s.synchronize()
            results[i] = (o.cpu(), lse.cpu(), [g.cpu() for g in grads])
        except Exception as e:  # reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    fa.fa_check_device_error()
    for i in range(4):
        compare(results[i][0], results[i][1], ref[0], ref[1], f"thread {i}")
    # the backward's dK and dV are written once per key: identical across threads
    for i in range(1, 4):
        assert torch.equal(results[i][2][1], results[0][2][1]) and torch.equal(results[i][2][2], results[0][2][2])


def test_repeated_calls_keep_memory_flat():
    """200 calls of each allocating entry point: the workspace pool reuses its
    memory, so the device's free memory does not shrink call after call."""
    import exact_attention_29_gb300 as fa

    q, kc, vc, sl = wl.decode_inputs(4, 8, 4096, 128, seed=35, device="cuda")
    pq, pk, pv = wl.prefill_inputs(1, 4, 1024, 128, seed=36, device="cuda")
    dout = wl.backward_inputs(1, 4, 1024, 128, seed=36, device="cuda")
    mask = torch.ones((8, 8), dtype=torch.uint8, device="cuda")

    def round_():
        for _ in range(50):
            fa.fa_decode(q, kc, vc, sl, 16)
            o, lse = fa.fa_fwd_sparse(pq, pk, pv, mask)
            fa.fa_bwd(pq, pk, pv, o, lse, dout)
        torch.cuda.synchronize()

    round_()
    free_before = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        round_()
    free_after = torch.cuda.mem_get_info()[0]
    fa.fa_check_device_error()
    assert free_before - free_after < 64 << 20, (free_before, free_after)
