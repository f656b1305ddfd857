"""The fp64 grouped-K/V decode oracle against its pins (CPU only).

Lecture 5 notes, Exercise 7: g = Hq / Hkv query heads share one K/V head. The
oracle is pinned to (1) the multi-head decode oracle (itself pinned to the
last causal row of the prefill oracle) run on K/V heads repeated g times, which
fixes the head grouping, and (2) a direct numpy evaluation of softmax(q K^T /
sqrt(d)) V on tiny inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_29_gb300 import workloads as wl


@pytest.fixture(scope="module", autouse=True)
def _build():
    oracle.build()


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (6, 3), (5, 1), (4, 4)])
def test_equals_multi_head_decode_on_repeated_kv(Hq, Hkv):
    q, k, v, _ = wl.decode_gqa_inputs(2, Hq, Hkv, 40, 16, seed=Hq * 10 + Hkv)
    seqlens = torch.tensor([40, 13], dtype=torch.int32)
    o, lse = oracle.decode_gqa(q, k, v, seqlens)
    g = Hq // Hkv
    # consecutive query heads share a K/V head: repeat each K/V head g times in place
    k_rep = k.repeat_interleave(g, dim=1)
    v_rep = v.repeat_interleave(g, dim=1)
    o_ref, lse_ref = oracle.decode(q, k_rep, v_rep, seqlens)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-13)


def test_grouping_is_consecutive_not_strided():
    """Query head h uses K/V head h // g; the strided reading h % Hkv differs."""
    q, k, v, _ = wl.decode_gqa_inputs(1, 4, 2, 20, 8, seed=3)
    seqlens = torch.tensor([20], dtype=torch.int32)
    o, _ = oracle.decode_gqa(q, k, v, seqlens)
    o_strided, _ = oracle.decode(q, k.repeat(1, 2, 1, 1), v.repeat(1, 2, 1, 1), seqlens)
    assert np.abs(o[0, 1] - o_strided[0, 1]).max() > 1e-3


def test_numpy_brute_force():
    B, Hq, Hkv, L, d = 2, 6, 2, 9, 4
    q, k, v, _ = wl.decode_gqa_inputs(B, Hq, Hkv, L, d, seed=5)
    seqlens = torch.tensor([9, 4], dtype=torch.int32)
    o, lse = oracle.decode_gqa(q, k, v, seqlens)
    qn, kn, vn = (t.double().numpy() for t in (q, k, v))
    for b in range(B):
        n = int(seqlens[b])
        for h in range(Hq):
            kv = h // (Hq // Hkv)
            s = kn[b, kv, :n] @ qn[b, h] / np.sqrt(d)
            w = np.exp(s - s.max())
            np.testing.assert_allclose(o[b, h], (w / w.sum()) @ vn[b, kv, :n], rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(lse[b, h], s.max() + np.log(w.sum()), rtol=0, atol=1e-12)


def test_rejects_indivisible_heads():
    q, k, v, _ = wl.decode_gqa_inputs(1, 6, 4, 8, 8, seed=1)
    with pytest.raises(Exception):
        oracle.decode_gqa(q[:, :5], k, v, torch.tensor([8], dtype=torch.int32))
