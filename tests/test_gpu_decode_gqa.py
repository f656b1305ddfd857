"""Flash-Decoding with grouped K/V heads on the GPU (through the C ABI) against
the fp64 oracle."""
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


def _run(q, kc, vc, seqlens, splits):
    import exact_attention_29_gb300 as fa

    o, lse = fa.fa_decode_gqa(q.cuda(), kc.cuda(), vc.cuda(), seqlens.cuda(), num_splits=splits)
    fa.fa_check_device_error()
    return o, lse


# (Hq, Hkv): g = 4, 8 (MQA), 3 (not a power of two), 1, 32 (two groups of 16),
# 20 (a full group and a group of 4)
HEADS = [(8, 2), (8, 1), (6, 2), (4, 4), (32, 1), (40, 2)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("heads", HEADS, ids=lambda h: f"{h[0]}x{h[1]}")
@pytest.mark.parametrize("splits", [1, 3, 8])
def test_small_ragged(d, heads, splits):
    """Lengths 300 (several 128-key tiles and a ragged tail), 1, 77 and 128;
    with 8 splits the short sequences leave empty splits."""
    Hq, Hkv = heads
    q, kc, vc, _ = wl.decode_gqa_inputs(4, Hq, Hkv, 300, d, seed=d + splits + Hq)
    seqlens = torch.tensor([300, 1, 77, 128], dtype=torch.int32)
    o, lse = _run(q, kc, vc, seqlens, splits)
    o_ref, lse_ref = oracle.decode_gqa(q, kc, vc, seqlens)
    compare(o, lse, o_ref, lse_ref, f"d={d} heads={heads} splits={splits}")


@pytest.mark.parametrize("d", [64, 128])
def test_cache_beyond_length_may_hold_nan(d):
    """Entries at or past seqlens[b] are not part of the sequence: filling them
    with NaN must not change the result."""
    q, kc, vc, _ = wl.decode_gqa_inputs(2, 8, 2, 400, d, seed=21)
    seqlens = torch.tensor([257, 130], dtype=torch.int32)
    o_ref, lse_ref = oracle.decode_gqa(q, kc, vc, seqlens)
    kn, vn = kc.clone(), vc.clone()
    for b, n in enumerate(seqlens.tolist()):
        kn[b, :, n:] = float("nan")
        vn[b, :, n:] = float("nan")
    for splits in (1, 2, 5):
        o, lse = _run(q, kn, vn, seqlens, splits)
        compare(o, lse, o_ref, lse_ref, f"nan tail splits={splits}")


def test_large_scores_take_the_rescale_path():
    """A query scaled up 12x: the running max of a query moves by more than
    the threshold between tiles, so O is rescaled in TMEM."""
    q, kc, vc, _ = wl.decode_gqa_inputs(1, 16, 2, 2048, 128, seed=8)
    q = (q.float() * 12).bfloat16()
    seqlens = torch.tensor([2048], dtype=torch.int32)
    o, lse = _run(q, kc, vc, seqlens, 2)
    o_ref, lse_ref = oracle.decode_gqa(q, kc, vc, seqlens)
    compare(o, lse, o_ref, lse_ref, "rescale")


def test_group_of_one_agrees_with_multi_head_decode():
    import exact_attention_29_gb300 as fa

    q, kc, vc, _ = wl.decode_inputs(2, 4, 700, 128, seed=4)
    seqlens = torch.tensor([700, 333], dtype=torch.int32)
    o1, l1 = _run(q, kc, vc, seqlens, 4)
    o2, l2 = fa.fa_decode(q.cuda(), kc.cuda(), vc.cuda(), seqlens.cuda(), 4)
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-2
    assert (l1 - l2).abs().max().item() <= 1e-3


@pytest.mark.parametrize("name", ["decode_gqa8_32k", "decode_gqa8_32k_ragged", "decode_mqa_32k"])
def test_full_size_sampled(name):
    """Full-size launch with 8 and 16 splits; the oracle checks every query
    head of a seeded sample of (batch, K/V head) groups."""
    c = wl.DECODE_GQA[name]
    q, kc, vc, seqlens = wl.decode_gqa_inputs(c.B, c.Hq, c.Hkv, c.L, c.d, seed=0, ragged=c.ragged, device="cuda")
    outs = {s: _run(q, kc, vc, seqlens, s) for s in (8, 16)}
    gen = torch.Generator().manual_seed(3)
    pairs = torch.randperm(c.B * c.Hkv, generator=gen)[:4].tolist()
    sl = seqlens.cpu()
    for s, (o, lse) in outs.items():
        o_sel, l_sel, o_ref, l_ref = [], [], [], []
        for flat in pairs:
            b, kvh = divmod(flat, c.Hkv)
            n = int(sl[b])
            hs = slice(kvh * c.g, (kvh + 1) * c.g)
            ro, rl = oracle.decode_gqa(q[b:b + 1, hs].cpu(), kc[b:b + 1, kvh:kvh + 1, :n].cpu(),
                                       vc[b:b + 1, kvh:kvh + 1, :n].cpu(), torch.tensor([n], dtype=torch.int32))
            o_sel.append(o[b, hs].cpu())
            l_sel.append(lse[b, hs].cpu())
            o_ref.append(ro[0])
            l_ref.append(rl[0])
        compare(torch.cat(o_sel), torch.cat(l_sel), np.concatenate(o_ref), np.concatenate(l_ref), f"{name} S={s}")
    assert (outs[8][0].float() - outs[16][0].float()).abs().max().item() <= 2e-2
    assert (outs[8][1] - outs[16][1]).abs().max().item() <= 1e-3


def test_rejects_bad_tensors():
    import exact_attention_29_gb300 as fa

    q = torch.zeros((1, 6, 128), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((1, 4, 16, 128), dtype=torch.bfloat16, device="cuda")
    sl = torch.ones(1, dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        fa.fa_decode_gqa(q, kc, kc, sl, 2)
