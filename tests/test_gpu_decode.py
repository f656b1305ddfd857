"""Flash-Decoding on the GPU (through the C ABI) against the fp64 oracle."""
import os
from concurrent.futures import ThreadPoolExecutor

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

    o, lse = fa.fa_decode(q.cuda(), kc.cuda(), vc.cuda(), seqlens.cuda(), num_splits=splits)
    fa.fa_check_device_error()
    return o, lse


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("splits", [1, 3, 8, 64])
def test_small_ragged(d, splits):
    """Ragged lengths including 1 and lengths shorter than splits x 64 (empty splits)."""
    q, kc, vc, _ = wl.decode_inputs(3, 2, 300, d, seed=d + splits)
    seqlens = torch.tensor([300, 1, 77], dtype=torch.int32)
    o, lse = _run(q, kc, vc, seqlens, splits)
    o_ref, lse_ref = oracle.decode(q, kc, vc, seqlens)
    compare(o, lse, o_ref, lse_ref, f"d={d} splits={splits}")


def test_split_count_does_not_change_the_result():
    """CMU 15-779 Lecture 5 notes §8.4: cutting into 2, 4 or 7 segments gave identical generations."""
    q, kc, vc, _ = wl.decode_inputs(2, 4, 1500, 128, seed=11)
    seqlens = torch.tensor([1500, 999], dtype=torch.int32)
    outs = [_run(q, kc, vc, seqlens, s) for s in (1, 2, 4, 7, 16, 32)]
    o_ref, lse_ref = oracle.decode(q, kc, vc, seqlens)
    for o, lse in outs:
        compare(o, lse, o_ref, lse_ref, "splits")
    for o, lse in outs[1:]:
        assert (o.float() - outs[0][0].float()).abs().max().item() <= 2e-2
        assert (lse - outs[0][1]).abs().max().item() <= 1e-4


def test_decode_equals_last_causal_row():
    """The cached decode step equals the last row of causal prefill (Lecture 5 notes §8.2)."""
    import exact_attention_29_gb300 as fa

    q, k, v = wl.prefill_inputs(1, 4, 777, 128, seed=12)
    o_f, lse_f = fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    seqlens = torch.tensor([777], dtype=torch.int32)
    o_d, lse_d = _run(q[:, :, -1].contiguous(), k, v, seqlens, 5)
    assert (o_d.float() - o_f[:, :, -1].float()).abs().max().item() <= 2e-2
    assert (lse_d - lse_f[:, :, -1]).abs().max().item() <= 1e-3


def _oracle_all_heads(q, kc, vc, seqlens):
    """The oracle for every (b, h), a batch entry's cache copied to the host at a
    time and its heads spread over a thread pool (the oracle's C code runs
    without the GIL); returns fp64 (o [B,H,d], lse [B,H])."""
    B, H, L, d = kc.shape
    sl = seqlens.cpu().tolist()
    qc = q.cpu()
    ref_o = np.empty((B, H, d))
    ref_l = np.empty((B, H))
    with ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1))) as ex:
        for b in range(B):
            n = int(sl[b])
            kb, vb = kc[b, :, :n].cpu(), vc[b, :, :n].cpu()

            def one(h, b=b, n=n, kb=kb, vb=vb):
                ro, rl = oracle.decode(qc[b:b + 1, h:h + 1], kb[h:h + 1].unsqueeze(0), vb[h:h + 1].unsqueeze(0), [n])
                return h, ro[0, 0], rl[0, 0]

            for h, ro, rl in ex.map(one, range(H)):
                ref_o[b, h] = ro
                ref_l[b, h] = rl
    return ref_o, ref_l


@pytest.mark.parametrize("name", ["decode_32k", "decode_32k_ragged"])
def test_full_size_every_head(name):
    """B=16, H=32, L=32768, d=128 with 8, 16 and 32 splits: the whole output of
    each split count (all 512 (b, h) rows) against the oracle."""
    c = wl.DECODE[name]
    q, kc, vc, seqlens = wl.decode_inputs(c.B, c.H, c.L, c.d, seed=0, ragged=c.ragged, device="cuda")
    outs = {s: _run(q, kc, vc, seqlens, s) for s in wl.DECODE_SPLITS}
    ref_o, ref_l = _oracle_all_heads(q, kc, vc, seqlens)
    for s, (o, lse) in outs.items():
        compare(o, lse, ref_o, ref_l, f"{name} S={s} (all {c.B * c.H} heads)")


def test_decode_rejects_bad_tensors():
    import exact_attention_29_gb300 as fa

    q = torch.zeros((1, 1, 128), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((1, 1, 16, 128), dtype=torch.bfloat16, device="cuda")
    sl = torch.ones(1, dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        fa.fa_decode(q, kc, kc, sl.long(), 2)
    with pytest.raises(fa.FaError) as e:
        fa.fa_decode(q, kc, kc, sl, 0)
    assert e.value.status == fa.FA_ERR_INVALID_ARG
