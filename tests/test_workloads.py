"""The seeded input generators both sides read (CPU only).

The CUDA path, the oracle and the benchmark all take their inputs from
`exact_attention_29_gb300.workloads`; these checks hold the generators to the
recipe its docstring states: fixed shapes per named workload, bf16 draws that
repeat for a seed and differ across seeds and tensors, standard-normal values
(so q.k has variance d, CMU 15-779 Lecture 5 notes §2.3), ragged cache lengths
in their stated range, and block masks with the band, global and random blocks
block-sparse attention serves ("FlashAttention 完全拆解（一）", block-sparse
extension).
"""
import pytest
import torch

from exact_attention_29_gb300 import workloads as wl


def test_named_shapes():
    shapes = {name: (c.B, c.H, c.N, c.d, c.causal) for name, c in wl.PREFILL.items()}
    assert shapes == {
        "pr1": (1, 1, 128, 64, False),
        "gpt2_small": (8, 12, 1024, 64, False),
        "gpt2_small_causal": (8, 12, 1024, 64, True),
        "llama3_8b_prefill": (2, 32, 4096, 128, True),
        "llama3_8b_prefill_noncausal": (2, 32, 4096, 128, False),
        "long_16k": (1, 32, 16384, 128, True),
        "long_64k": (1, 32, 65536, 128, True),
    }
    assert {n: (c.B, c.H, c.L, c.d, c.ragged) for n, c in wl.DECODE.items()} == {
        "decode_32k": (16, 32, 32768, 128, False),
        "decode_32k_ragged": (16, 32, 32768, 128, True),
    }
    assert wl.DECODE_SPLITS == (8, 16, 32)
    for c in wl.DECODE_GQA.values():
        assert c.Hq % c.Hkv == 0 and c.g == c.Hq // c.Hkv
    # matmul FLOPs: two N x N x d products of 2 FLOPs per multiply-add, halved under the mask
    c = wl.PREFILL["llama3_8b_prefill"]
    assert c.flops == 2 * 2 * c.B * c.H * c.N * c.N * c.d / 2
    assert c.scale == pytest.approx(128 ** -0.5)


def test_prefill_draws_repeat_per_seed_and_differ_otherwise():
    a = wl.prefill_inputs(2, 3, 100, 64, seed=5)
    b = wl.prefill_inputs(2, 3, 100, 64, seed=5)
    c = wl.prefill_inputs(2, 3, 100, 64, seed=6)
    for x, y, z in zip(a, b, c):
        assert x.dtype == torch.bfloat16 and x.shape == (2, 3, 100, 64)
        assert torch.equal(x, y)
        assert not torch.equal(x, z)
    q, k, v = a
    assert not torch.equal(q, k) and not torch.equal(k, v)
    # dO comes from its own stream: not a copy of Q, K or V of the same seed
    do = wl.backward_inputs(2, 3, 100, 64, seed=5)
    assert do.shape == q.shape and do.dtype == torch.bfloat16
    assert all(not torch.equal(do, t) for t in a)


def test_prefill_values_are_standard_normal():
    q, k, _ = wl.prefill_inputs(4, 8, 512, 64, seed=0)
    x = q.float()
    assert abs(x.mean().item()) < 0.01
    assert abs(x.std().item() - 1.0) < 0.01
    # the raw scores q.k then have variance close to d
    s = (q.float()[0, 0] @ k.float()[0, 0].T).flatten()
    assert abs(s.var().item() / 64 - 1.0) < 0.05


def test_decode_lengths():
    full = wl.decode_seqlens(16, 32768, seed=3)
    assert full.dtype == torch.int32 and torch.equal(full, torch.full((16,), 32768, dtype=torch.int32))
    r = wl.decode_seqlens(16, 32768, seed=3, ragged=True)
    assert r.dtype == torch.int32 and torch.equal(r, wl.decode_seqlens(16, 32768, seed=3, ragged=True))
    assert int(r.min()) >= 1024 and int(r.max()) <= 32768 and len(set(r.tolist())) > 1
    # a cache shorter than the lower bound: every length is the whole cache or less
    short = wl.decode_seqlens(8, 500, seed=1, ragged=True)
    assert int(short.min()) >= 500 and int(short.max()) <= 500


def test_decode_input_shapes():
    q, k, v, sl = wl.decode_inputs(3, 4, 300, 64, seed=2, ragged=True, lo=10)
    assert q.shape == (3, 4, 64) and k.shape == v.shape == (3, 4, 300, 64)
    assert sl.shape == (3,) and int(sl.min()) >= 10 and int(sl.max()) <= 300
    q, k, v, sl = wl.decode_gqa_inputs(2, 16, 2, 200, 128, seed=2)
    assert q.shape == (2, 16, 128) and k.shape == v.shape == (2, 2, 200, 128)
    assert torch.equal(sl, torch.full((2,), 200, dtype=torch.int32))


def test_block_mask_structure():
    T, heads = 32, 4
    m = wl.block_mask_bigbird(T, heads=heads, seed=0)
    assert m.dtype == torch.uint8 and m.shape == (heads, T, T)
    assert torch.equal(m, wl.block_mask_bigbird(T, heads=heads, seed=0))
    assert not torch.equal(m, wl.block_mask_bigbird(T, heads=heads, seed=1))
    i = torch.arange(T)
    band = (i[:, None] - i[None, :]).abs() <= 1
    assert bool(m[:, band].all())            # the band of +-1 block
    assert bool(m[:, 0, :].all()) and bool(m[:, :, 0].all())  # the global block row and column
    per_row = m[:, 1:, :].sum(dim=2)          # band (<= 3) + global column + up to 2 random blocks
    assert int(per_row.max()) <= 6 and int(per_row.min()) >= 3
    assert not torch.equal(m[0], m[1])       # each head draws its own random blocks
    density = m.float().mean().item()
    assert 0.18 < density < 0.24, density


def test_row_subsets():
    r = wl.row_subsets(2, 3, 1000, 256, seed=4)
    assert r.shape == (2, 3, 256) and r.dtype == torch.int64
    assert torch.equal(r, wl.row_subsets(2, 3, 1000, 256, seed=4))
    for b in range(2):
        for h in range(3):
            rows = r[b, h].tolist()
            assert len(set(rows)) == 256 and min(rows) >= 0 and max(rows) < 1000
    assert not torch.equal(r[0, 0], r[0, 1])
    # fewer rows than asked for: every row once
    small = wl.row_subsets(1, 1, 50, 256, seed=0)
    assert sorted(small[0, 0].tolist()) == list(range(50))
