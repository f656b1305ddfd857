"""Block-sparse prefill on the GPU (through the C ABI) against the fp64
block-mask attention oracle."""
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


def _random_mask(H, T, seed, density=0.5, empty_row=True):
    g = torch.Generator().manual_seed(seed)
    m = (torch.rand((H, T, T), generator=g) < density).to(torch.uint8)
    if empty_row and T > 1:
        m[:, T - 1, :] = 0  # the last block row sees nothing: o = 0, lse = -inf
    return m


def _compare_sparse(o, lse, o_ref, lse_ref, what):
    lse_g = lse.cpu().numpy()
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse_g), empty), f"{what}: empty rows differ"
    assert np.all(o.float().cpu().numpy()[empty] == 0), f"{what}: empty rows must be 0"
    keep = ~empty
    if keep.any():
        compare(o.cpu()[torch.from_numpy(keep)], lse.cpu()[torch.from_numpy(keep)], o_ref[keep], lse_ref[keep], what)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 7, 128, 129, 300, 700])
def test_small_shapes_random_masks(N, d, causal):
    import exact_attention_29_gb300 as fa

    B, H = 2, 2
    T = (N + 127) // 128
    q, k, v = wl.prefill_inputs(B, H, N, d, seed=N + d + 1)
    mask = _random_mask(H, T, seed=N + d)
    o, lse = fa.fa_fwd_sparse(q.cuda(), k.cuda(), v.cuda(), mask.cuda(), causal=causal)
    fa.fa_check_device_error()
    o_ref, lse_ref = oracle.attention_block_mask(q, k, v, mask, causal, d ** -0.5)
    _compare_sparse(o, lse, o_ref, lse_ref, f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_all_ones_mask_equals_the_dense_kernel_bitwise(causal):
    """A step the mask removes for one Q tile of a pair adds exact zeros, so with
    every block kept the result is the dense kernel's, bit for bit."""
    import exact_attention_29_gb300 as fa

    q, k, v = wl.prefill_inputs(1, 4, 1000, 128, seed=5)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    mask = torch.ones((8, 8), dtype=torch.uint8, device="cuda")
    o1, l1 = fa.fa_fwd_sparse(q, k, v, mask, causal=causal)
    o2, l2 = fa.fa_fwd(q, k, v, causal=causal)
    fa.fa_check_device_error()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_one_mask_shared_by_all_heads():
    import exact_attention_29_gb300 as fa

    q, k, v = wl.prefill_inputs(2, 3, 520, 64, seed=8)
    mask = _random_mask(1, 5, seed=3, empty_row=False)[0]
    o, lse = fa.fa_fwd_sparse(q.cuda(), k.cuda(), v.cuda(), mask.cuda())
    fa.fa_check_device_error()
    o_ref, lse_ref = oracle.attention_block_mask(q, k, v, mask, False, 64 ** -0.5)
    _compare_sparse(o, lse, o_ref, lse_ref, "shared mask")


def test_bigbird_llama_shape_sampled_heads():
    """Full size (B2 H32 N4096 d128, non-causal) under the band + global + random
    mask, one mask per head; the oracle checks two whole heads."""
    import exact_attention_29_gb300 as fa

    c = wl.SPARSE_PREFILL
    T = c.N // 128
    q, k, v = wl.prefill_inputs(c.B, c.H, c.N, c.d, seed=0, device="cuda")
    mask = wl.block_mask_bigbird(T, heads=c.H, seed=0)
    o, lse = fa.fa_fwd_sparse(q, k, v, mask.cuda(), causal=c.causal)
    fa.fa_check_device_error()
    for b, h in ((0, 3), (1, 30)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        o_ref, lse_ref = oracle.attention_block_mask(q[sl].cpu(), k[sl].cpu(), v[sl].cpu(), mask[h], c.causal, c.scale)
        _compare_sparse(o[sl], lse[sl], o_ref, lse_ref, f"bigbird head ({b},{h})")


def _mixed_mask(H, T, seed):
    """Per block row a different kind: dense, empty, one block, a random
    density, a band; so the two Q tiles of a pair often keep very different
    numbers of K/V tiles, share few of them, or one keeps none."""
    g = torch.Generator().manual_seed(seed)
    m = torch.zeros((H, T, T), dtype=torch.uint8)
    for h in range(H):
        for i in range(T):
            kind = int(torch.randint(0, 5, (1,), generator=g))
            if kind == 0:
                m[h, i, :] = 1
            elif kind == 2:
                m[h, i, int(torch.randint(0, T, (1,), generator=g))] = 1
            elif kind == 3:
                dens = float(torch.rand((1,), generator=g))
                m[h, i] = (torch.rand((T,), generator=g) < dens).to(torch.uint8)
            elif kind == 4:
                m[h, i, max(0, i - 2): i + 3] = 1
    return m


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_mixed_row_masks_many_tiles(d, causal):
    """B1 H4 N4000 (32 tiles, a ragged last one): long private runs on one tile
    of a pair and short ones on the other, rows that keep nothing next to rows
    that keep everything; every head against the oracle."""
    import exact_attention_29_gb300 as fa

    B, H, N = 1, 4, 4000
    T = (N + 127) // 128
    q, k, v = wl.prefill_inputs(B, H, N, d, seed=17 + d)
    mask = _mixed_mask(H, T, seed=d + int(causal))
    o, lse = fa.fa_fwd_sparse(q.cuda(), k.cuda(), v.cuda(), mask.cuda(), causal=causal)
    fa.fa_check_device_error()
    o_ref, lse_ref = oracle.attention_block_mask(q, k, v, mask, causal, d ** -0.5)
    _compare_sparse(o, lse, o_ref, lse_ref, f"mixed rows d={d} causal={causal}")
