"""The fp64 block-mask attention oracle against its pins (CPU only).

"FlashAttention 完全拆解（一）", block-sparse extension: scores of blocks the
block mask removes take no part in the softmax. Pinned to the dense oracle
(all-ones mask, and a lower-triangular mask under the causal mask), to
independent attention over each diagonal block (a block-diagonal mask splits
the sequence into independent pieces), to a numpy evaluation, and to the empty
row convention.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_29_gb300 import workloads as wl


@pytest.fixture(scope="module", autouse=True)
def _build():
    oracle.build()


@pytest.mark.parametrize("causal", [False, True])
def test_all_ones_mask_is_dense_attention(causal):
    q, k, v = wl.prefill_inputs(1, 2, 70, 16, seed=1)
    mask = np.ones((5, 5), np.uint8)
    o, lse = oracle.attention_block_mask(q, k, v, mask, causal, 0.25, block=16)
    o_ref, lse_ref = oracle.attention(q, k, v, causal, 0.25)
    np.testing.assert_allclose(o, o_ref, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, atol=1e-13)


def test_lower_triangular_blocks_under_causal_equal_causal():
    q, k, v = wl.prefill_inputs(1, 1, 64, 8, seed=2)
    mask = np.tril(np.ones((4, 4), np.uint8))
    o, lse = oracle.attention_block_mask(q, k, v, mask, True, 0.3, block=16)
    o_ref, lse_ref = oracle.attention(q, k, v, True, 0.3)
    np.testing.assert_allclose(o, o_ref, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, atol=1e-13)


def test_block_diagonal_mask_splits_the_sequence():
    q, k, v = wl.prefill_inputs(1, 2, 48, 8, seed=3)
    o, lse = oracle.attention_block_mask(q, k, v, np.eye(3, dtype=np.uint8), False, 0.5, block=16)
    for blk in range(3):
        sl = slice(16 * blk, 16 * blk + 16)
        ro, rl = oracle.attention(q[:, :, sl], k[:, :, sl], v[:, :, sl], False, 0.5)
        np.testing.assert_allclose(o[:, :, sl], ro, atol=1e-13)
        np.testing.assert_allclose(lse[:, :, sl], rl, atol=1e-13)


def test_numpy_brute_force_with_per_head_masks():
    B, H, N, d, blk = 1, 2, 20, 4, 8
    q, k, v = wl.prefill_inputs(B, H, N, d, seed=4)
    g = np.random.default_rng(5)
    mask = (g.random((H, 3, 3)) < 0.6).astype(np.uint8)
    mask[:, np.arange(3), np.arange(3)] = 1
    o, lse = oracle.attention_block_mask(q, k, v, mask, False, 0.7, block=blk)
    qn, kn, vn = (t.double().numpy() for t in (q, k, v))
    for h in range(H):
        for i in range(N):
            vis = np.array([mask[h, i // blk, j // blk] for j in range(N)], bool)
            s = qn[0, h, i] @ kn[0, h, vis].T * 0.7
            w = np.exp(s - s.max())
            np.testing.assert_allclose(o[0, h, i], (w / w.sum()) @ vn[0, h, vis], atol=1e-12)
            np.testing.assert_allclose(lse[0, h, i], s.max() + np.log(w.sum()), atol=1e-12)


def test_rows_with_no_visible_key():
    q, k, v = wl.prefill_inputs(1, 1, 32, 8, seed=6)
    mask = np.array([[1, 0], [0, 0]], np.uint8)
    o, lse = oracle.attention_block_mask(q, k, v, mask, False, 0.5, block=16)
    assert np.all(o[0, 0, 16:] == 0) and np.all(np.isneginf(lse[0, 0, 16:]))
    assert np.all(np.isfinite(lse[0, 0, :16]))
