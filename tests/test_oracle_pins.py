"""The fp64 oracle against its pins (CPU only)."""
import json
import math
import os

import numpy as np
import pytest

import pins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _impl(oracle_mod):
    def impl(q, pos, k, v, causal, scale):
        return oracle_mod.attention_rows(q, pos, k, v, causal, scale, want_sp=True)

    return impl


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(oracle_mod, pin):
    msg = pin(_impl(oracle_mod))
    assert msg is None, msg


def test_batched_matches_rows(oracle_mod):
    """The batched entry point is the per-head row entry point over every head."""
    r = np.random.default_rng(11)
    B, H, N, d = 2, 3, 19, 8
    q, k, v = (r.standard_normal((B, H, N, d)) for _ in range(3))
    for causal in (False, True):
        o, lse = oracle_mod.attention(q, k, v, causal, 0.37)
        for b in range(B):
            for h in range(H):
                o1, l1, _, _ = oracle_mod.attention_rows(q[b, h], np.arange(N), k[b, h], v[b, h], causal, 0.37)
                assert np.array_equal(o[b, h], o1) and np.array_equal(lse[b, h], l1)


def test_row_subset_equals_full_rows(oracle_mod):
    """Evaluating a subset of rows (with their positions) gives those rows of the full result."""
    r = np.random.default_rng(12)
    N, d = 40, 8
    q, k, v = (r.standard_normal((N, d)) for _ in range(3))
    rows = np.array([39, 0, 17, 5])
    o_full, l_full, _, _ = oracle_mod.attention_rows(q, np.arange(N), k, v, True, 0.5)
    o_sub, l_sub, _, _ = oracle_mod.attention_rows(q[rows], rows, k, v, True, 0.5)
    assert np.array_equal(o_sub, o_full[rows]) and np.array_equal(l_sub, l_full[rows])


def test_decode_equals_last_causal_row(oracle_mod):
    """A cached decode step equals the last row of the causal prefill over the same
    sequence (CMU 15-779 Lecture 5 notes §8.2)."""
    r = np.random.default_rng(13)
    B, H, L, d = 2, 2, 33, 16
    kc, vc = r.standard_normal((B, H, L, d)), r.standard_normal((B, H, L, d))
    q = r.standard_normal((B, H, d))
    seqlens = np.array([33, 7])
    o, lse = oracle_mod.decode(q, kc, vc, seqlens)
    for b in range(B):
        n = int(seqlens[b])
        for h in range(H):
            qq = np.concatenate([r.standard_normal((n - 1, d)), q[b, h][None]], 0)
            op, lp, _, _ = oracle_mod.attention_rows(qq, np.arange(n), kc[b, h, :n], vc[b, h, :n], True, d ** -0.5)
            assert np.allclose(o[b, h], op[-1], rtol=0, atol=1e-14)
            assert abs(lse[b, h] - lp[-1]) <= 1e-14 * max(1, abs(lp[-1]))


def test_no_overflow_on_large_scores(oracle_mod):
    """Scores far beyond exp's range (x > 709 in fp64) stay finite: the row max is
    subtracted first (cicada blog §1.3; Lecture 5 notes §4.1-4.2)."""
    q = np.array([[30.0, 0.0], [0.0, 30.0]])
    k = np.array([[30.0, 0.0], [29.0, 1.0]])
    v = np.array([[1.0, 0.0], [0.0, 1.0]])
    o, lse, _, _ = oracle_mod.attention_rows(q, np.arange(2), k, v, False, 1.0)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    # row 0: scores 900, 870 -> weights 1/(1+e^-30), e^-30/(1+e^-30)
    w = 1 / (1 + math.exp(-30))
    assert np.allclose(o[0], [w, 1 - w], atol=1e-15)
    assert abs(lse[0] - (900 + math.log1p(math.exp(-30)))) < 1e-12


def test_oracle_rejects_bad_arguments(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.attention_rows(np.zeros((2, 3)), None, np.zeros((2, 3)), np.zeros((2, 3)), True, 1.0)
    with pytest.raises(RuntimeError):
        oracle_mod.decode(np.zeros((1, 1, 4)), np.zeros((1, 1, 5, 4)), np.zeros((1, 1, 5, 4)), np.array([6]))


def test_golden_fixtures_are_cited():
    for name in os.listdir(GOLDEN):
        if name.endswith(".json"):
            with open(os.path.join(GOLDEN, name)) as f:
                data = json.load(f)
            assert "source" in data and len(data["source"]) > 20, name
