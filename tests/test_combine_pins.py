"""The oracle's (m, l, o) summaries and combine operator against their pins (CPU only).

Sources: CMU 15-779 Lecture 5 notes §4.2-4.5 and Exercise 3; the printed
numbers are in tests/golden/online_softmax.json.
"""
import functools
import json
import math
import os
from decimal import Decimal, getcontext

import numpy as np
import pytest

from oracle import combine as cb

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden():
    with open(os.path.join(GOLDEN, "online_softmax.json")) as f:
        return json.load(f)


def _decimal_lse(x):
    getcontext().prec = 50
    return float(sum((Decimal(float(t)).exp() for t in x), Decimal(0)).ln())


def _fold(parts):
    return functools.reduce(cb.combine, parts, cb.identity())


def test_every_single_cut_equals_two_pass():
    r = np.random.default_rng(21)
    x = r.standard_normal(64) * 5
    ref = cb.summarize(x)
    for cut in range(0, len(x) + 1):
        got = cb.combine(cb.summarize(x[:cut]), cb.summarize(x[cut:]))
        assert got[0] == ref[0]
        assert abs(got[1] - ref[1]) <= 1e-13 * ref[1]


def test_every_split_of_a_short_row():
    """All 2^(n-1) ways of cutting a row of 10 into contiguous blocks."""
    r = np.random.default_rng(22)
    x = r.standard_normal(10) * 4
    ref = cb.lse(cb.summarize(x))
    n = len(x)
    for mask in range(1 << (n - 1)):
        cuts = [0] + [i + 1 for i in range(n - 1) if mask >> i & 1] + [n]
        parts = [cb.summarize(x[a:b]) for a, b in zip(cuts[:-1], cuts[1:])]
        assert abs(cb.lse(_fold(parts)) - ref) <= 1e-13 * max(1, abs(ref))


def test_four_merge_orders_match_decimal():
    """10000 numbers merged left to right, in 7 uneven blocks, as a pairwise tree
    and as shuffled blocks: all equal the 50-digit log-sum-exp within the page's
    fp64 figure's order of magnitude."""
    g = _golden()["combine"]
    r = np.random.default_rng(23)
    x = r.standard_normal(g["n"]) * 3
    exact = _decimal_lse(x)
    one = [cb.summarize(x[i:i + 1]) for i in range(len(x))]
    left = _fold(one)
    cuts = np.sort(r.choice(np.arange(1, len(x)), g["blocks"] - 1, replace=False))
    blocks = [cb.summarize(b) for b in np.split(x, cuts)]
    seven = _fold(blocks)
    level, depth = one, 0
    while len(level) > 1:
        level = [cb.combine(level[i], level[i + 1]) if i + 1 < len(level) else level[i]
                 for i in range(0, len(level), 2)]
        depth += 1
    assert depth == g["tree_levels"]
    tree = level[0]
    shuffled = _fold([blocks[i] for i in r.permutation(len(blocks))])
    for s in (left, seven, tree, shuffled):
        # the page reports 3.6e-15 max difference at this size; allow 10x for order
        assert abs(cb.lse(s) - exact) <= 10 * g["max_abs_diff_printed"] * max(1, abs(exact))


def test_triple_combine_equals_weighted_output():
    """(m, l, o) summaries of blocks combine to softmax(x) @ V (Lecture 5 notes §4.5)."""
    r = np.random.default_rng(24)
    x = r.standard_normal(50) * 6
    v = r.standard_normal((50, 7))
    w = np.exp(x - x.max())
    ref = (w / w.sum()) @ v
    for cuts in ([25], [1, 2, 3, 40], [10, 20, 30, 40, 49]):
        parts = [cb.summarize(xs, vs) for xs, vs in zip(np.split(x, cuts), np.split(v, cuts))]
        got = cb.output(_fold(parts))
        assert np.max(np.abs(got - ref)) <= 1e-13


def test_associative_and_commutative():
    r = np.random.default_rng(25)
    a, b, c = (cb.summarize(r.standard_normal(9) * 7, r.standard_normal((9, 3))) for _ in range(3))
    lhs = cb.combine(cb.combine(a, b), c)
    rhs = cb.combine(a, cb.combine(b, c))
    comm = cb.combine(b, a)
    ab = cb.combine(a, b)
    assert lhs[0] == rhs[0] and abs(lhs[1] - rhs[1]) <= 1e-13 * lhs[1]
    assert np.max(np.abs(lhs[2] - rhs[2])) <= 1e-12 * np.max(np.abs(lhs[2]))
    assert comm[0] == ab[0] and abs(comm[1] - ab[1]) <= 1e-14 * ab[1]


def test_empty_segment_is_identity():
    r = np.random.default_rng(26)
    s = cb.summarize(r.standard_normal(5), r.standard_normal((5, 2)))
    e = cb.identity(2)
    for got in (cb.combine(s, e), cb.combine(e, s)):
        assert got[0] == s[0] and got[1] == s[1] and np.array_equal(got[2], s[2])
    both = cb.combine(cb.identity(2), cb.identity(2))
    assert both[0] == float("-inf") and both[1] == 0.0 and cb.lse(both) == float("-inf")


def test_online_equals_two_pass():
    r = np.random.default_rng(27)
    x = r.standard_normal(500) * 10
    m, l, _ = cb.online(x)
    m2, l2, _ = cb.summarize(x)
    assert m == m2 and abs(l - l2) <= 1e-13 * l2


def test_online_rebase_count_is_about_ln_n():
    """On random data the running max is rebased about sum_{k=2}^N 1/k times;
    the page prints 7.9 for N = 4096."""
    g = _golden()["rebases"]
    n = g["N"]
    expected = sum(1.0 / k for k in range(2, n + 1))
    assert abs(expected - g["expected_printed"]) < 0.05
    r = np.random.default_rng(28)
    counts = [cb.online(r.standard_normal(n))[2] for _ in range(60)]
    mean = float(np.mean(counts))
    # standard deviation of the count is about sqrt(ln N) ~ 2.4; 60 runs -> ~0.3
    assert abs(mean - expected) < 1.5, mean


def test_combine_matches_decimal_with_huge_offsets():
    """Segments whose maxima differ by hundreds still combine exactly (no overflow)."""
    x = np.concatenate([np.linspace(-5, 5, 20) + 800.0, np.linspace(-5, 5, 20) - 600.0])
    parts = [cb.summarize(x[:20]), cb.summarize(x[20:])]
    assert abs(cb.lse(_fold(parts)) - _decimal_lse(x)) < 1e-12 * 800
