"""Softmax summaries and their combine operator, in plain Python/numpy fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

A segment of scores x_1..x_n (optionally with value rows v_j) is summarised by
  m = max_j x_j,  l = sum_j exp(x_j - m),  o = sum_j exp(x_j - m) v_j.
Two summaries combine as
  m = max(m_a, m_b)
  l = l_a exp(m_a - m) + l_b exp(m_b - m)
  o = o_a exp(m_a - m) + o_b exp(m_b - m)
and the softmax-weighted output of the union is o / l, its log-sum-exp m + ln l.

Sources:
  - CMU 15-779 Lecture 5 notes §4.2 (safe softmax, two passes), §4.3 (online
    softmax of Milakov & Gimelshein: keep (m, l), rebase l by exp(m - m_new)
    when the maximum grows; the number of rebases on random data is about
    ln N), §4.4 (the combine operator on (m, l), associative and commutative;
    Exercise 3), §4.5 (the triple (m, l, o) with the same rule, output o / l).
  - "已有的几种大模型上下文支持情况" (cicada blog) §2.3, frame 4:
    l_new = e^(m1 - m_new) l1 + e^(m2 - m_new) l2, and the matching update of
    the un-normalised output.

The empty segment is the identity element (m = -inf, l = 0, o = 0); the
combine never evaluates -inf - (-inf).
"""
from __future__ import annotations

import math

import numpy as np

NEG_INF = float("-inf")


def identity(d: int | None = None):
    """The summary of an empty segment."""
    return (NEG_INF, 0.0, None if d is None else np.zeros(d, dtype=np.float64))


def summarize(x, v=None):
    """Two-pass safe-softmax summary of one segment (m, l[, o])."""
    x = np.asarray(x, dtype=np.float64)
    if x.size == 0:
        return identity(None if v is None else np.asarray(v).shape[-1])
    m = float(np.max(x))
    e = np.exp(x - m)
    l = float(np.sum(e))
    if v is None:
        return (m, l, None)
    o = e @ np.asarray(v, dtype=np.float64)
    return (m, l, o)


def _weight(m_part: float, m: float) -> float:
    # exp(m_part - m) with the empty-segment convention exp(-inf - m) = 0
    if m_part == NEG_INF:
        return 0.0
    return math.exp(m_part - m)


def combine(a, b):
    """The combine operator on (m, l, o) summaries (o may be None)."""
    m_a, l_a, o_a = a
    m_b, l_b, o_b = b
    m = max(m_a, m_b)
    if m == NEG_INF:  # both empty
        return (NEG_INF, 0.0, o_a if o_a is not None else o_b)
    wa = _weight(m_a, m)
    wb = _weight(m_b, m)
    l = l_a * wa + l_b * wb
    o = None
    if o_a is not None or o_b is not None:
        o = (0.0 if o_a is None else o_a * wa) + (0.0 if o_b is None else o_b * wb)
    return (m, l, o)


def online(x):
    """One-pass online softmax over x, element by element.

    Returns (m, l, rebases): rebases counts the steps where the running
    maximum grew after the first element, i.e. l had to be rescaled.
    """
    m, l, rebases = NEG_INF, 0.0, 0
    for i, xi in enumerate(np.asarray(x, dtype=np.float64)):
        xi = float(xi)
        m_new = max(m, xi)
        if i > 0 and m_new > m:
            rebases += 1
        l = l * _weight(m, m_new) + math.exp(xi - m_new)
        m = m_new
    return m, l, rebases


def lse(summary) -> float:
    """Natural log-sum-exp of the segment a summary describes."""
    m, l, _ = summary
    if l == 0.0:
        return NEG_INF
    return m + math.log(l)


def output(summary):
    """The softmax-weighted value output o / l of a summary."""
    _, l, o = summary
    return o / l
