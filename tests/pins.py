"""Pins for the attention oracle: checks against what the pages and mathematics fix.

Each pin takes an implementation ``impl(q_rows, q_pos, k, v, causal, scale)``
returning ``(o, lse, s, p)`` (s = scaled, masked scores; p = probabilities)
and returns None when it holds, or a message when it does not. The real
oracle must satisfy all of them; ``test_oracle_mutants.py`` plants plausible
mistakes in copies of the method and checks that each one breaks a pin.

Sources of the facts pinned:
  - rows of P sum to 1 with entries in [0, 1]: cicada blog
    "已有的几种大模型上下文支持情况" §1.3 step 3;
  - masked weights are exactly 0: CMU 15-779 Lecture 5 notes §2.3;
  - the output is a convex combination of value rows (constant V, one-hot
    dominant "hard lookup"): Lecture 5 notes §2.2;
  - softmax is unchanged by a per-row shift: Lecture 5 notes §4.2;
  - P = exp(S - L): Lecture 5 notes §7.2 and cicada blog §3.2.3;
  - the N = 4 worked example: the cicada blog §1.3 walks through N = 4 words
    without printing values; the instance below is solved in closed form.
"""
from __future__ import annotations

import math

import numpy as np

from _brute import attention_decimal

TOL = 1e-13


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, tol=TOL):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.shape != b.shape:
        return False
    if not np.all(np.isfinite(a)):
        return False
    return bool(np.max(np.abs(a - b)) <= tol * max(1.0, float(np.max(np.abs(b)))))


def worked_example():
    """Q = K = I_4, V rows (1,2), (3,4), (5,6), (7,8) padded to d = 4, scale 1.

    Then S = I. Non-causal: P_ii = e/(e+3), P_ij = 1/(e+3), LSE_i = ln(e+3).
    Causal: row i sees keys 0..i with scores (0,..,0,1): P_ii = e/(e+i),
    P_ij = 1/(e+i) for j < i, LSE_i = ln(e+i).
    """
    e = math.e
    q = np.eye(4)
    k = np.eye(4)
    v = np.array([[1, 2, 0, 0], [3, 4, 0, 0], [5, 6, 0, 0], [7, 8, 0, 0]], dtype=np.float64)
    vrows = v[:, :2]
    o_nc = np.array([(e * vrows[i] + (vrows.sum(0) - vrows[i])) / (e + 3) for i in range(4)])
    lse_nc = np.full(4, math.log(e + 3))
    o_c = np.array([(e * vrows[i] + vrows[:i].sum(0)) / (e + i) for i in range(4)])
    lse_c = np.array([math.log(e + i) for i in range(4)])
    return q, k, v, (o_nc, lse_nc), (o_c, lse_c)


def pin_worked_example(impl):
    q, k, v, (o_nc, lse_nc), (o_c, lse_c) = worked_example()
    pos = np.arange(4)
    for causal, o_ref, lse_ref in ((False, o_nc, lse_nc), (True, o_c, lse_c)):
        o, lse, _, _ = impl(q, pos, k, v, causal, 1.0)
        if not (_close(o[:, :2], o_ref, 1e-14) and _close(o[:, 2:], np.zeros((4, 2)), 1e-14)):
            return f"worked example O wrong (causal={causal}): {o[:, :2]} vs {o_ref}"
        if not _close(lse, lse_ref, 1e-14):
            return f"worked example LSE wrong (causal={causal}): {lse} vs {lse_ref}"
    return None


def pin_rows_sum_to_one(impl):
    r = _rng(1)
    n, d = 24, 16
    q, k, v = r.standard_normal((n, d)), r.standard_normal((n, d)), r.standard_normal((n, d))
    for causal in (False, True):
        _, _, _, p = impl(q, np.arange(n), k, v, causal, 1 / math.sqrt(d))
        if not np.all(np.isfinite(p)):
            return "P has non-finite entries"
        if np.min(p) < 0 or np.max(p) > 1:
            return "P entries outside [0, 1]"
        if np.max(np.abs(p.sum(1) - 1)) > 1e-14:
            return f"P rows do not sum to 1 (causal={causal})"
    return None


def pin_masked_exactly_zero(impl):
    r = _rng(2)
    n, d = 20, 8
    q, k, v = r.standard_normal((n, d)), r.standard_normal((n, d)), r.standard_normal((n, d))
    _, _, _, p = impl(q, np.arange(n), k, v, True, 1 / math.sqrt(d))
    upper = np.triu(np.ones((n, n), dtype=bool), 1)
    if not np.all(p[upper] == 0.0):
        return "causal: weights above the diagonal are not exactly 0"
    if not np.all(p[~upper] > 0.0):
        return "causal: a visible weight is 0"
    return None


def pin_constant_v(impl):
    r = _rng(3)
    n, d = 17, 8
    q, k = r.standard_normal((n, d)) * 3, r.standard_normal((n, d)) * 3
    c = r.standard_normal(d)
    v = np.tile(c, (n, 1))
    for causal in (False, True):
        o, _, _, _ = impl(q, np.arange(n), k, v, causal, 1 / math.sqrt(d))
        if not _close(o, v, 1e-14):
            return f"constant V not reproduced (causal={causal})"
    return None


def pin_one_hot_dominant(impl):
    """Key j* = 400 q_i makes row i's score (about 1600) exceed every other by
    far more than exp can bridge: O_i = v_j* and LSE_i = that score. The score
    is large enough that exp without the max subtraction overflows in fp64."""
    r = _rng(4)
    n, d = 12, 16
    q, k, v = r.standard_normal((n, d)), r.standard_normal((n, d)), r.standard_normal((n, d))
    i, js = 5, 9
    k[js] = 400.0 * q[i]
    o, lse, _, _ = impl(q, np.arange(n), k, v, False, 1 / math.sqrt(d))
    if not _close(o[i], v[js], 1e-14):
        return "one-hot dominant row does not reproduce its value row"
    s_star = float(q[i] @ k[js]) / math.sqrt(d)
    if abs(lse[i] - s_star) > 1e-12 * abs(s_star):
        return "one-hot dominant row: LSE is not the dominant score"
    return None


def pin_brute_force(impl):
    r = _rng(5)
    for n, d, causal in ((1, 1, False), (3, 2, True), (5, 4, False), (8, 8, True), (7, 3, False), (6, 8, True)):
        q = r.standard_normal((n, d))
        k = r.standard_normal((n, d))
        v = r.standard_normal((n, d))
        o, lse, _, _ = impl(q, np.arange(n), k, v, causal, 1 / math.sqrt(d))
        od, lsed = attention_decimal(q, k, v, causal, scale_sq_inv=d)
        od = np.array([[float(x) for x in row] for row in od])
        lsed = np.array([float(x) for x in lsed])
        if not (_close(o, od) and _close(lse, lsed)):
            return f"disagrees with the 50-digit brute force at n={n}, d={d}, causal={causal}"
    return None


def pin_key_shift(impl):
    """Adding the same vector u to every key adds q_i.u to row i: P and O unchanged, LSE shifts."""
    r = _rng(6)
    n, d = 16, 8
    q, k, v = r.standard_normal((n, d)), r.standard_normal((n, d)), r.standard_normal((n, d))
    u = r.standard_normal(d)
    sc = 1 / math.sqrt(d)
    for causal in (False, True):
        o1, l1, _, p1 = impl(q, np.arange(n), k, v, causal, sc)
        o2, l2, _, p2 = impl(q, np.arange(n), k + u, v, causal, sc)
        if not (_close(o1, o2, 1e-12) and _close(p1, p2, 1e-12)):
            return "row shift changed P or O"
        if not _close(l2 - l1, sc * (q @ u), 1e-12):
            return "row shift did not shift LSE by the shift"
    return None


def pin_permutation(impl):
    r = _rng(7)
    n, d = 15, 8
    q, k, v = r.standard_normal((n, d)), r.standard_normal((n, d)), r.standard_normal((n, d))
    perm = r.permutation(n)
    o1, l1, _, _ = impl(q, np.arange(n), k, v, False, 0.3)
    o2, l2, _, _ = impl(q, np.arange(n), k[perm], v[perm], False, 0.3)
    if not (_close(o1, o2, 1e-13) and _close(l1, l2, 1e-13)):
        return "jointly permuting keys and values changed the result"
    return None


def pin_causal_row0(impl):
    r = _rng(8)
    n, d = 9, 8
    q, k, v = r.standard_normal((n, d)), r.standard_normal((n, d)), r.standard_normal((n, d))
    sc = 1 / math.sqrt(d)
    o, lse, _, _ = impl(q, np.arange(n), k, v, True, sc)
    if not np.array_equal(o[0], v[0]):
        return "causal row 0 is not exactly V_0"
    if abs(lse[0] - sc * float(q[0] @ k[0])) > 1e-14 * max(1.0, abs(lse[0])):
        return "causal row 0 LSE is not the single score"
    return None


def pin_lse_consistency(impl):
    r = _rng(9)
    n, d = 20, 16
    q, k, v = r.standard_normal((n, d)), r.standard_normal((n, d)), r.standard_normal((n, d))
    for causal in (False, True):
        _, lse, s, p = impl(q, np.arange(n), k, v, causal, 1 / math.sqrt(d))
        if not _close(np.exp(s - lse[:, None]), p, 1e-14):
            return "exp(S - LSE) does not reproduce P"
    return None


ALL_PINS = [
    pin_worked_example,
    pin_rows_sum_to_one,
    pin_masked_exactly_zero,
    pin_constant_v,
    pin_one_hot_dominant,
    pin_brute_force,
    pin_key_shift,
    pin_permutation,
    pin_causal_row0,
    pin_lse_consistency,
]
