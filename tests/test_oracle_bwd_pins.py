"""The fp64 backward oracle against its pins (CPU only).

Sources: CMU 15-779 Lecture 5 notes §7.1-7.4 (chain rule through the softmax
Jacobian, D_i = dO_i . O_i, dS = P (dP - D)); the gradients are pinned against
central finite differences of the separately pinned forward oracle.
"""
import numpy as np
import pytest

import oracle


def _loss(q, k, v, w, causal, scale):
    o, _ = oracle.attention(q, k, v, causal, scale)
    return float(np.sum(o * w))


def _fd_grad(q, k, v, w, causal, scale, which, h=1e-6):
    x = {"q": q, "k": k, "v": v}[which]
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        old = x[idx]
        x[idx] = old + h
        lp = _loss(q, k, v, w, causal, scale)
        x[idx] = old - h
        lm = _loss(q, k, v, w, causal, scale)
        x[idx] = old
        g[idx] = (lp - lm) / (2 * h)
    return g


@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_finite_differences(causal):
    r = np.random.default_rng(31 + causal)
    B, H, N, d = 1, 2, 6, 3
    q, k, v, w = (r.standard_normal((B, H, N, d)) for _ in range(4))
    scale = 0.7
    dq, dk, dv = oracle.attention_bwd(q, k, v, w, causal, scale)
    for name, got in (("q", dq), ("k", dk), ("v", dv)):
        fd = _fd_grad(q, k, v, w, causal, scale, name)
        assert np.max(np.abs(got - fd)) <= 1e-7 * max(1.0, np.max(np.abs(fd))), name


def test_identical_keys_give_zero_dq():
    """Rows of dS sum to zero (softmax Jacobian), so dQ = scale dS K vanishes when
    every key is the same vector."""
    r = np.random.default_rng(32)
    N, d = 7, 5
    q, v, w = (r.standard_normal((1, 1, N, d)) for _ in range(3))
    k = np.tile(r.standard_normal(d), (1, 1, N, 1))
    for causal in (False, True):
        dq, _, _ = oracle.attention_bwd(q, k, v, w, causal, 0.9)
        assert np.max(np.abs(dq)) <= 1e-13


def test_constant_upstream_gradient_dv_sums():
    """With every row of dO equal to c, dV_j = (sum_i P_ij) c, so sum_j dV_j = N c."""
    r = np.random.default_rng(33)
    N, d = 8, 4
    q, k, v = (r.standard_normal((1, 1, N, d)) for _ in range(3))
    c = r.standard_normal(d)
    w = np.tile(c, (1, 1, N, 1))
    for causal in (False, True):
        _, _, dv = oracle.attention_bwd(q, k, v, w, causal, 0.5)
        assert np.allclose(dv[0, 0].sum(0), N * c, rtol=0, atol=1e-12)


def test_causal_last_key_is_seen_by_the_last_query_only():
    """Under the causal mask key N-1 is visible to query N-1 alone:
    dV_{N-1} = P_{N-1,N-1} dO_{N-1}."""
    r = np.random.default_rng(34)
    N, d = 6, 4
    q, k, v, w = (r.standard_normal((1, 1, N, d)) for _ in range(4))
    _, _, dv = oracle.attention_bwd(q, k, v, w, True, 0.8)
    _, _, _, p = oracle.attention_rows(q[0, 0], np.arange(N), k[0, 0], v[0, 0], True, 0.8, want_sp=True)
    assert np.allclose(dv[0, 0, N - 1], p[N - 1, N - 1] * w[0, 0, N - 1], atol=1e-14)


def _bwd_mutant(q, k, v, w, causal, scale, mistake):
    """numpy restatement of the backward with one planted mistake."""
    q, k, v, w = (np.asarray(x[0, 0], dtype=np.float64) for x in (q, k, v, w))
    n = q.shape[0]
    s = scale * q @ k.T
    if causal:
        s = np.where(np.triu(np.ones((n, n), bool), 1), -np.inf, s)
    p = np.exp(s - s.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    dp = w @ v.T
    D = (p * dp).sum(1, keepdims=True)
    if mistake == "D_sign":
        D = -D
    ds = p * (dp - D)
    if mistake == "dS_transposed":
        ds = ds.T
    dq = scale * ds @ k
    if mistake == "dq_no_scale":
        dq = ds @ k
    return dq[None, None]


@pytest.mark.parametrize("mistake", ["D_sign", "dS_transposed", "dq_no_scale"])
def test_planted_backward_mistakes_fail_finite_differences(mistake):
    r = np.random.default_rng(35)
    q, k, v, w = (r.standard_normal((1, 1, 5, 3)) for _ in range(4))
    fd = _fd_grad(q, k, v, w, False, 0.7, "q")
    bad = _bwd_mutant(q, k, v, w, False, 0.7, mistake)
    good = _bwd_mutant(q, k, v, w, False, 0.7, None)
    assert np.max(np.abs(good - fd)) <= 1e-7
    assert np.max(np.abs(bad - fd)) > 1e-3
