"""Planted mistakes: each plausible error in the standard-attention steps must
break at least one oracle pin (CPU only).

The mutants are small numpy restatements of the four standard-attention steps
with exactly one mistake each. They show that the pins in ``pins.py`` are
strong enough to catch a dropped term, a wrong sign or index, or a transposed
operand anywhere in the oracle.
"""
import math

import numpy as np
import pytest

import pins


def _standard(q, pos, k, v, causal, scale, mistake=None):
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n, nk = q.shape[0], k.shape[0]
    pos = np.arange(n) if pos is None else np.asarray(pos)
    s = -(q @ k.T) if mistake == "sign" else q @ k.T
    if mistake != "no_scale":
        s = s * scale
    if causal:
        j = np.arange(nk)[None, :]
        i = pos[:, None]
        if mistake == "mask_diagonal":
            s = np.where(j >= i, -np.inf, s)
        elif mistake == "mask_zero":
            s = np.where(j > i, 0.0, s)
        elif mistake == "mask_transposed":
            s = np.where(j < i, -np.inf, s)
        else:
            s = np.where(j > i, -np.inf, s)
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        if mistake == "no_max":
            m = np.zeros((n, 1))
        elif mistake == "column_softmax":
            m = s.max(0, keepdims=True)
        else:
            m = s.max(1, keepdims=True)
        e = np.exp(s - m)
        l = e.sum(0, keepdims=True) if mistake == "column_softmax" else e.sum(1, keepdims=True)
        p = e / l
        if mistake == "o_from_k":
            o = p @ k
        elif mistake == "no_divide":
            o = e @ v
        elif mistake == "v_reversed":
            o = p @ v[::-1]
        else:
            o = p @ v
        if mistake == "column_softmax":
            lse = np.log(e.sum(1)) + m.ravel()[: n] if n == nk else np.log(e.sum(1))
        else:
            mm = m.ravel()
            ll = l.ravel()
            if mistake == "lse_log2":
                lse = mm + np.log2(ll)
            elif mistake == "lse_no_max":
                lse = np.log(ll)
            else:
                lse = mm + np.log(ll)
    return o, lse, s, p


MISTAKES = ["sign", "no_scale", "mask_diagonal", "mask_zero", "mask_transposed", "no_max",
            "column_softmax", "o_from_k", "no_divide", "v_reversed", "lse_log2", "lse_no_max"]


def _run_pins(impl):
    failed = []
    for pin in pins.ALL_PINS:
        try:
            msg = pin(impl)
        except Exception as exc:  # a crash counts as a caught mistake
            msg = f"raised {exc!r}"
        if msg is not None:
            failed.append((pin.__name__, msg))
    return failed


def test_unmutated_restatement_passes_all_pins():
    """Sanity of the harness: the same restatement without a mistake passes."""
    assert _run_pins(lambda *a: _standard(*a)) == []


@pytest.mark.parametrize("mistake", MISTAKES)
def test_planted_mistake_is_caught(mistake):
    failed = _run_pins(lambda *a: _standard(*a, mistake=mistake))
    assert failed, f"no pin catches the planted mistake {mistake!r}"
