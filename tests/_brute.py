"""50-digit decimal brute force of standard attention, for tiny inputs.

Independent of the oracle: pure Python ``decimal`` arithmetic, one element at a
time, following the definition softmax(scale * Q K^T [+ causal mask]) V and
LSE_i = ln sum_j exp(scale * q_i . k_j) over the visible keys.
"""
from __future__ import annotations

from decimal import Decimal, getcontext


def attention_decimal(q, k, v, causal: bool, scale_sq_inv: int | None = None, scale: float | None = None,
                      q_pos=None, digits: int = 50):
    """Return (o, lse) as lists of Decimal.

    The scale is 1/sqrt(scale_sq_inv) computed in decimal when scale_sq_inv is
    given, else the given float converted exactly.
    """
    getcontext().prec = digits
    if scale_sq_inv is not None:
        sc = Decimal(1) / Decimal(scale_sq_inv).sqrt()
    else:
        sc = Decimal(float(scale))
    Q = [[Decimal(float(x)) for x in row] for row in q]
    K = [[Decimal(float(x)) for x in row] for row in k]
    V = [[Decimal(float(x)) for x in row] for row in v]
    n, d, nk = len(Q), len(Q[0]), len(K)
    pos = list(range(n)) if q_pos is None else [int(p) for p in q_pos]
    O, LSE = [], []
    for i in range(n):
        vis = [j for j in range(nk) if not (causal and j > pos[i])]
        s = {j: sc * sum(Q[i][t] * K[j][t] for t in range(d)) for j in vis}
        z = sum((s[j].exp() for j in vis), Decimal(0))
        O.append([sum((s[j].exp() * V[j][c] for j in vis), Decimal(0)) / z for c in range(len(V[0]))])
        LSE.append(z.ln())
    return O, LSE
