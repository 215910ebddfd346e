"""Exact rational unrolled-product form of the gated delta rule (tiny inputs).

TEST INFRASTRUCTURE ONLY (see the package docstring).

This is not the step-by-step recurrence: it writes every state as the closed
sum of products

    S_t = sum_{j<=t} (A_t A_{t-1} ... A_{j+1}) B_j  +  (A_t ... A_1) h0,
    A_s = (I - b_s k_s k_s^T) Diag(a_s),    B_j = b_j k_j v_j^T,
    o_t = scale S_t^T q_t,

which is what the gated-delta-rule recurrence S_t = e^{g_t}(I - b k k^T) S_{t-1}
+ b k v^T unrolls to (decay first for a per-key gate; for a scalar gate the
two orders coincide). With base-2 gates whose logs are integers and rational
b, k, v, q, every quantity is an exact ``Fraction``, so the fp64 oracle can
be checked against exact values.
"""
from __future__ import annotations

from fractions import Fraction


def _eye(n):
    return [[Fraction(int(i == j)) for j in range(n)] for i in range(n)]


def _matmul(a, b):
    n, m, p = len(a), len(b), len(b[0])
    return [[sum((a[i][r] * b[r][c] for r in range(m)), Fraction(0)) for c in range(p)]
            for i in range(n)]


def _add(a, b):
    return [[x + y for x, y in zip(ra, rb)] for ra, rb in zip(a, b)]


def _pow2(e):
    e = Fraction(e)
    if e.denominator != 1:
        raise ValueError("exact base-2 gates need integer logs")
    return Fraction(2) ** int(e)


def transition(k, beta, a):
    """A = (I - beta k k^T) Diag(a) for one token (k, a are length-K lists)."""
    K = len(k)
    return [[((1 if i == j else 0) - beta * k[i] * k[j]) * a[j] for j in range(K)]
            for i in range(K)]


def states(q, k, v, loggate, beta, h0=None, scale=Fraction(1), per_key=False):
    """Exact o[t][c] and final state for one head of one sequence.

    q, k: [T][K]; v: [T][V]; loggate: [T] (scalar) or [T][K] (per key), base 2,
    integer values; beta: [T]; h0: [K][V] or None.
    Returns (o [T][V], S_T [K][V]).
    """
    T, K, V = len(k), len(k[0]), len(v[0])
    a = []
    for t in range(T):
        if per_key:
            a.append([_pow2(x) for x in loggate[t]])
        else:
            a.append([_pow2(loggate[t])] * K)
    A = [transition(k[t], Fraction(beta[t]), a[t]) for t in range(T)]
    B = [[[Fraction(beta[t]) * k[t][i] * v[t][c] for c in range(V)] for i in range(K)]
         for t in range(T)]
    h0 = h0 if h0 is not None else [[Fraction(0)] * V for _ in range(K)]

    def prod(i, t):  # A_t ... A_i (identity when i > t), tokens numbered 0..T-1
        P = _eye(K)
        for s in range(i, t + 1):
            P = _matmul(A[s], P)
        return P

    o, S = [], None
    for t in range(T):
        S = _matmul(prod(0, t), h0)
        for j in range(t + 1):
            S = _add(S, _matmul(prod(j + 1, t), B[j]))
        o.append([scale * sum((S[i][c] * q[t][i] for i in range(K)), Fraction(0))
                  for c in range(V)])
    return o, S


def transfer(k, loggate, beta, per_key=False):
    """Exact segment transfer M = A_T ... A_1 for one head."""
    T, K = len(k), len(k[0])
    M = _eye(K)
    for t in range(T):
        a = [_pow2(x) for x in loggate[t]] if per_key else [_pow2(loggate[t])] * K
        M = _matmul(transition(k[t], Fraction(beta[t]), a), M)
    return M
