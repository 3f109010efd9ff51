"""Pure-Python (lists of floats) Muon update for small matrices.

TEST INFRASTRUCTURE ONLY.  A second, independent restatement of the same
update with explicit loops, used to cross-check the NumPy oracle on small
cases (a 64 x 128 matrix takes a few seconds).  Same readings as
``muon_ref`` (M' = beta M + G; eps added to the Frobenius norm; wide
orientation; P' = P(1 - lr wd) - lr s O), written without NumPy.
"""
from __future__ import annotations

import math


def _matmul_nt(X, Y):
    """X (p x q) times Y^T where Y is (r x q): returns p x r."""
    return [[sum(xv * yv for xv, yv in zip(xr, yr)) for yr in Y] for xr in X]


def _transpose(X):
    return [list(col) for col in zip(*X)]


def naive_update(P, G, M, beta, lr, wd, k, a, b, c, eps, s, nesterov=False, rows_abc=None):
    """Returns (P', M', O) as nested lists; s is the shape scale.  With
    nesterov the iteration starts from U = G + beta M' (M' is still returned);
    rows_abc, if given, holds per-step (a, b, c) rows, the last repeating."""
    rows, cols = len(P), len(P[0])
    Mp = [[beta * M[i][j] + G[i][j] for j in range(cols)] for i in range(rows)]
    U = [[G[i][j] + beta * Mp[i][j] for j in range(cols)] for i in range(rows)] if nesterov else Mp
    sq = 0.0
    for i in range(rows):
        for j in range(cols):
            sq += U[i][j] * U[i][j]
    inv = 1.0 / (math.sqrt(sq) + eps)
    X = [[U[i][j] * inv for j in range(cols)] for i in range(rows)]
    tr = rows > cols
    if tr:
        X = _transpose(X)
    for step in range(k):
        if rows_abc:
            a, b, c = rows_abc[min(step, len(rows_abc) - 1)]
        A = _matmul_nt(X, X)                      # A = X X^T
        AA = _matmul_nt(A, _transpose(A))         # A A
        m = len(A)
        Bm = [[b * A[i][j] + c * AA[i][j] for j in range(m)] for i in range(m)]
        BX = _matmul_nt(Bm, _transpose(X))        # B X
        X = [[a * X[i][j] + BX[i][j] for j in range(len(X[0]))] for i in range(m)]
    if tr:
        X = _transpose(X)
    Pn = [[P[i][j] * (1.0 - lr * wd) - lr * s * X[i][j] for j in range(cols)]
          for i in range(rows)]
    return Pn, Mp, X
