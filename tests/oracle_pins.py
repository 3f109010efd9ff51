"""Pins for the CPU oracle: checks against mathematics, not against itself.

Each check takes the oracle module (so a test can plant a mistake in a copy of
it) and returns None or raises AssertionError.  Sources of each fact:

* closed form: for X = U S V^T one quintic step gives U p(S) V^T with
  p(s) = a s + b s^3 + c s^5, because X X^T = U S^2 U^T; k steps give p^k.
* the SVD of the oracle's output, from LAPACK, must equal p^k of the
  normalised input singular values (sorted; p^k is not monotone).
* a 1 x n matrix has one singular value, so its normalised form is a unit row
  v and the result is p^k(1) v exactly.
* transpose symmetry: NS(X^T) = NS(X)^T, and the tall form X <- aX +
  X(b X^T X + c (X^T X)^2) is the same map written on the other side.
* batch independence («MindSpore HyperParallel X 盘古,Muon优化器实现6倍性能跃升»,
  Muon亲和的专家切分, Fig. 4): the [E, M, N] result equals the per-expert results,
  so a [2, 4, 4] local shard gives the matching slice of the [4, 4, 4] result.
"""
from __future__ import annotations

import math

import numpy as np

A_, B_, C_ = 3.4445, -4.7750, 2.0315


def p_iter(s, k, a=A_, b=B_, c=C_):
    """Scalar polynomial iteration in plain Python floats (Horner form)."""
    out = []
    for v in np.ravel(s):
        v = float(v)
        for _ in range(k):
            v2 = v * v
            v = v * (a + v2 * (b + c * v2))
        out.append(v)
    return np.array(out).reshape(np.shape(s))


def pin_diagonal(ref, k=5):
    """X = diag(sigma) padded to 5 x 9 -> diag(p^k(sigma))."""
    sig = np.array([1.0, 0.8, 0.5, 0.11, 0.003])
    X = np.zeros((5, 9)); X[np.arange(5), np.arange(5)] = sig
    out = ref.newton_schulz(X, k, A_, B_, C_)
    want = np.zeros_like(X); want[np.arange(5), np.arange(5)] = p_iter(sig, k)
    assert np.max(np.abs(out - want)) <= 1e-12 * np.max(np.abs(want)), "diagonal closed form"


def _rand_orth(rng, n):
    q, r = np.linalg.qr(rng.standard_normal((n, n)))
    return q * np.sign(np.diag(r))


def pin_orthogonal_times_diagonal(ref, k=5, seed=1):
    """X = Q1 [D 0] Q2^T (rectangular) -> Q1 [p^k(D) 0] Q2^T."""
    rng = np.random.default_rng(seed)
    m, n = 6, 11
    d = np.array([0.9, 0.7, 0.45, 0.3, 0.05, 0.01])
    Q1, Q2 = _rand_orth(rng, m), _rand_orth(rng, n)
    S = np.zeros((m, n)); S[np.arange(m), np.arange(m)] = d
    Sk = np.zeros((m, n)); Sk[np.arange(m), np.arange(m)] = p_iter(d, k)
    out = ref.newton_schulz(Q1 @ S @ Q2.T, k, A_, B_, C_)
    want = Q1 @ Sk @ Q2.T
    assert np.linalg.norm(out - want) <= 1e-12 * np.linalg.norm(want), "U p(S) V^T"


def pin_svd_band(ref, k=5, seed=2):
    """Brute-force SVD on tiny random inputs through the full update path."""
    rng = np.random.default_rng(seed)
    for (r, c) in [(3, 7), (7, 3), (5, 5), (8, 32), (32, 8), (1, 6), (6, 1)]:
        M = rng.standard_normal((r, c)); G = rng.standard_normal((r, c))
        P = rng.standard_normal((r, c))
        beta, lr, wd, eps = 0.9, 0.01, 0.0, 1e-7
        _, Mp, O = ref.muon_update_ref(P, G, M, beta, lr, wd, k, A_, B_, C_, eps, "none")
        # momentum closed form, elementwise
        assert np.allclose(Mp, beta * M + G, rtol=0, atol=1e-15), "momentum"
        sig_in = np.linalg.svd(Mp, compute_uv=False)
        fro = math.sqrt(float(np.sum(sig_in ** 2)))
        want = np.sort(p_iter(sig_in / (fro + eps), k))
        got = np.sort(np.linalg.svd(O, compute_uv=False))
        assert np.max(np.abs(got - want)) <= 1e-10, f"svd closed form {r}x{c}"
        # the band the iterated polynomial predicts on [min, max] normalised sigma
        lo, hi = float(np.min(sig_in / (fro + eps))), float(np.max(sig_in / (fro + eps)))
        grid = p_iter(np.linspace(lo, hi, 4001), k)
        assert got.min() >= grid.min() - 1e-9 and got.max() <= grid.max() + 1e-9, "band"


def pin_single_row_exact(ref):
    """1 x 2 row [3, 4] (norm 5): O = p^k(1) [0.6, 0.8]; ||.||_F=5 exactly."""
    M = np.array([[3.0, 4.0]]); G = np.zeros((1, 2)); P = np.array([[1.0, -2.0]])
    for k in (0, 1, 2, 5):
        Pn, Mp, O = ref.muon_update_ref(P, G, M, 1.0, 0.5, 0.2, k, A_, B_, C_, 0.0, "none")
        pk = 1.0
        for _ in range(k):
            pk = A_ * pk + B_ * pk ** 3 + C_ * pk ** 5
        want_O = pk * np.array([[0.6, 0.8]])
        assert np.max(np.abs(O - want_O)) <= 1e-14, f"1-row O, k={k}"
        want_P = P * (1 - 0.5 * 0.2) - 0.5 * want_O
        assert np.max(np.abs(Pn - want_P)) <= 1e-14, f"1-row P', k={k}"


def pin_transpose_symmetry(ref, k=5, seed=3):
    """NS on a tall matrix equals the transpose of NS on its transpose, and the
    right-sided (tall) form of the same polynomial map."""
    rng = np.random.default_rng(seed)
    M = rng.standard_normal((13, 5))
    O_tall = ref.orthogonalize(M, k, A_, B_, C_, 1e-7)
    O_wide = ref.orthogonalize(M.T, k, A_, B_, C_, 1e-7)
    assert np.linalg.norm(O_tall - O_wide.T) <= 1e-12 * np.linalg.norm(O_tall), "transpose"
    X = M / (np.linalg.norm(M) + 1e-7)
    for _ in range(k):
        S = X.T @ X
        X = A_ * X + X @ (B_ * S + C_ * (S @ S))
    assert np.linalg.norm(O_tall - X) <= 1e-12 * np.linalg.norm(X), "tall form"


def pin_batch_independence(ref, k=5, seed=4):
    """[4, 4, 4] expert tensor: the local [2, 4, 4] shard's result equals the
    matching slice of the full result (Fig. 4 example of the expert section)."""
    rng = np.random.default_rng(seed)
    P, G, M = (rng.standard_normal((4, 4, 4)) for _ in range(3))
    full = ref.muon_step_ref([P], [G], [M], 0.95, 0.02, 0.1, k, A_, B_, C_)
    for r in range(2):
        sl = slice(2 * r, 2 * r + 2)
        part = ref.muon_step_ref([P[sl]], [G[sl]], [M[sl]], 0.95, 0.02, 0.1, k, A_, B_, C_)
        for t in range(3):
            assert np.array_equal(part[t][0], full[t][0][sl]), "shard slice"
    # and each expert equals the single-matrix update
    for e in range(4):
        one = ref.muon_update_ref(P[e], G[e], M[e], 0.95, 0.02, 0.1, k, A_, B_, C_)
        assert np.array_equal(one[0], full[0][0][e]), "expert vs single"


def pin_degenerate(ref):
    """Zero momentum and gradient: O = 0, P' = P (1 - lr wd).  k = 0: O is the
    normalised momentum, of Frobenius norm ||M'|| / (||M'|| + eps)."""
    rng = np.random.default_rng(5)
    P = rng.standard_normal((4, 9))
    Z = np.zeros((4, 9))
    Pn, Mp, O = ref.muon_update_ref(P, Z, Z, 0.95, 0.02, 0.1, 5, A_, B_, C_)
    assert np.all(O == 0) and np.all(Mp == 0), "zero input"
    assert np.max(np.abs(Pn - P * (1 - 0.02 * 0.1))) <= 1e-15, "zero input P'"
    G = rng.standard_normal((4, 9)); M = rng.standard_normal((4, 9))
    _, Mp, O = ref.muon_update_ref(P, G, M, 0.5, 0.02, 0.0, 0, A_, B_, C_, 1e-3, "none")
    n = float(np.linalg.norm(0.5 * M + G))
    assert abs(float(np.linalg.norm(O)) - n / (n + 1e-3)) <= 1e-12, "k=0 norm"
    assert np.allclose(O * (n + 1e-3), 0.5 * M + G, rtol=1e-13, atol=0), "k=0 direction"


ALL_PINS = [pin_diagonal, pin_orthogonal_times_diagonal, pin_svd_band,
            pin_single_row_exact, pin_transpose_symmetry, pin_batch_independence,
            pin_degenerate]


def pin_scale_and_decay(ref):
    """k = 0, eps = 0 on a tall 8 x 2 matrix: O = M'/||M'||, and
    P' = P (1 - lr wd) - lr s O with s = sqrt(8/2) = 2 ('sqrt_aspect') or
    s = 0.2 sqrt(8) ('rms_0_2'); for the wide 2 x 8 transpose s = 1."""
    rng = np.random.default_rng(6)
    M = rng.standard_normal((8, 2)); P = rng.standard_normal((8, 2)); Z = np.zeros((8, 2))
    O = M / math.sqrt(float(np.sum(M ** 2)))
    for mode, s in (("sqrt_aspect", 2.0), ("rms_0_2", 0.2 * math.sqrt(8.0)), ("none", 1.0)):
        Pn, _, _ = ref.muon_update_ref(P, Z, M, 1.0, 0.1, 0.3, 0, A_, B_, C_, 0.0, mode)
        assert np.max(np.abs(Pn - (P * (1 - 0.03) - 0.1 * s * O))) <= 1e-14, f"scale {mode}"
    Pn, _, _ = ref.muon_update_ref(P.T, Z.T, M.T, 1.0, 0.1, 0.3, 0, A_, B_, C_, 0.0, "sqrt_aspect")
    assert np.max(np.abs(Pn - (P.T * (1 - 0.03) - 0.1 * O.T))) <= 1e-14, "scale wide"


ALL_PINS.append(pin_scale_and_decay)


def p_iter_schedule(s, rows, k):
    """Scalar iteration with per-step coefficients, the last row repeating,
    in plain Python floats (Horner form)."""
    out = []
    for v in np.ravel(s):
        v = float(v)
        for t in range(k):
            a, b, c = rows[min(t, len(rows) - 1)]
            v2 = v * v
            v = v * (a + v2 * (b + c * v2))
        out.append(v)
    return np.array(out).reshape(np.shape(s))


# A per-step schedule of distinct rows: the quintic above, two milder
# steps, then the textbook quintic Newton-Schulz map for the polar factor,
# p(s) = (15 s - 10 s^3 + 3 s^5) / 8 (p(1) = 1, p'(1) = 0), which repeats.
SCHEDULE = [(A_, B_, C_), (3.0, -3.2, 1.2), (2.0, -1.5, 0.5), (1.875, -1.25, 0.375)]


def pin_schedule_diagonal(ref, k=6):
    """Per-step coefficients act on each singular value as the composed
    scalar maps p_{k-1}( ... p_0(s)), the last schedule row repeating: the
    closed form of the diagonal case, step by step."""
    sig = np.array([1.0, 0.8, 0.5, 0.11, 0.003])
    X = np.zeros((5, 9)); X[np.arange(5), np.arange(5)] = sig
    out = ref.newton_schulz(X, k, A_, B_, C_, SCHEDULE)
    want = np.zeros_like(X); want[np.arange(5), np.arange(5)] = p_iter_schedule(sig, SCHEDULE, k)
    assert np.max(np.abs(out - want)) <= 1e-12 * np.max(np.abs(want)), "schedule closed form"
    one = ref.newton_schulz(X, k, A_, B_, C_, [(A_, B_, C_)])
    assert np.array_equal(one, ref.newton_schulz(X, k, A_, B_, C_)), "one-row schedule = constant"


def pin_nesterov(ref):
    """Nesterov input U = G + beta M' on a 1 x n matrix (one singular value):
    O = p^k(1) U / ||U|| with eps = 0, while M' stays beta M + G; with
    beta = 0 the option changes nothing."""
    rng = np.random.default_rng(7)
    G = rng.standard_normal((1, 9)); M = rng.standard_normal((1, 9)); P = rng.standard_normal((1, 9))
    beta = 0.9
    U = G + beta * (beta * M + G)
    _, Mp, O = ref.muon_update_ref(P, G, M, beta, 0.02, 0.0, 5, A_, B_, C_, 0.0, "none", True)
    want = p_iter(np.array([1.0]), 5)[0] * U / math.sqrt(float(np.sum(U * U)))
    assert np.max(np.abs(O - want)) <= 1e-12, "nesterov direction"
    assert np.max(np.abs(Mp - (beta * M + G))) <= 1e-15, "nesterov keeps M'"
    G2 = rng.standard_normal((4, 7)); M2 = rng.standard_normal((4, 7)); P2 = rng.standard_normal((4, 7))
    r0 = ref.muon_update_ref(P2, G2, M2, 0.0, 0.02, 0.1, 5, A_, B_, C_, 1e-7, "sqrt_aspect", False)
    r1 = ref.muon_update_ref(P2, G2, M2, 0.0, 0.02, 0.1, 5, A_, B_, C_, 1e-7, "sqrt_aspect", True)
    assert all(np.array_equal(x, y) for x, y in zip(r0, r1)), "beta = 0"


ALL_PINS += [pin_schedule_diagonal, pin_nesterov]


def pin_sharded_equals_unsharded(ref, k=5, seed=8):
    """Column shards change nothing mathematically: the sum of per-shard
    partial Grams is the Gram matrix, and the per-shard sums of squares add up
    to ||M||_F^2.  So the sharded normalise + iteration equals the unsharded
    one (fp64 rounding only), for any shard count, including shards narrower
    than the matrix is tall."""
    rng = np.random.default_rng(seed)
    M = rng.standard_normal((6, 23))
    X0 = ref.frobenius_normalize(M, 1e-7)
    want = ref.newton_schulz(X0, k, A_, B_, C_)
    for t in (1, 2, 3, 8):
        Xs = ref.sharded_frobenius_normalize(M, 1e-7, t)
        assert np.max(np.abs(Xs - X0)) <= 1e-15, f"sharded norm t={t}"
        got = ref.newton_schulz_sharded(Xs, k, A_, B_, C_, t)
        assert np.max(np.abs(got - want)) <= 1e-12 * np.max(np.abs(want)), f"sharded NS t={t}"
    # and against the closed form on a diagonal input split across shards
    sig = np.array([1.0, 0.6, 0.2])
    X = np.zeros((3, 7)); X[np.arange(3), np.arange(3)] = sig
    got = ref.newton_schulz_sharded(X, k, A_, B_, C_, 3)
    assert np.max(np.abs(np.diag(got[:, :3]) - p_iter(sig, k))) <= 1e-12, "sharded diagonal"
    assert np.max(np.abs(got[:, 3:])) == 0.0 and np.max(np.abs(got - np.diag(np.diag(got[:, :3])) @ np.eye(3, 7))) <= 1e-12


ALL_PINS.append(pin_sharded_equals_unsharded)


def pin_eps_placement(ref):
    """eps is added to the norm, not to its square (the reading taken; the
    pages give no eps): a matrix whose Frobenius norm equals eps normalises
    to norm exactly 1/2, sharded or not, and with eps = 0 to norm 1."""
    M = np.zeros((3, 5)); M[1, 2] = 1e-7
    for X in (ref.frobenius_normalize(M, 1e-7), ref.sharded_frobenius_normalize(M, 1e-7, 2)):
        assert abs(np.linalg.norm(X) - 0.5) <= 1e-15, "eps on the norm"
    M = np.full((2, 4), 0.5)
    assert abs(np.linalg.norm(ref.frobenius_normalize(M, 0.0)) - 1.0) <= 1e-15, "eps = 0"


ALL_PINS.append(pin_eps_placement)
