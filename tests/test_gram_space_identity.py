"""The identity behind the skinny kernel, checked in fp64 against the oracle.

For a wide X_0 (m rows, m <= cols) one quintic step is X_{j+1} = Q_j X_j with
A_j = X_j X_j^T and Q_j = a_j I + b_j A_j + c_j A_j^2 («关于分布式Muon的想法整合及
讨论» §2).  Hence X_k = Pi_k X_0 with Pi_0 = I, Pi_{j+1} = Q_j Pi_j, and
A_{j+1} = Q_j A_j Q_j^T = Q_j^2 A_j, since Q_j is symmetric and a polynomial in
A_j.  The skinny GPU kernel evaluates Newton-Schulz that way: one Gram matrix
from the data, k steps on m x m matrices, one product Pi_k X_0.

These checks run that recurrence here, written out independently of both the
kernel and the oracle, and compare it with the oracle's direct iteration.  A
column-sharded X_0 needs the partial Grams added once, for A_0, after which
every shard's output columns are Pi_k times its own columns
(«关于分布式Muon的想法整合及讨论» §6 adds the partial Grams every step).
"""
import numpy as np
import pytest

from oracle import muon_ref

from oracle_pins import A_, B_, C_, SCHEDULE


def _gram_space(X0, coeffs, symmetric_form=False):
    m = X0.shape[0]
    I = np.eye(m)
    A = X0 @ X0.T
    Pi = I.copy()
    for a, b, c in coeffs:
        Q = a * I + b * A + c * (A @ A)
        Pi = Q @ Pi
        A = Q @ A @ Q.T if symmetric_form else (Q @ Q) @ A
    return Pi


def _x0(rng, m, n, spread=True):
    X = rng.standard_normal((m, n))
    if spread:  # singular values over several decades, as in a momentum
        X = X * np.logspace(0, -3, m)[:, None]
    return muon_ref.frobenius_normalize(X, 1e-7)


@pytest.mark.parametrize("m,n", [(1, 300), (7, 9), (24, 1024), (64, 512), (64, 64)])
@pytest.mark.parametrize("k", [1, 5, 10])
def test_gram_space_equals_direct_iteration(m, n, k):
    rng = np.random.default_rng(1000 * m + n + k)
    X0 = _x0(rng, m, n)
    coeffs = muon_ref.step_coefficients(k, A_, B_, C_)
    want = muon_ref.newton_schulz(X0, k, A_, B_, C_)
    for sym in (False, True):
        got = _gram_space(X0, coeffs, sym) @ X0
        err = np.linalg.norm(got - want) / np.linalg.norm(want)
        assert err <= 1e-11, (m, n, k, sym, err)


@pytest.mark.parametrize("m,n,k", [(24, 2048, 6), (64, 256, 64), (3, 40, 64)])
def test_gram_space_with_a_schedule(m, n, k):
    """Per-step rows; the last one is the contractive textbook map, so the
    two orderings of the arithmetic stay together over 64 steps."""
    rng = np.random.default_rng(7 * m + k)
    X0 = _x0(rng, m, n)
    coeffs = muon_ref.step_coefficients(k, A_, B_, C_, SCHEDULE)
    want = muon_ref.newton_schulz(X0, k, A_, B_, C_, SCHEDULE)
    got = _gram_space(X0, coeffs) @ X0
    assert np.linalg.norm(got - want) / np.linalg.norm(want) <= 1e-10


def test_gram_space_on_the_transposed_side():
    """A tall matrix is orthogonalised through its transpose; the Gram-space
    form of that transpose, transposed back, equals the oracle's update."""
    rng = np.random.default_rng(5)
    M = rng.standard_normal((700, 20))
    want = muon_ref.orthogonalize(M, 5, A_, B_, C_, 1e-7)
    X0 = muon_ref.frobenius_normalize(M, 1e-7).T
    got = (_gram_space(X0, muon_ref.step_coefficients(5, A_, B_, C_)) @ X0).T
    assert np.linalg.norm(got - want) / np.linalg.norm(want) <= 1e-11


@pytest.mark.parametrize("shards", [1, 2, 4, 8])
def test_gram_space_with_column_shards(shards):
    """One sum of partial Grams for A_0, then Pi_k applied shard by shard,
    equals the oracle's sharded iteration, which sums them every step."""
    rng = np.random.default_rng(40 + shards)
    M = rng.standard_normal((24, 1000))
    X0 = muon_ref.sharded_frobenius_normalize(M, 1e-7, shards)
    parts = np.array_split(X0, shards, axis=1)
    A0 = sum(p @ p.T for p in parts)
    coeffs = muon_ref.step_coefficients(5, A_, B_, C_)
    m = X0.shape[0]
    I = np.eye(m)
    A, Pi = A0, I.copy()
    for a, b, c in coeffs:
        Q = a * I + b * A + c * (A @ A)
        Pi, A = Q @ Pi, (Q @ Q) @ A
    got = np.concatenate([Pi @ p for p in parts], axis=1)
    want = muon_ref.newton_schulz_sharded(X0, 5, A_, B_, C_, shards)
    assert np.linalg.norm(got - want) / np.linalg.norm(want) <= 1e-11


def test_a_dropped_square_is_caught():
    """The check is sharp: updating A with Q instead of Q^2 drifts far off."""
    rng = np.random.default_rng(9)
    X0 = _x0(rng, 24, 1024)
    want = muon_ref.newton_schulz(X0, 5, A_, B_, C_)
    I = np.eye(24)
    A, Pi = X0 @ X0.T, I.copy()
    for _ in range(5):
        Q = A_ * I + B_ * A + C_ * (A @ A)
        Pi, A = Q @ Pi, Q @ A
    got = Pi @ X0
    assert np.linalg.norm(got - want) / np.linalg.norm(want) > 1e-2
