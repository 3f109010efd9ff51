"""The O tolerance of bf16 mode (2e-2, relative Frobenius) is wide enough for
correct low-precision arithmetic and narrow enough to catch plausible slips.

The tensor path stores the Newton-Schulz operands (X, A = X X^T, B = bA + cA^2)
in a 16-bit type and accumulates every product in fp32.  The skinny path
(m <= 64) rounds the normalised data to that type once and iterates in Gram
space on m x m matrices held to about fp32 precision.  Here both are emulated
in NumPy: each stored operand rounds to nearest-even fp16 or bf16, and each
product is an fp32 matrix product.  The steps are the plain quintic step of
«关于分布式Muon的想法整合及讨论» §2, compared with the fp64 oracle on seeded
Gaussian momenta:

* fp16 operands (the default) land inside the tolerance with a 4x margin on
  both paths up to k = 10, and bf16 operands do on the skinny path;
* bf16 operands on the tensor path land inside at k = 5 but outgrow the
  tolerance by k = 10, which is why fp16 is the default operand type;
* a dropped A^2 term, a flipped sign of b, the Gram of the wrong side, one
  Newton-Schulz step too few, and a missing normalisation each land outside;
* momenta whose singular values spread over several decades use up most of
  the margin, because the iteration stretches their small directions.
"""
import numpy as np
import pytest

from oracle import muon_ref
from oracle_pins import A_, B_, C_
from parity import TOL_O

TOL_BF16_MODE = TOL_O["bf16"]


def round_f16(x):
    return np.asarray(x, np.float32).astype(np.float16).astype(np.float32)


def round_bf16(x):
    """Round-to-nearest-even to bfloat16 (finite inputs), kept in fp32."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def emulated_ns(Mp, k, rnd, *, drop_c=False, flip_b=False, wrong_side=False, normalise=True):
    X = np.asarray(Mp, np.float32)
    if normalise:
        X = X / (np.sqrt(np.sum(X.astype(np.float64) ** 2)).astype(np.float32) + np.float32(1e-7))
    X = rnd(X)
    a, b, c = np.float32(A_), np.float32(-B_ if flip_b else B_), np.float32(0.0 if drop_c else C_)
    for _ in range(k):
        if wrong_side:  # X^T X padded into the top-left m x m corner
            A = rnd((X.T @ X)[: X.shape[0], : X.shape[0]])
        else:
            A = rnd(X @ X.T)
        B = rnd(b * A + c * (A @ A))
        X = rnd(a * X + B @ X)
    return X.astype(np.float64)


def emulated_gram_space(Mp, k, rnd):
    """The skinny path's order: X0 rounded once, then A0 = X0 X0^T, k steps of
    Q = aI + bA + cA^2, Pi <- Q Pi, A <- Q^2 A in fp32, and O = Pi X0."""
    X = np.asarray(Mp, np.float32)
    X = rnd(X / (np.sqrt(np.sum(X.astype(np.float64) ** 2)).astype(np.float32) + np.float32(1e-7)))
    I = np.eye(X.shape[0], dtype=np.float32)
    A, Pi = X @ X.T, I.copy()
    for _ in range(k):
        Q = np.float32(A_) * I + np.float32(B_) * A + np.float32(C_) * (A @ A)
        Pi, A = Q @ Pi, (Q @ Q) @ A
    return rnd(Pi @ X).astype(np.float64)


def _momentum(m, n, seed):
    rng = np.random.default_rng(seed)
    G = rng.standard_normal((m, n)) * 1e-3
    M = rng.standard_normal((m, n)) * 1e-3
    return (np.float32(0.95) * M.astype(np.float32) + G.astype(np.float32)).astype(np.float64)


def _rel(got, want):
    return float(np.linalg.norm(got - want) / np.linalg.norm(want))


def _want(Mp, k):
    return muon_ref.orthogonalize(Mp, k, A_, B_, C_, 1e-7)


SKINNY = [(24, 10240, 5), (64, 2048, 5), (24, 2048, 10)]
TENSOR = [(128, 512, 5), (256, 1024, 5), (256, 768, 10)]


@pytest.mark.parametrize("m,n,k", SKINNY)
def test_skinny_path_arithmetic_is_inside(m, n, k):
    Mp = _momentum(m, n, m + n + k)
    want = _want(Mp, k)
    for rnd in (round_f16, round_bf16):
        err = _rel(emulated_gram_space(Mp, k, rnd), want)
        assert err <= TOL_BF16_MODE / 4, (rnd.__name__, err)


@pytest.mark.parametrize("m,n,k", SKINNY + TENSOR)
def test_fp16_operands_are_inside(m, n, k):
    Mp = _momentum(m, n, m + n + k)
    err = _rel(emulated_ns(Mp, k, round_f16), _want(Mp, k))
    assert err <= TOL_BF16_MODE / 4, err


def test_bf16_operands_on_the_tensor_path():
    """Inside at k = 5; past the tolerance at k = 10, where fp16 stays inside."""
    Mp = _momentum(256, 1024, 3)
    assert _rel(emulated_ns(Mp, 5, round_bf16), _want(Mp, 5)) <= TOL_BF16_MODE
    Mp = _momentum(256, 2048, 4)
    want = _want(Mp, 10)
    assert _rel(emulated_ns(Mp, 10, round_bf16), want) > TOL_BF16_MODE
    assert _rel(emulated_ns(Mp, 10, round_f16), want) <= TOL_BF16_MODE / 4


@pytest.mark.parametrize("m,n,k", SKINNY[:2] + TENSOR[:1])
@pytest.mark.parametrize("slip", ["drop_c", "flip_b", "wrong_side", "one_step_short",
                                  "no_normalise"])
def test_plausible_slips_are_outside(m, n, k, slip):
    Mp = _momentum(m, n, m + n + k)
    want = muon_ref.orthogonalize(Mp, k, A_, B_, C_, 1e-7)
    kw = {}
    kk = k
    if slip == "one_step_short":
        kk = k - 1
    elif slip == "no_normalise":
        kw["normalise"] = False
    else:
        kw[slip] = True
    with np.errstate(over="ignore", invalid="ignore"):
        got = emulated_ns(Mp, kk, round_f16, **kw)
    err = _rel(got, want) if np.all(np.isfinite(got)) else np.inf
    assert err > TOL_BF16_MODE, (slip, err)


def test_bf16_rounding_helper():
    """Round-to-nearest-even at the bf16 boundary, ties to even."""
    one = np.float32(1.0)
    ulp = np.float32(2.0 ** -7)
    x = np.array([one, one + ulp / 2, one + 3 * ulp / 2, one + ulp / 4, -one - ulp / 2],
                 np.float32)
    np.testing.assert_array_equal(round_bf16(x),
                                  np.array([1.0, 1.0, 1.0 + 2 * ulp, 1.0, -1.0], np.float32))


def _spread_momentum(m, n, decades, seed):
    """A momentum whose singular values fall log-evenly over `decades`."""
    rng = np.random.default_rng(seed)
    U, _ = np.linalg.qr(rng.standard_normal((m, m)))
    V, _ = np.linalg.qr(rng.standard_normal((n, m)))
    X = (U * np.logspace(0, -decades, m)) @ V.T * 1e-2
    return X.astype(np.float32).astype(np.float64)


def _hi_lo_f16(x):
    hi = round_f16(x)
    return hi + round_f16(x - hi)


def test_spread_spectra_use_up_the_headroom():
    """Five steps stretch directions with small singular values by up to
    a^5 (about 486), so the one rounding of X0 dominates the error.  With the
    spectrum over four decades, fp16 operands come within a factor 2 of the
    tolerance and bf16 operands exceed it several times over.  Rounding X0
    as an fp16 pair (high part plus residual) for the final product
    O = Pi X0 brings the Gram-space error back to about 1e-3."""
    Mp = _spread_momentum(24, 10240, 4, seed=0)
    want = _want(Mp, 5)
    e16 = _rel(emulated_gram_space(Mp, 5, round_f16), want)
    ebf = _rel(emulated_gram_space(Mp, 5, round_bf16), want)
    assert TOL_BF16_MODE / 2 <= e16 <= TOL_BF16_MODE, e16
    assert ebf > 4 * TOL_BF16_MODE, ebf
    # the same iteration with only the last product's operand split
    X = np.asarray(Mp, np.float32)
    X = X / (np.sqrt(np.sum(X.astype(np.float64) ** 2)).astype(np.float32) + np.float32(1e-7))
    Xr = round_f16(X)
    I = np.eye(24, dtype=np.float32)
    A, Pi = Xr @ Xr.T, I.copy()
    for _ in range(5):
        Q = np.float32(A_) * I + np.float32(B_) * A + np.float32(C_) * (A @ A)
        Pi, A = Q @ Pi, (Q @ Q) @ A
    e_split = _rel((Pi @ _hi_lo_f16(X)).astype(np.float64), want)
    assert e_split <= TOL_BF16_MODE / 10, e_split
    # concentrated spectra, like the seeded Gaussian workloads, keep a wide margin
    Mp = _spread_momentum(24, 10240, 0.3, seed=0)
    assert _rel(emulated_gram_space(Mp, 5, round_f16), _want(Mp, 5)) <= TOL_BF16_MODE / 20


def test_fp32_mode_keeps_its_margin_on_spread_spectra():
    """fp32 mode (every product an fp32 FMA) against its 1e-4 tolerance, on a
    spectrum over four decades: about 5e-6."""
    Mp = _spread_momentum(64, 512, 4, seed=2)
    err = _rel(emulated_ns(Mp, 5, lambda x: np.asarray(x, np.float32)), _want(Mp, 5))
    assert err <= TOL_O["fp32"] / 10, err
