"""The oracle against its pins (CPU only), plus planted-mistake checks showing
that each plausible slip in the oracle makes at least one pin fail."""
import json
import math
import os
import time
import types

import numpy as np
import pytest

import oracle
from oracle import muon_ref
from oracle.naive import naive_update

from oracle_pins import ALL_PINS, A_, B_, C_

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(muon_ref)


def _mutant(old, new):
    src = open(muon_ref.__file__, encoding="utf-8").read()
    assert src.count(old) == 1, old
    mod = types.ModuleType("muon_ref_mutant")
    exec(compile(src.replace(old, new), "muon_ref_mutant", "exec"), mod.__dict__)
    return mod


MUTANTS = {
    "drop_c_term": ("B = b * A + c * (A @ A)", "B = b * A"),
    "flip_b_sign": ("B = b * A + c * (A @ A)", "B = -b * A + c * (A @ A)"),
    "gram_wrong_side": ("A = X @ X.T", "A = X.T @ X"),
    "minus_update": ("X = a * X + B @ X", "X = a * X - B @ X"),
    "no_untranspose": ("return X.T if transposed else X", "return X"),
    "norm_squared": ("math.sqrt(float(np.sum(M * M)))", "float(np.sum(M * M))"),
    "damped_momentum": ("return float(beta) * np.asarray(M, np.float64) + np.asarray(G, np.float64)",
                        "return float(beta) * np.asarray(M, np.float64) + (1.0 - float(beta)) * np.asarray(G, np.float64)"),
    "additive_decay": ("Pn = P * (1.0 - float(lr) * float(wd))", "Pn = P - float(lr) * float(wd)"),
    "scale_swapped": ("scale_factor(P.shape[0], P.shape[1], scale_mode)",
                      "scale_factor(P.shape[1], P.shape[0], scale_mode)"),
    "one_step_short": ("for a, b, c in coeffs:", "for a, b, c in coeffs[1:]:"),
    "schedule_reversed": ("return [rows[min(s, len(rows) - 1)] for s in range(int(k))]",
                          "return [rows[::-1][min(s, len(rows) - 1)] for s in range(int(k))]"),
    "schedule_first_repeats": ("return [rows[min(s, len(rows) - 1)] for s in range(int(k))]",
                               "return [rows[s] if s < len(rows) else rows[0] for s in range(int(k))]"),
    "nesterov_undamped": ("return np.asarray(G, np.float64) + float(beta) * np.asarray(Mp, np.float64)",
                          "return np.asarray(G, np.float64) + np.asarray(Mp, np.float64)"),
    "shard_gram_last_only": ("            A = A + p @ p.T", "            A = p @ p.T"),
    "shard_update_own_gram": ("        parts = [a_s * p + B @ p for p in parts]",
                              "        parts = [a_s * p + (b_s * (p @ p.T) + c_s * (p @ p.T) @ (p @ p.T)) @ p for p in parts]"),
    "nesterov_on_old_m": ("U = nesterov_input(Mp, G, beta) if nesterov else Mp",
                          "U = nesterov_input(M, G, beta) if nesterov else Mp"),
    "eps_in_square": ("math.sqrt(float(np.sum(M * M))) + float(eps)",
                      "math.sqrt(float(np.sum(M * M)) + float(eps))"),
    "sharded_eps_in_square": ("return M / (math.sqrt(ss) + float(eps))",
                              "return M / math.sqrt(ss + float(eps))"),
    "sharded_norm_last_shard": ("        ss += float(np.sum(p * p))", "        ss = float(np.sum(p * p))"),
    "transpose_wrong_way": ("transposed = X.shape[0] > X.shape[1]",
                            "transposed = X.shape[0] < X.shape[1]"),
    "decay_after_update": ("Pn = P * (1.0 - float(lr) * float(wd)) - float(lr) * s * O",
                           "Pn = (P - float(lr) * s * O) * (1.0 - float(lr) * float(wd))"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    mod = _mutant(*MUTANTS[name])
    failed = []
    for pin in ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mod)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin catches mutant {name}"


def test_naive_loops_match_numpy_oracle_64x128():
    """Pure-Python loops vs the NumPy oracle on the 64 x 128 fp32 case."""
    rng = np.random.default_rng(11)
    P, G, M = (rng.standard_normal((64, 128)).astype(np.float32).astype(np.float64)
               for _ in range(3))
    beta, lr, wd, k, eps = float(np.float32(0.95)), float(np.float32(0.02)), 0.0, 5, 1e-7
    t = time.time()
    nP, nM, nO = naive_update(P.tolist(), G.tolist(), M.tolist(), beta, lr, wd, k,
                              A_, B_, C_, eps, 1.0)
    assert time.time() - t < 120
    rP, rM, rO = muon_ref.muon_update_ref(P, G, M, beta, lr, wd, k, A_, B_, C_, eps)
    assert np.linalg.norm(np.array(nO) - rO) <= 1e-12 * np.linalg.norm(rO)
    assert np.max(np.abs(np.array(nP) - rP)) <= 1e-12
    assert np.array_equal(np.array(nM), rM)


def test_naive_loops_match_tall():
    rng = np.random.default_rng(12)
    P, G, M = (rng.standard_normal((19, 6)) for _ in range(3))
    s = math.sqrt(19 / 6)
    nP, _, nO = naive_update(P.tolist(), G.tolist(), M.tolist(), 0.9, 0.1, 0.1, 4,
                             A_, B_, C_, 1e-7, s)
    rP, _, rO = muon_ref.muon_update_ref(P, G, M, 0.9, 0.1, 0.1, 4, A_, B_, C_, 1e-7)
    assert np.linalg.norm(np.array(nO) - rO) <= 1e-12 * np.linalg.norm(rO)
    assert np.max(np.abs(np.array(nP) - rP)) <= 1e-12


def _golden_shapes(case):
    s = case["shapes"]
    if "repeat" in s:
        return [s["shape"]] * s["repeat"]
    return s["list"]


def test_bucketing_matches_pages_examples():
    cases = json.load(open(os.path.join(HERE, "golden", "pages_shapes.json"), encoding="utf-8"))["cases"]
    for case in cases:
        groups = muon_ref.bucket_shapes(_golden_shapes(case))
        got = [{"rows": g["rows"], "cols": g["cols"], "batch": len(g["members"])} for g in groups]
        assert got == case["groups"], case["cite"]


def test_bucketing_order_and_expansion():
    shapes = [[4, 8], [3, 8, 4], [4, 8], [2, 3, 8], [8, 4]]
    g = muon_ref.bucket_shapes(shapes)
    assert [(x["rows"], x["cols"]) for x in g] == [(4, 8), (8, 4), (3, 8)]
    assert g[0]["members"] == [(0, 0), (2, 0)]
    assert g[1]["members"] == [(1, 0), (1, 1), (1, 2), (4, 0)]
    assert g[2]["members"] == [(3, 0), (3, 1)]
    for bad in ([[0, 4]], [[4]], [[1, 2, 3, 4]], [[2, 0, 3]]):
        with pytest.raises(ValueError):
            muon_ref.bucket_shapes(bad)


def test_scale_factor_values():
    assert muon_ref.scale_factor(4096, 16384) == 1.0
    assert muon_ref.scale_factor(16384, 4096) == 2.0
    assert muon_ref.scale_factor(24, 10240, "rms_0_2") == pytest.approx(0.2 * math.sqrt(10240), rel=1e-15)
    assert muon_ref.scale_factor(7, 5, "none") == 1.0
    with pytest.raises(ValueError):
        muon_ref.scale_factor(2, 2, "bogus")


def test_ns_band_for_normalised_inputs():
    """Band of p^5 and p^10 over normalised sigma in [0.01, 1]: recomputed by
    iteration, then checked on oracle outputs of random 24 x 96 inputs."""
    from oracle_pins import p_iter
    grid = np.linspace(0.01, 1.0, 20001)
    for k in (5, 10):
        band = p_iter(grid, k)
        lo, hi = band.min(), band.max()
        assert 0.5 < lo < 0.8 and 1.0 < hi < 1.3
        rng = np.random.default_rng(k)
        for _ in range(3):
            O = muon_ref.orthogonalize(rng.standard_normal((24, 96)), k, A_, B_, C_, 1e-7)
            s = np.linalg.svd(O, compute_uv=False)
            assert s.min() >= lo - 1e-9 and s.max() <= hi + 1e-9


def test_package_exports():
    assert oracle.NS_COEFFS_QUINTIC == (A_, B_, C_)
    assert set(oracle.SCALE_MODES) == {"sqrt_aspect", "rms_0_2", "none"}


def test_naive_loops_match_nesterov_and_schedule():
    """The pure-Python loops and the NumPy oracle agree on the Nesterov input
    and on a per-step schedule (tall matrix: the transposed iteration)."""
    from oracle_pins import SCHEDULE
    rng = np.random.default_rng(9)
    P, G, M = (rng.standard_normal((12, 5)) for _ in range(3))
    s = muon_ref.scale_factor(12, 5)
    for nest, sched in ((True, None), (False, SCHEDULE), (True, SCHEDULE)):
        rP, rM, rO = muon_ref.muon_update_ref(P, G, M, 0.9, 0.05, 0.1, 6, A_, B_, C_, 1e-7, "sqrt_aspect",
                                              nest, sched)
        nP, nM, nO = naive_update(P.tolist(), G.tolist(), M.tolist(), 0.9, 0.05, 0.1, 6, A_, B_, C_, 1e-7, s,
                                  nesterov=nest, rows_abc=sched)
        assert np.max(np.abs(np.array(nO) - rO)) <= 1e-12
        assert np.max(np.abs(np.array(nP) - rP)) <= 1e-12
        assert np.max(np.abs(np.array(nM) - rM)) == 0.0
