"""Host-side helpers of bench.py and the workload module (CPU only): the
algorithmic work counts, the executed share of the symmetric GEMMs, the
roofline ridge, and the per-group mixed-bag workloads."""
import math
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from newton_schulz_bucket_gb300 import workloads as W  # noqa: E402


def test_algorithmic_work_counts():
    # c2: 14 B per element, dense k (4 m^2 n + 2 m^3) per matrix
    w = W.get("c2_skinny_74x24x10240")
    b, f = bench.algorithmic_work(w.shapes, w.mode, w.ns_steps)
    assert b == 74 * 24 * 10240 * 14
    assert f == 74 * 5 * (4 * 24 * 24 * 10240 + 2 * 24 ** 3)
    # an expert tensor counts E matrices; a tall matrix iterates on its transpose
    b, f = bench.algorithmic_work([[3, 512, 2048], [2048, 512]], "bf16", 2)
    assert b == 4 * 512 * 2048 * 14
    assert f == 4 * 2 * (4 * 512 * 512 * 2048 + 2 * 512 ** 3)


def test_executed_flop_fraction():
    # m = 4096, BN = 256: 272 of the 512 tiles of each symmetric product
    m, n = 4096, 12288
    sym = 272 / 512
    want = (sym * (2 * m * m * n + 2 * m ** 3) + 2 * m * m * n) / (4 * m * m * n + 2 * m ** 3)
    assert bench.executed_flop_fraction(m, n) == pytest.approx(want, rel=1e-12)
    assert bench.executed_flop_fraction(n, m) == pytest.approx(want, rel=1e-12)
    # one tile per product: nothing to skip
    assert bench.executed_flop_fraction(128, 4096) == 1.0
    # square: between 2/3 and 1
    f = bench.executed_flop_fraction(7168, 7168)
    assert 2 / 3 < f < 0.7


def test_roofline_ridge_splits_the_mixed_bag():
    """Groups whose dense FLOPs per compulsory byte fall below the ridge
    (measured bf16 rate / copy rate) are HBM-bound: the skinny shapes and
    [128, 4096]; [512, 2048] and larger are tensor-bound."""
    peaks = bench.load_peaks()
    ridge = peaks["bf16_tflops_sustained"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    intensity = {}
    for s in W.C5_SHAPES:
        b, f = bench.algorithmic_work([s], "bf16", 5)
        intensity[tuple(s)] = f / b
    for s in ([24, 10240], [64, 7168], [128, 4096]):
        assert intensity[tuple(s)] < ridge, s
    for s in ([512, 2048], [1024, 1024], [4096, 4096], [7168, 7168]):
        assert intensity[tuple(s)] > ridge, s


def test_mixed_bag_group_workloads():
    full = W.get("c5_mixed_1000")
    counts = W.c5_counts(5)
    for s, n in zip(W.C5_SHAPES, counts):
        g = W.get(f"c5_group_{s[0]}x{s[1]}")
        assert g.shapes == [s] * n and len(g.g_std) == n
    assert sum(counts) == 1000 == len(full.shapes)
    with pytest.raises(KeyError):
        W.get("c5_group_3x3")


def test_cpu_baseline_thread_count_and_blas():
    """cores = CPU time over wall time, rounded up, at least 1; the BLAS name
    is a string whatever NumPy reports."""
    assert bench.busy_cores(2.0, 2.0) == 1
    assert bench.busy_cores(1.0, 7.2) == 8
    assert bench.busy_cores(1.0, 7.96) == 8
    assert bench.busy_cores(1.0, 0.3) == 1
    assert bench.busy_cores(0.0, 0.0) == 1
    assert isinstance(bench.blas_name(), str) and bench.blas_name()


def test_host_member_inputs_draw_single_members():
    """The oracle's timing inputs: one [rows, cols] member at a time, with
    the member's own law (per-expert stds of a 3-D parameter included)."""
    w = W.custom([[3, 40, 96], [24, 64]], seed=4)
    w.g_std = [[1e-4, 1e-3, 1e-2], 1e-3]
    get = bench.host_member_inputs(w)
    for (i, e), std in [((0, 0), 1e-4), ((0, 2), 1e-2), ((1, 0), 1e-3)]:
        P, G, M = get(i, e)
        assert P.shape == G.shape == M.shape == tuple(w.shapes[i][-2:])
        assert P.dtype == G.dtype == M.dtype
        assert abs(float(G.std()) / std - 1) < 0.1 and abs(float(M.std()) / std - 1) < 0.1
        assert abs(float(P.std()) / 0.02 - 1) < 0.1
    a, b = get(0, 1), get(0, 1)
    assert all((x == y).all() for x, y in zip(a, b))


def test_oracle_estimate_samples_and_extrapolates():
    """The CPU baseline's estimate: with a generous budget every group is
    timed (members of the cheapest first); with a tiny one only the cheapest
    group is, and the others are extrapolated by FLOPs at the measured rate."""
    w = W.custom([[24, 512]] * 3 + [[96, 256]] * 2 + [[160, 320]], seed=5)
    get = bench.host_member_inputs(w)
    t, wall, cpu, note = bench.oracle_estimate(w, 30.0, get)
    assert t > 0 and wall > 0 and cpu >= 0
    assert "extrapolated" not in note
    assert note.count(" of ") == 3
    t2, _, _, note2 = bench.oracle_estimate(w, 1e-9, get)
    assert t2 > 0 and note2.count(" of ") == 1 and "extrapolated" in note2
    assert "[24, 512]" in note2.split("extrapolated")[0]


def test_report_groups_match_the_planner():
    """bench.py restates the planner's default bucketing and path choice in
    Python (so its reference arm never loads the library); it must agree
    with muon_plan_describe on every configuration."""
    import newton_schulz_bucket_gb300 as pkg
    for name in W.ALL:
        w = W.get(name)
        want = [{k: g[k] for k in ("rows", "cols", "batch", "path")}
                for g in pkg.describe(w.shapes, mode=w.mode)["groups"]]
        assert bench.shape_groups(w.shapes, w.mode) == want, name


def test_path_option():
    """--path forces one kernel path on every group's plan (and is recorded in
    the line's config); the default leaves the choice to the planner."""
    class A:
        path = "auto"
    assert bench.plan_options(A()) == {}
    A.path = "resident"
    assert bench.plan_options(A()) == {"path": "resident"}
