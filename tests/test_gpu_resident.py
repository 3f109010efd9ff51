"""GPU parity of the resident path (one kernel per group, the iterate held in
a cluster's shared memory for all k steps; min dim <= 128, max dim <= 4096)
against the oracle, and its batch invariance.  The planner takes it only
when asked for (path="resident").

The shapes cover every access form of its passes: 16-byte vectors along the
parameter's rows (rows <= cols, n % 8 == 0), the 8 x 8 transposing blocks
(rows > cols, m % 8 == 0), the element-wise form for the rest, clusters of
1, 2, 4 and 8 CTAs, ragged last column chunks, and a cluster whose last CTA
owns no column at all ([80, 2049]: 8 CTAs of 320 columns)."""
import numpy as np
import pytest

from newton_schulz_bucket_gb300 import workloads as W
from oracle_pins import SCHEDULE

from parity import GpuRun, check_all

pytestmark = pytest.mark.gpu

CASES = {
    "c5_shape_cluster8": [[2, 128, 4096]],
    "transposed_vectors": [[4096, 128], [1000, 96]],
    "element_wise": [[100, 700], [700, 100], [2, 72, 333]],
    "empty_last_cta": [[80, 2049], [2049, 80]],
    "small_clusters": [[65, 65], [3, 128, 128], [70, 130], [120, 1536]],
    "skinny_sizes": [[24, 4096], [4096, 40], [1, 300]],
}


def _resident(run):
    assert {g["path"] for g in run.plan.groups()} == {"resident"}, run.plan.groups()


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("k", [0, 1, 5, 10])
def test_resident_against_oracle(name, k):
    w = W.custom(CASES[name], seed=61, ns_steps=k)
    run = GpuRun(w, path="resident")
    _resident(run)
    check_all(run)
    run.close()


@pytest.mark.parametrize("scale_mode", ["sqrt_aspect", "rms_0_2"])
def test_resident_merged_orientations(scale_mode):
    w = W.custom([[128, 1000], [1000, 128], [2, 96, 2048]], seed=62)
    run = GpuRun(w, merge_transposed=True, scale=scale_mode, path="resident")
    _resident(run)
    assert run.plan.groups()[0]["transposed"] == "mixed"
    check_all(run, scale_mode=scale_mode)
    run.close()


def test_resident_bf16_operands():
    run = GpuRun(W.custom([[128, 2048], [2048, 96]], seed=63), ns_dtype="bf16", path="resident")
    _resident(run)
    check_all(run)
    run.close()


def test_resident_schedule_and_nesterov():
    w = W.custom([[128, 1024], [1024, 128], [100, 700]], seed=64, ns_steps=6)
    w.coeffs = SCHEDULE
    run = GpuRun(w, path="resident")
    _resident(run)
    check_all(run)
    run.close()
    w = W.custom([[128, 1024], [1024, 128], [100, 700]], seed=65)
    w.nesterov = True
    run = GpuRun(w, path="resident")
    _resident(run)
    check_all(run)
    run.close()


def test_resident_spread_spectrum():
    """Momenta whose singular values spread over two decades."""
    w = W.custom([[128, 4096], [2048, 96]], seed=66, spectrum_decades=2)
    run = GpuRun(w, path="resident")
    _resident(run)
    check_all(run)
    run.close()


def test_resident_batch_invariance_bitwise():
    """Each member runs in its own cluster with a reduction order fixed by the
    shape, so a member computed alone equals the same member inside a batch,
    bit for bit."""
    w = W.custom([[5, 128, 1536]], seed=67)
    P, G, M = W.make_tensors(w, "cuda")
    full = GpuRun(w, tensors=([P[0].clone()], [G[0].clone()], [M[0].clone()]), path="resident")
    _resident(full)
    one = W.custom([[1, 128, 1536]], seed=0)
    run = GpuRun(one, tensors=([P[0][3:4].clone()], [G[0][3:4].clone()], [M[0][3:4].clone()]),
                 path="resident")
    assert np.array_equal(run.p1(0, 0), full.p1(0, 3))
    assert np.array_equal(run.m1(0, 0), full.m1(0, 3))
    assert np.array_equal(run.O(0, 0), full.O(0, 3))
    full.close()
    run.close()


@pytest.mark.parametrize("case", range(6))
def test_random_resident_shapes_against_the_oracle(case):
    """Seeded random resident groups: m in [65, 128], n in [m, 4096], either
    orientation, sometimes 3-D, k in 1..6."""
    rng = np.random.default_rng(5000 + case)
    shapes = []
    for _ in range(int(rng.integers(1, 3))):
        m = int(rng.integers(65, 129))
        n = int(rng.integers(m, 4097))
        r, c = (n, m) if rng.random() < 0.5 else (m, n)
        shapes.append([2, r, c] if rng.random() < 0.25 else [r, c])
    w = W.custom(shapes, seed=6000 + case, ns_steps=int(rng.integers(1, 7)))
    run = GpuRun(w, path="resident")
    _resident(run)
    check_all(run)
    run.close()
