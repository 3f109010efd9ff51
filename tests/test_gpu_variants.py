"""GPU parity of the step's variants against the oracle: per-step coefficient
schedules (muon_step_schedule) and the Nesterov input U = G + beta M'
(MUON_FLAG_NESTEROV), on every path."""
import ctypes as C

import numpy as np
import pytest
import torch

import newton_schulz_bucket_gb300 as pkg
from newton_schulz_bucket_gb300 import workloads as W

from oracle_pins import SCHEDULE
from parity import GpuRun, check_all

pytestmark = pytest.mark.gpu

# (shapes, plan options, ns_steps): one case per path
PATHS = [
    ([[24, 4096], [40, 1000], [2, 64, 2048]], {}, 6),      # skinny, Gram space (m <= 64)
    ([[24, 2048], [48, 1000]], {}, 70),                     # skinny, direct iteration (k > 64)
    ([[256, 512], [512, 256]], {}, 6),                      # tensor cores (tcgen05)
    ([[96, 200], [2, 70, 33]], {"path": "simt"}, 6),        # SIMT, bf16 mode
    ([[128, 1000], [1000, 128], [2, 96, 520], [100, 700]], {"path": "resident"}, 6),  # resident
]
IDS = ["gram_space", "direct", "tensor", "simt", "resident"]


def _workload(shapes, k, seed, mode="bf16", **kw):
    w = W.custom(shapes, mode=mode, seed=seed, ns_steps=k)
    for key, v in kw.items():
        setattr(w, key, v)
    return w


@pytest.mark.parametrize("shapes,opts,k", PATHS, ids=IDS)
def test_schedule_matches_oracle(shapes, opts, k):
    w = _workload(shapes, k, 31, coeffs=SCHEDULE)
    run = GpuRun(w, **opts)
    check_all(run)
    run.close()


def _long_run_coeffs(k):
    """Beyond a few steps the constant quintic does not converge: singular
    values keep moving inside [0.68, 1.13] under a map that stretches some
    distances, so two roundings (fp16 iterate vs the fp64 oracle) drift
    apart.  Long runs therefore end in the contractive textbook map (the
    schedule's last row), under which the two agree."""
    return SCHEDULE if k > 10 else pkg.QUINTIC


@pytest.mark.parametrize("shapes,opts,k", PATHS, ids=IDS)
def test_nesterov_matches_oracle(shapes, opts, k):
    w = _workload(shapes, 5 if k < 64 else k, 32, nesterov=True, coeffs=_long_run_coeffs(k))
    run = GpuRun(w, **opts)
    check_all(run)
    run.close()


def test_fp32_mode_schedule_and_nesterov():
    w = _workload([[64, 128], [30, 70]], 7, 33, mode="fp32", coeffs=SCHEDULE, nesterov=True)
    run = GpuRun(w)
    errs = check_all(run)
    assert max(errs) <= 1e-4
    run.close()


def test_one_row_schedule_equals_constant_coefficients():
    """A one-row schedule is muon_step itself: same bits on every path."""
    shapes = [[24, 4096], [256, 512], [24, 2048]]
    w = W.custom(shapes, seed=34, ns_steps=5)
    outs = []
    for coeffs in (pkg.QUINTIC, [pkg.QUINTIC]):
        P, G, M = W.make_tensors(w, "cuda")
        plan = pkg.MuonPlan(w.shapes)
        plan.step(P, G, M, w.beta, w.lr, w.wd, 5, coeffs)
        torch.cuda.synchronize()
        outs.append([t.clone() for t in P + M])
        plan.close()
    for x, y in zip(*outs):
        assert torch.equal(x, y)


def test_nesterov_batch_invariance_bitwise():
    """Under Nesterov a member alone equals the member inside a batch."""
    w = W.custom([[24, 4096]] * 6 + [[64, 1024]] * 3, seed=35)
    w.nesterov = True
    P, G, M = W.make_tensors(w, "cuda")
    keep = [t.clone() for t in P + G + M]
    full = GpuRun(w, tensors=(P, G, M))
    n = len(w.shapes)
    for i in (4, 7):
        sub = W.custom([w.shapes[i]], seed=0)
        sub.nesterov = True
        one = GpuRun(sub, tensors=([keep[i].clone()], [keep[n + i].clone()], [keep[2 * n + i].clone()]))
        assert np.array_equal(one.p1(0), full.p1(i))
        assert np.array_equal(one.m1(0), full.m1(i))
        assert np.array_equal(one.O(0), full.O(i))
        one.close()
    full.close()


def test_schedule_argument_errors():
    w = W.custom([[24, 512]], seed=36)
    P, G, M = W.make_tensors(w, "cuda")
    plan = pkg.MuonPlan(w.shapes)
    L = pkg.load_library()
    Pp, Gp, Mp = plan.bind(P, G, M)
    st = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    rows = (C.c_float * 6)(3.0, -3.2, 1.2, float("nan"), 0.0, 0.0)
    for ptr, n in ((rows, 0), (rows, 65), (None, 1), (rows, 2)):
        r = L.muon_step_schedule(plan._h, Pp, Gp, Mp, 0.9, 0.02, 0.1, 5, ptr, n, st)
        assert r == 1, (n, r)  # MUON_ERR_INVALID_ARG
    assert L.muon_step_schedule(plan._h, Pp, Gp, Mp, 0.9, 0.02, 0.1, 5, rows, 1, st) == 0
    torch.cuda.synchronize()
    plan.close()


# orientation-merged buckets (MUON_FLAG_MERGE_TRANSPOSED): one case per path
MERGED = [
    ([[24, 4096], [4096, 24], [2, 24, 4096], [64, 1000], [1000, 64]], {}, 5),   # skinny, Gram space
    ([[24, 2048], [2048, 24]], {}, 70),                                         # skinny, direct
    ([[256, 512], [512, 256], [2, 512, 256]], {}, 5),                           # tensor cores
    ([[96, 200], [200, 96]], {"path": "simt"}, 5),                              # SIMT
    ([[128, 1000], [1000, 128], [2, 100, 700], [700, 100]], {"path": "resident"}, 5),  # resident
]


@pytest.mark.parametrize("shapes,opts,k", MERGED, ids=IDS)
def test_merged_orientations_match_oracle_and_unmerged_plan(shapes, opts, k):
    """[r, c] and [c, r] in one group: every member matches the oracle, and
    equals, bit for bit, the same member in a plan with separate groups."""
    w = W.custom(shapes, seed=37, ns_steps=k)
    w.coeffs = _long_run_coeffs(k)
    P, G, M = W.make_tensors(w, "cuda")
    keep = [[t.clone() for t in ts] for ts in (P, G, M)]
    merged = GpuRun(w, tensors=(P, G, M), merge_transposed=True, **opts)
    assert any(g["transposed"] == "mixed" for g in merged.plan.groups())
    assert len(merged.plan.groups()) < len(pkg.describe(shapes, **opts)["groups"])
    check_all(merged)
    sep = GpuRun(w, tensors=tuple([t.clone() for t in ts] for ts in keep), **opts)
    for (i, e) in merged.members:
        assert np.array_equal(merged.p1(i, e), sep.p1(i, e))
        assert np.array_equal(merged.m1(i, e), sep.m1(i, e))
        assert np.array_equal(merged.O(i, e), sep.O(i, e))
    merged.close()
    sep.close()


def test_merged_orientations_fp32_mode():
    w = W.custom([[30, 70], [70, 30], [64, 128]], mode="fp32", seed=38, ns_steps=5)
    run = GpuRun(w, merge_transposed=True)
    assert len(run.plan.groups()) == 2
    errs = check_all(run)
    assert max(errs) <= 1e-4
    run.close()


# column shards on the skinny path (plan option column_shards): one CTA per
# contiguous column shard, partial Grams and sums of squares added in shard
# order through distributed shared memory
@pytest.mark.parametrize("t", [1, 4, 8])
def test_column_shards_match_oracle(t):
    w = W.custom([[24, 4096], [64, 1000], [2, 40, 3000], [4096, 24], [17, 333]], seed=39)
    run = GpuRun(w, column_shards=t)
    assert all(g["path"] == "skinny" for g in run.plan.groups())
    check_all(run)
    run.close()


def test_column_shards_direct_iteration():
    w = W.custom([[24, 2048], [48, 1000]], seed=40, ns_steps=70)
    w.coeffs = SCHEDULE
    run = GpuRun(w, column_shards=4)
    check_all(run)
    run.close()


def test_column_shards_batch_invariance_bitwise():
    """For a fixed shard count a member alone equals the member in a batch."""
    w = W.custom([[24, 4096]] * 5, seed=41)
    P, G, M = W.make_tensors(w, "cuda")
    keep = [[t.clone() for t in ts] for ts in (P, G, M)]
    full = GpuRun(w, tensors=(P, G, M), column_shards=8)
    sub = W.custom([w.shapes[3]], seed=0)
    one = GpuRun(sub, tensors=([keep[0][3]], [keep[1][3]], [keep[2][3]]), column_shards=8)
    assert np.array_equal(one.p1(0), full.p1(3))
    assert np.array_equal(one.O(0), full.O(3))
    one.close()
    full.close()


@pytest.mark.parametrize("k", [5, 70])
def test_all_options_together(k):
    """Nesterov, a per-step schedule, merged orientations and 4 column shards
    at once, on skinny (Gram-space or direct) and tensor groups."""
    w = W.custom([[24, 4096], [4096, 24], [2, 64, 1000], [256, 512], [512, 256]], seed=42, ns_steps=k)
    w.nesterov = True
    w.coeffs = SCHEDULE
    run = GpuRun(w, merge_transposed=True, column_shards=4)
    assert len(run.plan.groups()) == 3
    check_all(run)
    run.close()
