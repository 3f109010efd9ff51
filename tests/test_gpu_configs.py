"""Full-size workloads in the launch configuration bench.py times, checked on
sampled members: every shape group of every config has at least one member
compared with the CPU oracle element by element (up to about 20 TFLOP of
fp64 per test for the largest shapes), and further members are checked by
bitwise equality with the same member computed alone (batch invariance) or
by the spectral property the iteration must satisfy."""
import time

import numpy as np
import pytest
import torch

from newton_schulz_bucket_gb300 import workloads as W
from oracle_pins import p_iter

from parity import GpuRun, check_member

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _alone(run, i, e):
    """The member (i, e) of a finished run, recomputed in a plan of its own."""
    w = run.w
    shp = w.shapes[i]
    one = W.custom([shp[-2:]], mode=w.mode, seed=0)
    one.beta, one.lr, one.wd, one.ns_steps = w.beta, w.lr, w.wd, w.ns_steps
    dev = torch.device("cuda")
    pdt = torch.bfloat16 if w.mode == "bf16" else torch.float32
    P = torch.tensor(run.p0(i, e), dtype=torch.float32, device=dev).to(pdt)
    G = torch.tensor(run.g0(i, e), dtype=torch.float32, device=dev).to(pdt)
    M = torch.tensor(run.m0(i, e), dtype=torch.float32, device=dev)
    return GpuRun(one, tensors=([P], [G], [M]))


def _assert_same(run, i, e, alone):
    assert np.array_equal(alone.p1(0), run.p1(i, e))
    assert np.array_equal(alone.m1(0), run.m1(i, e))
    assert np.array_equal(alone.O(0), run.O(i, e))


def _spectral_check(run, i, e):
    """O O^T (wide side) has the eigenvectors of X0 X0^T and eigenvalues
    p^k(sigma)^2: check u^T (O O^T) u against p^k(sigma)^2 on all eigenpairs."""
    w = run.w
    Mp = run.m1(i, e)
    O = run.O(i, e)
    if Mp.shape[0] > Mp.shape[1]:
        Mp, O = Mp.T, O.T
    X0 = Mp / (np.linalg.norm(Mp) + 1e-7)
    evals, U = np.linalg.eigh(X0 @ X0.T)
    sig = np.sqrt(np.maximum(evals, 0))
    want = p_iter(sig, w.ns_steps) ** 2
    OU = O.T @ U
    got = np.einsum("ij,ij->j", OU, OU)
    rel = np.linalg.norm(got - want) / np.linalg.norm(want)
    assert rel <= 4e-2, f"spectral rel err {rel:.3e}"


def test_c3_moe_and_skinny_full_size():
    w = W.get("c3_moe_64x2048x7168_32x24x10240")
    run = GpuRun(w, sample=[(0, 0), (0, 37), (0, 63), (1, 0), (1, 19), (1, 31)])
    paths = {(g["rows"], g["cols"]): g["path"] for g in run.plan.groups()}
    assert paths == {(2048, 7168): "tensor", (24, 10240): "skinny"}
    t = time.time()
    for (i, e) in [(0, 0), (0, 37), (1, 0), (1, 19), (1, 31)]:
        check_member(run, i, e)
    print(f"c3 oracle on 5 members: {time.time() - t:.1f} s")
    alone = _alone(run, 0, 63)
    _assert_same(run, 0, 63, alone)
    alone.close()
    run.close()


def test_c4_dense_full_size():
    """One member of each of the four groups against the oracle, element by
    element (about 20 TFLOP of fp64 on the host), plus the spectral property
    and alone == batched on others."""
    w = W.get("c4_dense_h4096")
    run = GpuRun(w, sample=[(1, 0), (0, 0), (126, 0), (3, 0), (127, 0), (64, 0)])
    groups = run.plan.groups()
    assert [g["path"] for g in groups] == ["tensor"] * 4 and groups[3]["transposed"]
    for i in (1, 0, 126, 3):  # [4096, 4096], [4096, 12288], [4096, 16384], [16384, 4096]
        t = time.time()
        check_member(run, i, 0)
        print(f"c4 oracle {w.shapes[i]}: {time.time() - t:.1f} s")
    _spectral_check(run, 127, 0)             # a second [16384, 4096] member (layer 31)
    for i in (64, 127):                      # [4096, 12288] and [16384, 4096]: alone == batched
        alone = _alone(run, i, 0)
        _assert_same(run, i, 0, alone)
        alone.close()
    run.close()


@pytest.mark.parametrize("k", [5, 10])
def test_c5_mixed_full_size(k):
    w = W.get("c5_mixed_1000", ns_steps=k)
    counts = W.c5_counts()
    starts = np.cumsum([0] + counts)
    # the first and last member of shapes 0-4 and the first of every larger
    # shape against the oracle; at k = 10 the three largest shapes are
    # checked alone == batched instead (their k = 5 oracle runs cover them)
    oracle_members = sorted({int(starts[s]) for s in range(12 if k == 5 else 9)} |
                            {int(starts[s + 1] - 1) for s in range(5)})
    alone_members = [int(starts[9] - 1), int(starts[12] - 1)]
    run = GpuRun(w, sample=[(i, 0) for i in oracle_members + alone_members])
    assert len(run.plan.groups()) == 12
    for i in oracle_members:
        t = time.time()
        check_member(run, i, 0)
        if w.shapes[i][0] * w.shapes[i][1] >= 2 ** 24:
            print(f"c5 oracle (k={k}) {w.shapes[i]}: {time.time() - t:.1f} s")
    for i in alone_members:                  # [4096, 4096] and [7168, 7168]: alone == batched
        alone = _alone(run, i, 0)
        _assert_same(run, i, 0, alone)
        alone.close()
    run.close()
