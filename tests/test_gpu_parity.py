"""GPU parity: the C-ABI path against the CPU oracle on seeded inputs."""
import numpy as np
import pytest
import torch

import newton_schulz_bucket_gb300 as pkg
from newton_schulz_bucket_gb300 import workloads as W

from parity import F32, GpuRun, check_all

pytestmark = pytest.mark.gpu


def test_c1_fp32_64x128():
    run = GpuRun(W.get("c1_fp32_64x128"))
    assert run.plan.groups()[0]["path"] == "simt"
    errs = check_all(run)
    assert max(errs) <= 1e-4
    run.close()


def test_c2_skinny_74x24x10240_all_members():
    run = GpuRun(W.get("c2_skinny_74x24x10240"))
    g = run.plan.groups()
    assert len(g) == 1 and g[0]["batch"] == 74 and g[0]["path"] == "skinny"
    errs = check_all(run)
    assert max(errs) <= 2e-2
    run.close()


SKINNY_SHAPES = [
    [[24, 10240]],
    [[3, 24, 1000]],             # ragged last CTA slice
    [[10240, 24], [4096, 8]],    # transposed (rows > cols)
    [[64, 7168]],                # m = 64
    [[17, 333]],                 # odd dims: scalar (unaligned) access path
    [[1, 64], [64, 1]],          # single row / column
    [[48, 2048], [40, 96]],
    [[5, 16], [16, 16]],
    [[2, 33, 70]],               # 3-D, odd
    [[32, 4096]],                # m = 32: two full m16 tiles
    [[8, 4096], [16, 4096]],     # one m16 tile (half / full)
    [[25, 1000]],                # m = 25, ragged 32-column superblock
    [[24, 1004]],                # cols % 8 != 0: scalar access path
    [[56, 3000]],                # m = 56: last m16 tile padded, ragged superblock
    [[2048, 36], [7168, 64]],    # transposed, three and four m16 tiles
    [[4, 64, 1504]],             # 3-D, m = 64
    [[1000, 24], [3000, 40]],    # transposed, ragged last block of 32 rows
    [[2, 520, 16], [4104, 64]],  # transposed 3-D, m = 16; m = 64 with a ragged block
]


@pytest.mark.parametrize("shapes", SKINNY_SHAPES, ids=lambda s: "x".join("_".join(map(str, t)) for t in s))
def test_skinny_shapes(shapes):
    run = GpuRun(W.custom(shapes, seed=7))
    for g in run.plan.groups():
        assert g["path"] == "skinny", g
    check_all(run)
    run.close()


@pytest.mark.parametrize("shapes", [[[128, 384], [200, 130]], [[2, 70, 33]], [[256, 256]]])
def test_simt_path_bf16_mode(shapes):
    run = GpuRun(W.custom(shapes, seed=8), path="simt")
    check_all(run)
    run.close()


@pytest.mark.parametrize("shapes", [[[24, 700], [700, 24]], [[9, 40]]])
def test_fp32_mode_small(shapes):
    run = GpuRun(W.custom(shapes, mode="fp32", g_std=1.0, p_std=1.0, seed=9))
    check_all(run)
    run.close()


def test_bf16_ns_operands_k5():
    w = W.custom([[24, 10240]] * 4 + [[64, 7168]], seed=10)
    run = GpuRun(w, ns_dtype="bf16")
    check_all(run)
    run.close()


def test_scale_mode_rms():
    run = GpuRun(W.custom([[24, 4096], [4096, 24]], seed=11), scale="rms_0_2")
    check_all(run, scale_mode="rms_0_2")
    run.close()


def test_ns_steps_zero_and_ten():
    for k in (0, 10):
        w = W.custom([[24, 10240], [3, 40, 640]], seed=12, ns_steps=k)
        run = GpuRun(w)
        check_all(run)
        run.close()


def test_spread_spectrum_inputs():
    """Momenta whose singular values fall log-evenly over several decades,
    unlike the concentrated spectra of Gaussian draws: two decades in bf16
    mode on every path (Gram-space wide and transposed members, m = 64
    experts, tensor path), four in fp32 mode."""
    run = GpuRun(W.custom([[24, 4096], [4096, 24], [2, 64, 2048], [256, 1024], [200, 600]],
                          seed=31, spectrum_decades=2))
    check_all(run)
    run.close()
    run = GpuRun(W.custom([[64, 128], [24, 4096], [128, 512]], mode="fp32", seed=31,
                          spectrum_decades=4))
    check_all(run)
    run.close()


@pytest.mark.parametrize("ns_dtype,margin", [("fp16", 5e-3), ("bf16", 1e-2)])
def test_four_decade_spectra_on_the_skinny_path(ns_dtype, margin):
    """Four decades in bf16 mode on the skinny shapes of the pages' batch and
    the mixed bag, wide and transposed.  Five steps stretch the small
    directions by up to a^5 (about 486), so a single 16-bit rounding of X0
    would use most of the 2e-2 budget with fp16 operands (emulated 1.6e-2)
    and exceed it with bf16 (1.3e-1).  The Gram-space kernel reads X0 as a
    16-bit high part plus residual in its final product O = Pi X0, which keeps
    the error well inside: each member must land within `margin`."""
    w = W.custom([[24, 10240], [64, 7168], [10240, 24], [7168, 64]], seed=33,
                 spectrum_decades=4)
    run = GpuRun(w, ns_dtype=ns_dtype)
    assert {g["path"] for g in run.plan.groups()} == {"skinny"}
    errs = check_all(run)
    assert max(errs) <= margin, errs
    run.close()


@pytest.mark.parametrize("shape,k,path", [([24, 2048], 5, "auto"), ([2048, 40], 5, "auto"),
                                          ([24, 2048], 70, "auto"), ([256, 768], 5, "tensor"),
                                          ([128, 1024], 5, "resident"), ([1000, 100], 5, "resident")],
                         ids=["gram_space", "gram_space_transposed", "direct_k70", "tensor",
                              "resident", "resident_transposed"])
def test_zero_gradient_and_momentum(shape, k, path):
    """M' = 0 gives X = 0, O = 0 and P' = P (1 - lr wd) exactly: one fp32
    rounding of 1 - lr wd, one of the product, then round-to-nearest-even to
    bf16 -- on every kernel that writes P."""
    w = W.custom([shape], seed=13, g_std=0.0, m_zero=True, ns_steps=k, lr=0.3, wd=0.7)
    run = GpuRun(w, path=path)
    assert np.all(run.O(0) == 0)
    decay = np.float32(1.0 - np.float64(np.float32(w.lr)) * np.float64(np.float32(w.wd)))
    want = torch.tensor(run.p0(0).astype(np.float32) * decay, dtype=torch.float32)
    want = want.to(torch.bfloat16).double().numpy()
    assert np.array_equal(run.p1(0), want)
    assert np.all(run.m1(0) == 0)
    run.close()


@pytest.mark.parametrize("k,rows", [(10, 24), (64, 24), (64, 64)])
def test_gram_space_zero_rows(k, rows):
    """Zero rows of M' are exact null directions of X_0, along which the
    Gram-space product Pi_k = Q_{k-1} ... Q_0 grows like a^k: O keeps them
    exactly zero and the other rows match the oracle."""
    w = W.custom([[rows, 4096]], seed=21, ns_steps=k)
    P, G, M = W.make_tensors(w, "cuda")
    zero = (3, 20, rows - 1)
    for r in zero:
        G[0][r] = 0
        M[0][r] = 0
    run = GpuRun(w, tensors=(P, G, M))
    check_all(run)
    O = run.O(0)
    assert np.all(np.isfinite(O)) and np.all(O[list(zero)] == 0)
    run.close()


def test_many_steps_direct_iteration():
    """Step counts beyond the Gram-space range run the direct iteration.  The
    run ends in the contractive textbook map (see the schedule's last row):
    under the constant quintic, 70 fp16-rounded steps drift from the fp64
    oracle (singular values keep moving inside [0.68, 1.13]) for some inputs."""
    from oracle_pins import SCHEDULE
    w = W.custom([[24, 2048], [2, 16, 512], [64, 1024], [40, 512]], seed=22, ns_steps=70)
    w.coeffs = SCHEDULE
    run = GpuRun(w)
    check_all(run)
    run.close()


def _member_tensors(w, idx):
    """Inputs of a sub-workload made of members `idx` of w (exact copies)."""
    P, G, M = W.make_tensors(w, "cuda")
    return [P[i].clone() for i in idx], [G[i].clone() for i in idx], [M[i].clone() for i in idx]


def test_batch_invariance_bitwise():
    """A member computed inside a batch of 74 equals the same member computed
    alone, and inside a batch of 7, bit for bit (P', M' and O)."""
    w = W.get("c2_skinny_74x24x10240")
    full = GpuRun(w)
    for idx in ([5], [0, 3, 5, 11, 40, 41, 73]):
        sub = W.custom([w.shapes[i] for i in idx], seed=0)
        sub.beta, sub.lr, sub.wd = w.beta, w.lr, w.wd
        run = GpuRun(sub, tensors=_member_tensors(w, idx))
        for j, i in enumerate(idx):
            assert np.array_equal(run.p1(j), full.p1(i))
            assert np.array_equal(run.m1(j), full.m1(i))
            assert np.array_equal(run.O(j), full.O(i))
        run.close()
    full.close()


def test_batch_invariance_bitwise_m64():
    """The same for four 16-row tiles (m = 64): a member alone equals the
    member inside a batch of 9."""
    w = W.custom([[64, 7168]] * 9, seed=23)
    full = GpuRun(w)
    sub = W.custom([w.shapes[6]], seed=0)
    run = GpuRun(sub, tensors=_member_tensors(w, [6]))
    assert np.array_equal(run.p1(0), full.p1(6))
    assert np.array_equal(run.m1(0), full.m1(6))
    assert np.array_equal(run.O(0), full.O(6))
    run.close()
    full.close()


def test_graph_replay_equals_direct_launch():
    w = W.custom([[24, 10240]] * 3 + [[96, 200]] + [[2, 64, 64]], seed=14)
    a = GpuRun(w)
    b = GpuRun(w, no_graph=True)
    for (i, e) in a.members:
        assert np.array_equal(a.p1(i, e), b.p1(i, e))
        assert np.array_equal(a.m1(i, e), b.m1(i, e))
    a.close(); b.close()


def test_three_steps_match_oracle_iterated():
    from oracle import muon_ref
    w = W.custom([[24, 4096], [4096, 24]], seed=15)
    run = GpuRun(w, steps=3)
    a, b, c = run.coeffs
    for i, shp in enumerate(w.shapes):
        P, M = run.p0(i), run.m0(i)
        for _ in range(3):
            P, M, O = muon_ref.muon_update_ref(P, run.g0(i), M, F32(w.beta), F32(w.lr), F32(w.wd),
                                               w.ns_steps, a, b, c)
            P = torch.tensor(P, dtype=torch.float32).to(torch.bfloat16).double().numpy()
            M = M.astype(np.float32).astype(np.float64)
        assert np.max(np.abs(run.m1(i) - M)) <= 1e-5 * np.max(np.abs(M))
        dP_ref, dP = P - run.p0(i), run.p1(i) - run.p0(i)
        assert np.linalg.norm(dP - dP_ref) / np.linalg.norm(dP_ref) <= 3e-2
    run.close()


def test_step_host_equals_device_step():
    w = W.custom([[24, 10240]] * 5 + [[2, 24, 10240]], seed=16)
    P, G, M = W.make_tensors(w, "cuda")
    hP = [t.cpu().pin_memory() for t in P]
    hG = [t.cpu().pin_memory() for t in G]
    hM = [t.cpu().pin_memory() for t in M]
    dev = pkg.MuonPlan(w.shapes)
    host = pkg.MuonPlan(w.shapes, host_staging=True)
    c = tuple(F32(v) for v in w.coeffs)
    dev.step(P, G, M, w.beta, w.lr, w.wd, w.ns_steps, c)
    host.step_host(hP, hG, hM, w.beta, w.lr, w.wd, w.ns_steps, c)
    torch.cuda.synchronize()
    for i in range(len(P)):
        assert torch.equal(P[i].cpu(), hP[i])
        assert torch.equal(M[i].cpu(), hM[i])
    dev.close(); host.close()


@pytest.mark.parametrize("shapes,opts", [
    ([[256, 512], [24, 2048], [512, 256], [256, 512], [2, 64, 768]], {}),
    ([[6, 256, 512], [24, 2048], [300, 256], [5, 96, 640]], {}),
    ([[12, 128, 640], [640, 128], [3, 100, 700]], {"path": "resident"}),
], ids=["groups", "expert_slices", "resident"])
def test_step_host_by_group_equals_device_step(shapes, opts):
    """Plans that are not all skinny pipeline the host step in slices of whole
    members of a group (copy in, kernels, copy out on three streams; slices
    may cut a 3-D parameter): same bits as the device step, over two steps."""
    w = W.custom(shapes, seed=17)
    P, G, M = W.make_tensors(w, "cuda")
    hP = [t.cpu().pin_memory() for t in P]
    hG = [t.cpu().pin_memory() for t in G]
    hM = [t.cpu().pin_memory() for t in M]
    dev = pkg.MuonPlan(w.shapes, **opts)
    host = pkg.MuonPlan(w.shapes, host_staging=True, **opts)
    c = tuple(F32(v) for v in w.coeffs)
    for _ in range(2):
        dev.step(P, G, M, w.beta, w.lr, w.wd, w.ns_steps, c)
        host.step_host(hP, hG, hM, w.beta, w.lr, w.wd, w.ns_steps, c)
    torch.cuda.synchronize()
    for i in range(len(P)):
        assert torch.equal(P[i].cpu(), hP[i])
        assert torch.equal(M[i].cpu(), hM[i])
    dev.close(); host.close()


def test_bound_step_equals_step():
    w = W.custom([[24, 4096]] * 3, seed=19)
    P1, G1, M1 = W.make_tensors(w, "cuda")
    P2, G2, M2 = (list(t.clone() for t in ts) for ts in (P1, G1, M1))
    plan = pkg.MuonPlan(w.shapes)
    plan.step(P1, G1, M1, w.beta, w.lr, w.wd, w.ns_steps, w.coeffs)
    plan.step_bound(plan.bind(P2, G2, M2), w.beta, w.lr, w.wd, w.ns_steps, w.coeffs)
    torch.cuda.synchronize()
    for i in range(3):
        assert torch.equal(P1[i], P2[i]) and torch.equal(M1[i], M2[i])
    plan.close()


def test_group_timing_events():
    w = W.custom([[24, 4096]] * 4 + [[256, 512]] * 2, seed=18)
    P, G, M = W.make_tensors(w, "cuda")
    plan = pkg.MuonPlan(w.shapes, group_timing=True)
    plan.step(P, G, M, w.beta, w.lr, w.wd, w.ns_steps, w.coeffs)
    for g in range(len(plan.groups())):
        assert 0.0 < plan.group_elapsed_ms(g) < 1000.0
    plan.close()


def test_argument_errors():
    w = W.custom([[24, 512]], seed=17)
    P, G, M = W.make_tensors(w, "cuda")
    plan = pkg.MuonPlan(w.shapes)
    with pytest.raises(ValueError):
        plan.step([p.float() for p in P], G, M, 0.9, 0.1, 0.0)
    with pytest.raises(ValueError):
        plan.step(P, G, [m[:, :256] for m in M], 0.9, 0.1, 0.0)
    with pytest.raises(pkg.MuonError) as ei:
        plan.step(P, G, M, 0.9, 0.1, 0.0, ns_steps=-1)
    assert ei.value.status == 1
    with pytest.raises(pkg.MuonError):
        plan.step(P, G, M, float("nan"), 0.1, 0.0)
    with pytest.raises(pkg.MuonError) as ei:
        plan.debug_update(0)
    assert ei.value.status == 2  # plan made without keep_update
    plan.step(P, G, M, 0.9, 0.1, 0.0)
    plan.check_error()
    plan.close()


def test_batch_invariance_bitwise_transposed():
    """The transposed members' vector path: a member of a 74-member batch
    (2-CTA clusters of 16 warps) equals, bit for bit, the same member alone
    and in a batch of 5 (4-CTA clusters of 8 warps)."""
    w = W.custom([[10240, 24]] * 74, seed=25)
    full = GpuRun(w, sample=[(3, 0), (40, 0), (73, 0)])
    for idx in ([40], [3, 9, 40, 41, 73]):
        sub = W.custom([w.shapes[i] for i in idx], seed=0)
        sub.beta, sub.lr, sub.wd = w.beta, w.lr, w.wd
        run = GpuRun(sub, tensors=_member_tensors(w, idx))
        for j, i in enumerate(idx):
            if (i, 0) not in full.members:
                continue
            assert np.array_equal(run.p1(j), full.p1(i))
            assert np.array_equal(run.m1(j), full.m1(i))
            assert np.array_equal(run.O(j), full.O(i))
        run.close()
    full.close()


@pytest.mark.parametrize("case", range(12))
def test_random_skinny_shapes_against_the_oracle(case):
    """Seeded random skinny groups: m in [1, 64], n up to 6000, either
    orientation, 1-3 parameters (some 3-D), k in 0..10 -- across the vector,
    transposed-vector and element-wise paths and both launch forms."""
    rng = np.random.default_rng(1000 + case)
    shapes = []
    for _ in range(int(rng.integers(1, 4))):
        m = int(rng.integers(1, 65))
        n = int(rng.integers(m, 6001))
        if rng.random() < 0.3:
            m = 8 * max(1, m // 8)  # often a multiple of 8 (vector paths)
        r, c = (n, m) if rng.random() < 0.5 else (m, n)
        shapes.append([int(rng.integers(2, 5)), r, c] if rng.random() < 0.3 else [r, c])
    k = int(rng.integers(0, 11))
    w = W.custom(shapes, seed=2000 + case, ns_steps=k)
    run = GpuRun(w)
    for g in run.plan.groups():
        assert g["path"] == "skinny", g
    check_all(run)
    run.close()
