"""GPU tests of the TENSOR path (tcgen05 / TMEM / TMA GEMMs).

The single products are checked against PyTorch fp32 matmuls of the same
16-bit inputs; the whole step against the CPU oracle."""
import ctypes as C

import numpy as np
import pytest
import torch

import newton_schulz_bucket_gb300 as pkg

from newton_schulz_bucket_gb300 import _capi
from newton_schulz_bucket_gb300 import workloads as W

from parity import GpuRun, check_all

pytestmark = pytest.mark.gpu

DT = {"fp16": (torch.float16, 0), "bf16": (torch.bfloat16, 1)}


def _tc(op, dt, B, m, n, y=None, a=None, q=None, out=None, alpha=1.0, pa=0.0, pb=0.0, pc=0.0):
    L = _capi.load()
    ptr = lambda t: None if t is None else C.c_void_p(t.data_ptr())
    st = L.muon_testing_tc_gemm(op, DT[dt][1], B, m, n, ptr(y), ptr(a), ptr(q), ptr(out),
                                alpha, pa, pb, pc, None)
    torch.cuda.synchronize()
    _capi.check(st, "muon_testing_tc_gemm")


def _close(got, ref, dt):
    got, ref = got.float(), ref.float()
    rel = (got - ref).norm() / ref.norm()
    lim = 4e-3 if dt == "fp16" else 2e-2
    assert rel <= lim, f"rel err {rel:.3e}"
    ulp = 2 ** -10 if dt == "fp16" else 2 ** -7
    assert (got - ref).abs().max() <= 4 * ulp * ref.abs().max() + 1e-6


SHAPES = [(1, 128, 256), (2, 256, 512), (3, 384, 1024), (1, 136, 1000), (2, 64, 200),
          (1, 512, 4096), (2, 1024, 2048)]


@pytest.mark.parametrize("dt", ["fp16", "bf16"])
@pytest.mark.parametrize("B,m,n", SHAPES)
def test_tc_gram(dt, B, m, n):
    g = torch.Generator(device="cuda").manual_seed(m * 7 + n)
    y = (torch.randn(B, m, n, device="cuda", generator=g) * 0.5).to(DT[dt][0])
    out = torch.full((B, m, m), float("nan"), device="cuda", dtype=DT[dt][0])
    alpha = 4.0
    _tc(0, dt, B, m, n, y=y, out=out, alpha=alpha)
    ref = torch.bmm(y.float(), y.float().transpose(1, 2)) / alpha ** 2
    _close(out, ref, dt)


@pytest.mark.parametrize("dt", ["fp16", "bf16"])
@pytest.mark.parametrize("B,m,n", SHAPES)
def test_tc_poly(dt, B, m, n):
    g = torch.Generator(device="cuda").manual_seed(m * 11 + n)
    x = torch.randn(B, m, n, device="cuda", generator=g) / (m * n) ** 0.5
    a = torch.bmm(x, x.transpose(1, 2)).to(DT[dt][0])
    out = torch.full((B, m, m), float("nan"), device="cuda", dtype=DT[dt][0])
    pa, pb, pc = 3.4445, -4.7750, 2.0315
    _tc(1, dt, B, m, n, a=a, out=out, pa=pa, pb=pb, pc=pc)
    af = a.float()
    ref = pa * torch.eye(m, device="cuda") + pb * af + pc * torch.bmm(af, af)
    _close(out, ref, dt)


@pytest.mark.parametrize("dt", ["fp16", "bf16"])
@pytest.mark.parametrize("B,m,n", SHAPES)
def test_tc_update(dt, B, m, n):
    g = torch.Generator(device="cuda").manual_seed(m * 13 + n)
    q = (torch.randn(B, m, m, device="cuda", generator=g) / m ** 0.5).to(DT[dt][0])
    y = torch.randn(B, m, n, device="cuda", generator=g).to(DT[dt][0])
    out = torch.full((B, m, n), float("nan"), device="cuda", dtype=DT[dt][0])
    _tc(2, dt, B, m, n, y=y, q=q, out=out)
    ref = torch.bmm(q.float(), y.float())
    _close(out, ref, dt)


TENSOR_SHAPES = [
    [[256, 1024]],
    [[384, 640], [640, 384]],    # wide and transposed
    [[3, 200, 520]],             # 3-D, ragged tiles
    [[130, 700]],                # pitches padded (136, 704)
    [[100, 100], [2, 72, 72]],   # square, m < tile
    [[1024, 4096]],
]


@pytest.mark.parametrize("shapes", TENSOR_SHAPES,
                         ids=lambda s: "x".join("_".join(map(str, t)) for t in s))
def test_tensor_path_parity(shapes):
    run = GpuRun(W.custom(shapes, seed=21), path="tensor")
    for g in run.plan.groups():
        assert g["path"] == "tensor"
    check_all(run)
    run.close()


def test_tensor_path_bf16_operands_and_k10():
    run = GpuRun(W.custom([[256, 768]], seed=22), path="tensor", ns_dtype="bf16")
    check_all(run)
    run.close()
    # bf16 operands rounded on every step are limited to 5 steps (the emulated
    # error reaches 1.7e-2 at 6 steps and 2.5e-2 at 10, against 2e-2); the
    # Gram-space skinny kernel rounds the data once and takes up to 64
    w = W.custom([[256, 768]], seed=22, ns_steps=6)
    P, G, M = W.make_tensors(w, "cuda")
    before = P[0].clone()
    plan = pkg.MuonPlan(w.shapes, path="tensor", ns_dtype="bf16")
    with pytest.raises(pkg.MuonError) as ei:
        plan.step(P, G, M, w.beta, w.lr, w.wd, 6)
    assert ei.value.status == 2  # UNSUPPORTED, nothing launched
    torch.cuda.synchronize()
    assert torch.equal(P[0], before)
    plan.close()
    sk = pkg.MuonPlan([[24, 1024]], ns_dtype="bf16")
    ws = W.custom([[24, 1024]], seed=22)
    P, G, M = W.make_tensors(ws, "cuda")
    sk.step(P, G, M, 0.95, 0.02, 0.1, 10)
    with pytest.raises(pkg.MuonError) as ei:
        sk.step(P, G, M, 0.95, 0.02, 0.1, 70)  # the direct iteration rounds every step
    assert ei.value.status == 2
    sk.close()
    run = GpuRun(W.custom([[24, 4096], [4096, 24]], seed=22, ns_steps=10), ns_dtype="bf16")
    check_all(run)
    run.close()
    run = GpuRun(W.custom([[256, 768], [512, 512]], seed=23, ns_steps=10), path="tensor")
    check_all(run)
    run.close()


def test_tensor_batch_invariance_bitwise():
    w = W.custom([[4, 256, 512]], seed=24)
    P, G, M = W.make_tensors(w, "cuda")
    full = GpuRun(w, path="tensor", tensors=([P[0].clone()], [G[0].clone()], [M[0].clone()]))
    one = W.custom([[1, 256, 512]], seed=0)
    run = GpuRun(one, path="tensor", tensors=([P[0][2:3].clone()], [G[0][2:3].clone()],
                                              [M[0][2:3].clone()]))
    assert np.array_equal(run.p1(0, 0), full.p1(0, 2))
    assert np.array_equal(run.m1(0, 0), full.m1(0, 2))
    assert np.array_equal(run.O(0, 0), full.O(0, 2))
    full.close(); run.close()


@pytest.mark.parametrize("case", range(8))
def test_random_tensor_shapes_against_the_oracle(case):
    """Seeded random tensor-path groups: m in [65, 700] (one-CTA form below
    256, CTA-pair form from 256), n up to 2500, either orientation, ragged
    tiles, sometimes 3-D, k in 1..6."""
    rng = np.random.default_rng(3000 + case)
    shapes = []
    for _ in range(int(rng.integers(1, 3))):
        m = int(rng.integers(65, 701))
        n = int(rng.integers(m, 2501))
        r, c = (n, m) if rng.random() < 0.5 else (m, n)
        shapes.append([2, r, c] if rng.random() < 0.25 else [r, c])
    k = int(rng.integers(1, 7))
    w = W.custom(shapes, seed=4000 + case, ns_steps=k)
    run = GpuRun(w, path="tensor")
    for g in run.plan.groups():
        assert g["path"] == "tensor", g
    check_all(run)
    run.close()
