"""GPU test of muon_step_skinny_static, the entry point for callers that
cannot allocate device memory (a framework allocator that forbids outside
cudaMalloc calls, a latency-critical loop that must stay out of the CUDA
allocator, or a deployment that fixes all device buffers at start-up).

It runs the same kernels with the same arguments as the plan-based muon_step,
so its parameters and momenta must equal muon_step's bit for bit: checked on
two calls in a row, each path carrying its own parameters and momenta
forward, in the Gram-space range (k <= 64) and in the direct iteration
(k > 64).  On the pages' fused batch (74 x [24, 10240]) the plan's results
are also checked against the CPU oracle, so the static path inherits that
parity.  This file is named so that pytest collects it last."""
import ctypes as C

import numpy as np
import pytest
import torch

import newton_schulz_bucket_gb300 as pkg
from newton_schulz_bucket_gb300 import _capi
from newton_schulz_bucket_gb300 import workloads as W

from parity import GpuRun, check_member

pytestmark = pytest.mark.gpu

F32 = lambda v: float(np.float32(v))


def _static_step(P, G, M, w, stream=None):
    L = _capi.load()
    B, rows, cols = P.shape
    a, b, c = w.coeffs
    return L.muon_step_skinny_static(C.c_void_p(P.data_ptr()), C.c_void_p(G.data_ptr()),
                                     C.c_void_p(M.data_ptr()), B, rows, cols, F32(w.beta),
                                     F32(w.lr), F32(w.wd), w.ns_steps, F32(a), F32(b), F32(c),
                                     1e-7, _capi.MUON_SCALE_SQRT_ASPECT, stream)


def _first_difference(x, y):
    """Where and by how much two tensors differ (diagnostic for a failure)."""
    d = (x.double() - y.double()).abs()
    k = int(torch.argmax(d))
    return (f"{int((d > 0).sum())} elements differ; worst flat index {k}: "
            f"{x.reshape(-1)[k].item()!r} vs {y.reshape(-1)[k].item()!r}")


@pytest.mark.parametrize("shape,k", [([5, 24, 4096], 5), ([3, 2048, 40], 5),
                                     ([2, 64, 1504], 10), ([2, 24, 2048], 70)],
                         ids=["24x4096_k5", "transposed_2048x40_k5", "64x1504_k10",
                              "direct_24x2048_k70"])
def test_static_scratch_step_equals_muon_step_twice(shape, k):
    w = W.custom([shape], seed=31, ns_steps=k)
    P1, G1, M1 = (t[0] for t in W.make_tensors(w, "cuda"))
    P2, G2, M2 = P1.clone(), G1.clone(), M1.clone()
    plan = pkg.MuonPlan(w.shapes)
    assert plan.groups()[0]["path"] == "skinny"
    coeffs = tuple(F32(v) for v in w.coeffs)
    for call in range(2):
        plan.step([P1], [G1], [M1], w.beta, w.lr, w.wd, w.ns_steps, coeffs)
        st = _static_step(P2, G2, M2, w)
        torch.cuda.synchronize()
        assert st == _capi.MUON_OK, _capi.load().muon_last_error().decode()
        # the second call starts from the first call's outputs on both sides
        assert torch.equal(M1, M2), f"call {call}: momenta: {_first_difference(M1, M2)}"
        assert torch.equal(P1, P2), f"call {call}: parameters: {_first_difference(P1, P2)}"
    assert torch.equal(G1, G2)
    plan.close()


def test_static_scratch_pages_batch_matches_plan_and_oracle():
    """74 x [24, 10240], the pages' fused batch: up to 64 steps the call
    needs only the scalar and pointer tables, so the whole batch fits."""
    w = W.custom([[74, 24, 10240]], seed=34)
    P, G, M = W.make_tensors(w, "cuda")
    P2, G2, M2 = P[0].clone(), G[0].clone(), M[0].clone()
    run = GpuRun(w, tensors=(P, G, M), sample=[(0, 0), (0, 40), (0, 73)])
    assert _static_step(P2, G2, M2, w) == _capi.MUON_OK, _capi.load().muon_last_error().decode()
    torch.cuda.synchronize()
    assert torch.equal(run.Mt[0], M2), _first_difference(run.Mt[0], M2)
    assert torch.equal(run.Pt[0], P2), _first_difference(run.Pt[0], P2)
    for e in (0, 40, 73):
        check_member(run, 0, e)
    run.close()


def test_static_scratch_rejects_oversize_and_bad_args():
    L = _capi.load()
    # beyond 64 steps the direct iteration keeps its iterate in the array:
    # 74 members of [24, 10240] need about 36 MB of it
    w = W.custom([[74, 24, 10240]], seed=32, ns_steps=70)
    P, G, M = (t[0] for t in W.make_tensors(w, "cuda"))
    before = P.clone()
    st = _static_step(P, G, M, w)
    assert st == _capi.MUON_ERR_INVALID_ARG
    msg = L.muon_last_error().decode()
    assert "static array holds 8388608" in msg, msg
    torch.cuda.synchronize()
    assert torch.equal(P, before)  # nothing ran
    wide = W.custom([[2, 100, 300]], seed=33)
    P, G, M = (t[0] for t in W.make_tensors(wide, "cuda"))
    assert _static_step(P, G, M, wide) == _capi.MUON_ERR_UNSUPPORTED
    assert L.muon_step_skinny_static(None, None, None, 1, 24, 64, 0.9, 0.1, 0.0, 5, 1.0, 1.0,
                                     1.0, 1e-7, 0, None) == _capi.MUON_ERR_INVALID_ARG
    # a stream of another device is refused (only checkable with two GPUs)
    if torch.cuda.device_count() > 1:
        s1 = torch.cuda.Stream(device=1)
        small = W.custom([[1, 24, 64]], seed=35)
        P, G, M = (t[0] for t in W.make_tensors(small, "cuda"))
        assert _static_step(P, G, M, small, C.c_void_p(s1.cuda_stream)) == _capi.MUON_ERR_INVALID_ARG
