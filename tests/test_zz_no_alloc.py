"""GPU test of muon_step_skinny_static, the entry point for callers that
cannot allocate device memory (a framework allocator that forbids outside
cudaMalloc calls, a latency-critical loop that must stay out of the CUDA
allocator, or a deployment that fixes all device buffers at start-up).

It must give the same update as the plan-based muon_step on the same inputs:
checked on two calls in a row, each path carrying its own parameters and
momenta forward.  This file is named so that pytest collects it last."""
import ctypes as C

import numpy as np
import pytest
import torch

import newton_schulz_bucket_gb300 as pkg
from newton_schulz_bucket_gb300 import _capi
from newton_schulz_bucket_gb300 import workloads as W

pytestmark = pytest.mark.gpu

F32 = lambda v: float(np.float32(v))


def _static_step(P, G, M, w, stream=None):
    L = _capi.load()
    B, rows, cols = P.shape
    a, b, c = w.coeffs
    st = L.muon_step_skinny_static(C.c_void_p(P.data_ptr()), C.c_void_p(G.data_ptr()),
                                   C.c_void_p(M.data_ptr()), B, rows, cols, F32(w.beta),
                                   F32(w.lr), F32(w.wd), w.ns_steps, F32(a), F32(b), F32(c),
                                   1e-7, _capi.MUON_SCALE_SQRT_ASPECT, stream)
    return st


def _bf16_ulp(x):
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(ax)) - 7)


@pytest.mark.parametrize("shape", [[5, 24, 4096], [3, 2048, 40]])
def test_static_scratch_step_matches_muon_step_twice(shape):
    w = W.custom([shape], seed=31)
    P1, G1, M1 = (t[0] for t in W.make_tensors(w, "cuda"))
    P2, G2, M2 = P1.clone(), G1.clone(), M1.clone()
    plan = pkg.MuonPlan(w.shapes)
    assert plan.groups()[0]["path"] == "skinny"
    coeffs = tuple(F32(v) for v in w.coeffs)
    for call in range(2):
        P0 = P1.float().cpu().double().numpy()
        plan.step([P1], [G1], [M1], w.beta, w.lr, w.wd, w.ns_steps, coeffs)
        st = _static_step(P2, G2, M2, w)
        torch.cuda.synchronize()
        assert st == _capi.MUON_OK, _capi.load().muon_last_error().decode()
        p1 = P1.float().cpu().double().numpy()
        p2 = P2.float().cpu().double().numpy()
        m1 = M1.cpu().double().numpy()
        m2 = M2.cpu().double().numpy()
        # momentum: fp32 of the same inputs, 1e-6 relative per element
        assert np.all(np.abs(m1 - m2) <= 1e-6 * np.abs(m1) + 1e-38), f"call {call}: momentum"
        # update: relative Frobenius within the bf16-mode tolerance (2e-2) and
        # each element within one bf16 ulp of the other entry point's result
        d1, d2 = p1 - P0, p2 - P0
        assert np.linalg.norm(d2 - d1) <= 2e-2 * np.linalg.norm(d1), f"call {call}: update"
        assert np.all(np.abs(p1 - p2) <= _bf16_ulp(p1)), f"call {call}: parameters"
        # the second call starts from the first call's outputs on both sides
    plan.close()


def test_static_scratch_rejects_oversize_and_bad_args():
    L = _capi.load()
    w = W.custom([[74, 24, 10240]], seed=32)
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
