"""The binding's marshalling checks, on the host: a tensor list that does not
match the plan (count, shape, dtype, layout, device) is refused with a
ValueError before any pointer reaches the C ABI.  The plan object here is
never created in the library, so a check that let a bad list through would
fail on the null library handle instead of raising ValueError."""
import ctypes as C

import pytest
import torch

import newton_schulz_bucket_gb300 as pkg


def _fake_plan(shapes, mode="bf16"):
    plan = object.__new__(pkg.MuonPlan)
    plan.shapes = [list(s) for s in shapes]
    plan.mode = mode
    plan.device = 0
    plan.keep_update = False
    plan._L = None
    plan._h = C.c_void_p()
    return plan


def _host(shapes, pd=torch.bfloat16):
    P = [torch.zeros(s, dtype=pd) for s in shapes]
    G = [torch.zeros(s, dtype=pd) for s in shapes]
    M = [torch.zeros(s, dtype=torch.float32) for s in shapes]
    return P, G, M


SHAPES = [[4, 8], [2, 3, 8]]


@pytest.mark.parametrize("bad,match", [
    (lambda P, G, M: (P[:1], G, M), "expected 2 tensors"),
    (lambda P, G, M: ([P[0], torch.zeros(2, 8, 3, dtype=torch.bfloat16)], G, M), "shape"),
    (lambda P, G, M: (P, [G[0].float(), G[1]], M), "dtype"),
    (lambda P, G, M: (P, G, [M[0], M[1].half()]), "dtype"),
    (lambda P, G, M: ([torch.zeros(8, 4, dtype=torch.bfloat16).t(), P[1]], G, M), "contiguous"),
])
def test_host_step_refuses_mismatched_tensors(bad, match):
    plan = _fake_plan(SHAPES)
    P, G, M = bad(*_host(SHAPES))
    with pytest.raises(ValueError, match=match):
        plan.step_host(P, G, M, 0.9, 0.02, 0.0)


def test_device_step_refuses_host_tensors():
    plan = _fake_plan(SHAPES)
    with pytest.raises(ValueError, match="cuda:0"):
        plan.step(*_host(SHAPES), 0.9, 0.02, 0.0)
    with pytest.raises(ValueError, match="cuda:0"):
        plan.bind(*_host(SHAPES))


def test_fp32_mode_wants_fp32_params():
    plan = _fake_plan(SHAPES, mode="fp32")
    with pytest.raises(ValueError, match="dtype"):
        plan.step_host(*_host(SHAPES), 0.9, 0.02, 0.0)


def test_host_step_refuses_a_schedule():
    plan = _fake_plan(SHAPES)
    with pytest.raises(ValueError, match="schedule"):
        plan.step_host(*_host(SHAPES), 0.9, 0.02, 0.0, 5,
                       coeffs=[(3.4445, -4.775, 2.0315), (1.875, -1.25, 0.375)])
    with pytest.raises(ValueError, match="schedule"):
        plan.step_host(*_host(SHAPES), 0.9, 0.02, 0.0, 5,
                       coeffs=[(3.4445, -4.775, 2.0315)] * 3)
