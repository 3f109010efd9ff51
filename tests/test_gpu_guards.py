"""Bounds and resume checks on the GPU.

* Guard bands: every caller buffer (P, G, M) is a view into a larger
  allocation whose bytes before and after carry a known pattern; after the
  steps the pattern must be intact (no kernel writes outside a member), and
  G must be bit-identical (it is read only).  Odd shapes, ragged tails and
  both orientations exercise the scalar and vector access paths.
* Resume: two steps in one plan equal one step, a copy of P and M through
  host memory, a new plan and a second step, bit for bit (the plan keeps no
  state across steps besides its cached graphs).
"""
import math

import numpy as np
import pytest
import torch

import newton_schulz_bucket_gb300 as pkg
from newton_schulz_bucket_gb300 import workloads as W

pytestmark = pytest.mark.gpu

PAD = 4096  # elements of guard band on each side


def _guarded(t):
    """A copy of t living inside a larger buffer with patterned guard bands;
    returns (view, backing, pattern value)."""
    n = t.numel()
    back = torch.empty(n + 2 * PAD, dtype=t.dtype, device=t.device)
    fill = -12345.0 if t.dtype == torch.float32 else -123.0
    back.fill_(fill)
    view = back[PAD:PAD + n].view(t.shape)
    view.copy_(t)
    return view, back, fill


def _bands_intact(back, n, fill):
    lo, hi = back[:PAD], back[PAD + n:]
    return bool(torch.all(lo == fill)) and bool(torch.all(hi == fill))


CASES = [
    ([[24, 10240], [3, 24, 1000], [10240, 24], [17, 333], [24, 1004]], {}, 5),      # skinny, Gram space
    ([[64, 1000], [1000, 64], [2, 40, 96]], {}, 5),                                  # skinny, m > 32
    ([[1000, 24], [3000, 40], [2, 520, 16]], {}, 5),                                # transposed skinny, ragged blocks
    ([[24, 2048], [2048, 24]], {}, 70),                                              # skinny, direct
    ([[256, 520], [520, 256], [2, 130, 384]], {}, 5),                                # tensor cores
    ([[96, 200], [2, 70, 33]], {"path": "simt"}, 5),                                 # SIMT
    ([[24, 4096], [4096, 24], [64, 256]], {"merge_transposed": True, "column_shards": 8}, 5),
    ([[100, 700], [700, 100], [2, 128, 520], [96, 2049], [2049, 96]], {"path": "resident"}, 5),
]


@pytest.mark.parametrize("shapes,opts,k", CASES,
                         ids=["gram_space", "gram_space_m64", "transposed_ragged", "direct", "tensor", "simt", "merged_shards",
                              "resident"])
def test_guard_bands_intact(shapes, opts, k):
    w = W.custom(shapes, seed=51, ns_steps=k)
    P, G, M = W.make_tensors(w, "cuda")
    gp = [_guarded(t) for t in P]
    gg = [_guarded(t) for t in G]
    gm = [_guarded(t) for t in M]
    g_before = [t.clone() for t in G]
    plan = pkg.MuonPlan(w.shapes, keep_update=True, **opts)
    for _ in range(2):
        plan.step([v for v, _, _ in gp], [v for v, _, _ in gg], [v for v, _, _ in gm],
                  w.beta, w.lr, w.wd, k)
    torch.cuda.synchronize()
    plan.check_error()
    for i, s in enumerate(w.shapes):
        n = math.prod(s)
        for v, back, fill in (gp[i], gg[i], gm[i]):
            assert _bands_intact(back, n, fill), f"parameter {i} {s}: guard band overwritten"
        assert torch.equal(gg[i][0], g_before[i]), f"parameter {i}: gradient modified"
        assert torch.isfinite(gp[i][0].float()).all() and torch.isfinite(gm[i][0]).all()
    plan.close()


@pytest.mark.parametrize("shapes", [[[24, 4096]] * 3 + [[2, 64, 1000]], [[256, 512], [24, 2048]]])
def test_resume_through_host_equals_continuous(shapes):
    w = W.custom(shapes, seed=52)
    P, G, M = W.make_tensors(w, "cuda")
    P2, G2, M2 = [t.clone() for t in P], [t.clone() for t in G], [t.clone() for t in M]
    a = pkg.MuonPlan(w.shapes)
    a.step(P, G, M, w.beta, w.lr, w.wd, 5)
    a.step(P, G, M, w.beta, w.lr, w.wd, 5)
    torch.cuda.synchronize()
    a.close()
    b = pkg.MuonPlan(w.shapes)
    b.step(P2, G2, M2, w.beta, w.lr, w.wd, 5)
    torch.cuda.synchronize()
    b.close()
    # "checkpoint": P, M through host memory; a fresh plan resumes
    hP = [t.cpu() for t in P2]
    hM = [t.cpu() for t in M2]
    P3 = [t.cuda() for t in hP]
    M3 = [t.cuda() for t in hM]
    c = pkg.MuonPlan(w.shapes)
    c.step(P3, G2, M3, w.beta, w.lr, w.wd, 5)
    torch.cuda.synchronize()
    c.close()
    for x, y in zip(P + M, P3 + M3):
        assert torch.equal(x, y)


@pytest.mark.parametrize("shapes,opts", [([[24, 4096]] * 6, {}), ([[64, 1000]] * 4, {}), ([[256, 512]] * 3, {}),
                                         ([[2, 130, 384]], {}), ([[128, 1024]] * 3, {"path": "resident"})],
                         ids=["gram_space", "gram_space_m64", "tensor", "tensor_experts", "resident"])
def test_nonfinite_member_stays_isolated(shapes, opts):
    """A NaN in one member's gradient propagates into that member only (no
    special casing, as stated); every other member gives the same bits as in
    a run without it."""
    w = W.custom(shapes, seed=53)
    P, G, M = W.make_tensors(w, "cuda")
    clean = [[t.clone() for t in ts] for ts in (P, G, M)]
    bad_param, bad_expert = (1, 0) if len(shapes) > 1 else (0, 1)
    target = G[bad_param][bad_expert] if len(shapes[bad_param]) == 3 else G[bad_param]
    target[3, 5] = float("nan")
    for tensors in ((P, G, M), clean):
        plan = pkg.MuonPlan(w.shapes, **opts)
        plan.step(*tensors, w.beta, w.lr, w.wd, 5)
        torch.cuda.synchronize()
        plan.close()
    for i, s in enumerate(w.shapes):
        E = s[0] if len(s) == 3 else 1
        for e in range(E):
            sl = (lambda t: t[e]) if len(s) == 3 else (lambda t: t)
            if (i, e) == (bad_param, bad_expert):
                assert torch.isnan(sl(M[i])).any() and torch.isnan(sl(P[i]).float()).any()
            else:
                assert torch.equal(sl(P[i]), sl(clean[0][i])), (i, e)
                assert torch.equal(sl(M[i]), sl(clean[2][i])), (i, e)
