"""Helpers for GPU-vs-oracle parity: run one step through the C ABI on seeded
inputs, run the CPU oracle on byte-identical copies, compare per member.

Tolerances (relative Frobenius error of O per member, from the workload
contract): 1e-4 in fp32 mode, 2e-2 in bf16 mode.  M' is an fp32 FMA of the
same inputs (<= 1e-6 relative per element).  P' in bf16 mode may differ by one
bf16 ulp of rounding plus lr*s*|dO| plus fp32 rounding of its two terms; in
fp32 mode dP = P' - P agrees to 1e-4.
"""
from __future__ import annotations

from typing import List

import numpy as np
import torch

import newton_schulz_bucket_gb300 as pkg
from newton_schulz_bucket_gb300 import workloads as W
from oracle import muon_ref

F32 = lambda v: float(np.float32(v))
TOL_O = {"bf16": 2e-2, "fp32": 1e-4}


def host64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def members_of(shapes):
    out = []
    for i, s in enumerate(shapes):
        E = s[0] if len(s) == 3 else 1
        for e in range(E):
            out.append((i, e))
    return out


def sl(t, dim3, e):
    return t[e] if dim3 else t


class GpuRun:
    """One (or more) steps of workload `w` on cuda:0.  Host fp64 copies of the
    inputs and outputs are kept for the sampled members only (all by default),
    so full-size workloads do not need their whole state on the host."""

    def __init__(self, w: W.Workload, steps: int = 1, tensors=None, sample=None, **plan_opts):
        self.w = w
        P, G, M = tensors if tensors is not None else W.make_tensors(w, "cuda")
        self.members = list(sample) if sample is not None else members_of(w.shapes)
        d3 = lambda i: len(w.shapes[i]) == 3
        self.inp = {(i, e): (host64(sl(P[i], d3(i), e)), host64(sl(G[i], d3(i), e)),
                             host64(sl(M[i], d3(i), e))) for (i, e) in self.members}
        plan_opts.setdefault("keep_update", True)
        plan_opts.setdefault("nesterov", w.nesterov)
        self.plan = pkg.MuonPlan(w.shapes, mode=w.mode, **plan_opts)
        self.nesterov = plan_opts["nesterov"]
        if isinstance(w.coeffs[0], (tuple, list)):  # per-step schedule
            self.coeffs = [tuple(F32(v) for v in r) for r in w.coeffs]
        else:
            self.coeffs = tuple(F32(v) for v in w.coeffs)
        for _ in range(steps):
            self.plan.step(P, G, M, w.beta, w.lr, w.wd, w.ns_steps, self.coeffs)
        torch.cuda.synchronize()
        self.out = {(i, e): (host64(sl(P[i], d3(i), e)), host64(sl(M[i], d3(i), e)))
                    for (i, e) in self.members}
        self.Pt, self.Gt, self.Mt = P, G, M

    def p0(self, i, e=0): return self.inp[(i, e)][0]
    def g0(self, i, e=0): return self.inp[(i, e)][1]
    def m0(self, i, e=0): return self.inp[(i, e)][2]
    def p1(self, i, e=0): return self.out[(i, e)][0]
    def m1(self, i, e=0): return self.out[(i, e)][1]

    def O(self, i, e=0) -> np.ndarray:
        return self.plan.debug_update(i, e).astype(np.float64)

    def close(self):
        self.plan.close()


def oracle_member(run: GpuRun, i: int, e: int, scale_mode="sqrt_aspect", eps=1e-7):
    w = run.w
    schedule = run.coeffs if isinstance(run.coeffs, list) else None
    a, b, c = schedule[0] if schedule else run.coeffs
    return muon_ref.muon_update_ref(run.p0(i, e), run.g0(i, e), run.m0(i, e), F32(w.beta),
                                    F32(w.lr), F32(w.wd), w.ns_steps, a, b, c, eps, scale_mode,
                                    run.nesterov, schedule)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(ax)) - 7)


def check_member(run: GpuRun, i: int, e: int, scale_mode="sqrt_aspect", tol_o=None,
                 eps=1e-7) -> float:
    """Asserts parity of one member; returns the relative Frobenius error of O."""
    w = run.w
    shp = w.shapes[i]
    rP, rM, rO = oracle_member(run, i, e, scale_mode, eps)
    gO = run.O(i, e)
    gP = run.p1(i, e)
    gM = run.m1(i, e)
    tol = TOL_O[w.mode] if tol_o is None else tol_o
    nO = np.linalg.norm(rO)
    err = np.linalg.norm(gO - rO) / nO if nO > 0 else np.linalg.norm(gO)
    assert err <= tol, f"member ({i},{e}) {shp}: O rel err {err:.3e} > {tol}"
    dm = np.abs(gM - rM)
    assert np.all(dm <= 1e-6 * np.abs(rM) + 1e-38), f"member ({i},{e}): momentum mismatch {dm.max():.3e}"
    s = muon_ref.scale_factor(shp[-2], shp[-1], scale_mode)
    P0 = run.p0(i, e)
    if w.mode == "bf16":
        # one bf16 ulp of the stored result, the O difference scaled by lr*s,
        # and fp32 rounding of the two terms P (1 - lr wd) and lr s O
        lrs = F32(w.lr) * s
        bound = (bf16_ulp(np.maximum(np.abs(rP), np.abs(gP))) + lrs * np.abs(gO - rO)
                 + 2.0 ** -22 * (np.abs(P0) + lrs * np.abs(rO)) + 1e-30)
        bad = np.abs(gP - rP) > bound
        if bad.any():
            k = int(np.argmax(np.abs(gP - rP) - bound))
            raise AssertionError(
                f"member ({i},{e}): {int(bad.sum())} P' elements out of bound; worst flat index {k}: "
                f"gpu {gP.flat[k]!r} ref {rP.flat[k]!r} P0 {P0.flat[k]!r} O {gO.flat[k]!r}/{rO.flat[k]!r} "
                f"bound {bound.flat[k]!r}")
    else:
        d_ref, d_gpu = rP - P0, gP - P0
        nd = np.linalg.norm(d_ref)
        if nd > 0:
            rel = np.linalg.norm(d_gpu - d_ref) / nd
            assert rel <= 1e-4, f"member ({i},{e}): dP rel err {rel:.3e}"
    return float(err)


def check_all(run: GpuRun, members=None, **kw) -> List[float]:
    ms = members if members is not None else run.members
    return [check_member(run, i, e, **kw) for (i, e) in ms]
