"""Seeded synthetic workloads (shapes, value laws, step scalars).

This module holds no part of the Muon arithmetic: it only draws tensors.  Both
the tests (which hand the same tensors to the CUDA library and to the CPU
oracle) and ``bench.py`` take their inputs from here.

Shapes come from the pages' own examples -- [24, 10240] x 74 and
[32, 24, 10240] («MindSpore HyperParallel X 盘古,Muon优化器实现6倍性能跃升»,
矩阵融合优化, Fig. 6-7) -- and from the benchmark configurations of this
library (an MoE expert tensor, a dense h=4096 transformer, a mixed bag of
1000 matrices).  The pages measure no public dataset; gradients and momenta
are Gaussian with the stated standard deviations.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import torch

QUINTIC = (3.4445, -4.7750, 2.0315)


@dataclass
class Workload:
    name: str
    shapes: List[List[int]]
    mode: str                      # "bf16" (bf16 P/G, fp32 M) or "fp32"
    beta: float
    lr: float
    wd: float
    ns_steps: int
    coeffs: tuple = QUINTIC        # (a, b, c), or a per-step schedule [(a_0, b_0, c_0), ...]
    nesterov: bool = False         # orthogonalise U = G + beta M' instead of M'
    p_std: List[float] = field(default_factory=list)     # per parameter
    g_std: List[object] = field(default_factory=list)    # per parameter: float or per-expert list
    m_zero: bool = False
    seed: int = 0
    describe: str = ""
    spectrum_decades: float = 0.0  # > 0: M and G share singular values log-spaced over this many decades

    @property
    def n_params(self) -> int:
        return len(self.shapes)

    def n_elements(self) -> int:
        return sum(math.prod(s) for s in self.shapes)


C5_SHAPES = [[24, 10240], [64, 7168], [128, 4096], [512, 2048], [1024, 1024],
             [1536, 7168], [2048, 7168], [7168, 2048], [4096, 4096], [4096, 11008],
             [11008, 4096], [7168, 7168]]


def c5_counts(seed: int = 5) -> List[int]:
    """1 + multinomial(988, w ~ 1/(rows*cols)) over the 12 mixed-bag shapes."""
    g = torch.Generator().manual_seed(seed)
    w = torch.tensor([1.0 / (r * c) for r, c in C5_SHAPES], dtype=torch.float64)
    draws = torch.multinomial(w / w.sum(), 988, replacement=True, generator=g)
    counts = torch.bincount(draws, minlength=len(C5_SHAPES)) + 1
    return [int(x) for x in counts]


def _log_uniform(g: torch.Generator, lo: float, hi: float, n: int) -> List[float]:
    u = torch.rand(n, generator=g, dtype=torch.float64)
    return [float(math.exp(math.log(lo) + float(x) * (math.log(hi) - math.log(lo)))) for x in u]


def get(name: str, ns_steps: Optional[int] = None) -> Workload:
    """The named workload.  Names: 'c1_fp32_64x128', 'c2_skinny_74x24x10240',
    'c3_moe_64x2048x7168_32x24x10240', 'c4_dense_h4096', 'c5_mixed_1000',
    'c5_group_<rows>x<cols>' (one shape group of the mixed bag),
    'group_<rows>x<cols>_b<B>' (B matrices of one shape, for profiling one
    group at a reduced batch), plus small parity cases built by ``custom``."""
    beta, lr = 0.95, 0.02
    if name == "c1_fp32_64x128":
        w = Workload(name, [[64, 128]], "fp32", beta, lr, 0.0, 5,
                     p_std=[1.0], g_std=[1.0], seed=1,
                     describe="one 64x128 fp32 matrix, P,G,M ~ N(0,1)")
    elif name == "c2_skinny_74x24x10240":
        w = Workload(name, [[24, 10240]] * 74, "bf16", beta, lr, 0.1, 5,
                     p_std=[0.02] * 74, g_std=[1e-3] * 74, seed=2,
                     describe="74 params [24,10240] bf16, fp32 momentum, G,M ~ N(0,1e-3^2), P ~ N(0,0.02^2)")
    elif name == "c3_moe_64x2048x7168_32x24x10240":
        g = torch.Generator().manual_seed(3)
        w = Workload(name, [[64, 2048, 7168], [32, 24, 10240]], "bf16", beta, lr, 0.1, 5,
                     p_std=[0.02, 0.02], g_std=[_log_uniform(g, 1e-4, 1e-2, 64), 1e-3], seed=3,
                     describe="expert tensor [64,2048,7168] (per-expert std log-uniform [1e-4,1e-2]) + [32,24,10240]")
    elif name == "c4_dense_h4096":
        layer = [[4096, 12288], [4096, 4096], [4096, 16384], [16384, 4096]]
        shapes = [s for _ in range(32) for s in layer]
        w = Workload(name, shapes, "bf16", beta, lr, 0.1, 5,
                     p_std=[0.02] * len(shapes), g_std=[1e-3] * len(shapes), seed=4,
                     describe="h=4096, 32 layers x {[4096,12288],[4096,4096],[4096,16384],[16384,4096]}")
    elif name == "c5_mixed_1000":
        counts = c5_counts(5)
        shapes = [s for s, n in zip(C5_SHAPES, counts) for _ in range(n)]
        g = torch.Generator().manual_seed(55)
        w = Workload(name, shapes, "bf16", beta, lr, 0.1, 5,
                     p_std=[0.02] * len(shapes), g_std=_log_uniform(g, 1e-5, 1e-2, len(shapes)),
                     seed=5, describe="1000 matrices over 12 shapes, per-matrix std log-uniform [1e-5,1e-2]")
    elif name.startswith("c5_group_"):
        # one shape group of the mixed bag alone (its count and value law),
        # for per-group profiling: e.g. 'c5_group_64x7168'
        shape = [int(x) for x in name[len("c5_group_"):].split("x")]
        if shape not in C5_SHAPES:
            raise KeyError(name)
        full = get("c5_mixed_1000")
        idx = [i for i, s in enumerate(full.shapes) if s == shape]
        w = Workload(name, [shape] * len(idx), "bf16", beta, lr, 0.1, 5,
                     p_std=[full.p_std[i] for i in idx], g_std=[full.g_std[i] for i in idx], seed=5,
                     describe=f"the {shape} group of the mixed bag ({len(idx)} matrices)")
    elif name.startswith("group_"):
        # B matrices of one shape with the dense model's value law, for
        # profiling one group at a reduced batch: e.g. 'group_16384x4096_b2'
        try:
            dims, b = name[len("group_"):].split("_b")
            rows, cols = (int(x) for x in dims.split("x"))
            B = int(b)
        except ValueError:
            raise KeyError(name)
        if min(rows, cols) < 1 or B < 1:
            raise KeyError(name)
        w = Workload(name, [[rows, cols]] * B, "bf16", beta, lr, 0.1, 5,
                     p_std=[0.02] * B, g_std=[1e-3] * B, seed=6,
                     describe=f"{B} matrices [{rows},{cols}], G,M ~ N(0,1e-3^2), P ~ N(0,0.02^2)")
    else:
        raise KeyError(name)
    if ns_steps is not None:
        w.ns_steps = int(ns_steps)
    return w


def custom(shapes: Sequence[Sequence[int]], mode: str = "bf16", seed: int = 0,
           g_std: float = 1e-3, p_std: float = 0.02, beta: float = 0.95, lr: float = 0.02,
           wd: float = 0.1, ns_steps: int = 5, m_zero: bool = False,
           spectrum_decades: float = 0.0) -> Workload:
    shapes = [list(map(int, s)) for s in shapes]
    return Workload("custom", shapes, mode, beta, lr, wd, ns_steps,
                    p_std=[p_std] * len(shapes), g_std=[g_std] * len(shapes),
                    m_zero=m_zero, seed=seed, describe=f"custom {shapes}",
                    spectrum_decades=float(spectrum_decades))


def spread_matrix(rows: int, cols: int, decades: float, std: float,
                  g: torch.Generator) -> torch.Tensor:
    """A seeded fp64 [rows, cols] matrix U diag(s) V^T with random orthonormal
    U, V (QR of Gaussian draws) and s log-spaced from 1 down to 10^-decades,
    scaled so that its entries have root-mean-square `std`."""
    r = min(rows, cols)
    U = torch.linalg.qr(torch.randn(rows, r, generator=g, dtype=torch.float64))[0]
    V = torch.linalg.qr(torch.randn(cols, r, generator=g, dtype=torch.float64))[0]
    s = torch.logspace(0, -float(decades), r, dtype=torch.float64)
    X = (U * s) @ V.T
    return X * (std * math.sqrt(rows * cols) / float(torch.linalg.norm(X)))


def make_tensors(w: Workload, device="cpu"):
    """Draw (params, grads, momenta) for a workload.

    bf16 mode: P, G bf16 (fp32 draw, round-to-nearest-even cast), M fp32.
    fp32 mode: all fp32.  M0 follows the same law as G (so beta matters)
    unless ``m_zero``.  Per-expert stds scale each expert slice.  With
    ``spectrum_decades`` > 0, G and M0 are one spread_matrix per member (the
    same draw), so their singular values fall log-evenly over that many
    decades, unlike the concentrated spectra of Gaussian draws.
    """
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(w.seed)
    pdt = torch.bfloat16 if w.mode == "bf16" else torch.float32
    params, grads, moms = [], [], []
    if w.spectrum_decades > 0:
        # M0 and G share their singular vectors, so M' = beta M0 + G keeps
        # the log-spaced spectrum (up to the rounding of G); drawn on the host
        hg = torch.Generator().manual_seed(w.seed)
        for i, shp in enumerate(w.shapes):
            E = shp[0] if len(shp) == 3 else 1
            X = torch.stack([spread_matrix(shp[-2], shp[-1], w.spectrum_decades,
                                           float(w.g_std[i]), hg) for _ in range(E)])
            X = X.reshape(shp).float()
            P = (torch.randn(shp, generator=hg, dtype=torch.float32) * w.p_std[i]).to(pdt)
            params.append(P.to(dev).contiguous())
            grads.append(X.to(pdt).to(dev).contiguous())
            moms.append((torch.zeros_like(X) if w.m_zero else X).to(dev).contiguous())
        return params, grads, moms
    for i, shp in enumerate(w.shapes):
        gs = w.g_std[i]
        if isinstance(gs, (list, tuple)):
            std = torch.tensor(gs, dtype=torch.float32, device=dev).view(-1, *([1] * (len(shp) - 1)))
        else:
            std = float(gs)
        P = (torch.randn(shp, generator=g, device=dev, dtype=torch.float32) * w.p_std[i]).to(pdt)
        G = (torch.randn(shp, generator=g, device=dev, dtype=torch.float32) * std).to(pdt)
        if w.m_zero:
            M = torch.zeros(shp, device=dev, dtype=torch.float32)
        else:
            M = torch.randn(shp, generator=g, device=dev, dtype=torch.float32) * std
        params.append(P.contiguous()); grads.append(G.contiguous()); moms.append(M.contiguous())
    return params, grads, moms


ALL = ["c1_fp32_64x128", "c2_skinny_74x24x10240", "c3_moe_64x2048x7168_32x24x10240",
       "c4_dense_h4096", "c5_mixed_1000"]
