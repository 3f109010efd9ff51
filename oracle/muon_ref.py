"""Plain NumPy fp64 restatement of the shape-fused Muon update (test oracle).

TEST INFRASTRUCTURE ONLY -- see the package docstring.  Every function works on
one matrix at a time in float64, in the order the method is described; there
is no blocking, fusion or reordering.  Batches are plain Python loops over
independent matrices, because the pages state that the orthogonalisation of a
member depends only on that member's trailing two dims.
"""
from __future__ import annotations

import math
from typing import Dict, List, Sequence, Tuple

import numpy as np

# Quintic coefficients (a, b, c) used by every seeded workload.  The
# pages print no coefficients (the formula block of «关于分布式Muon的想法整合及
# 讨论» §2 was lost in extraction); these are the values the workloads fix and
# every call takes them as arguments anyway.
NS_COEFFS_QUINTIC = (3.4445, -4.7750, 2.0315)

SCALE_MODES = ("sqrt_aspect", "rms_0_2", "none")


def momentum(M: np.ndarray, G: np.ndarray, beta: float) -> np.ndarray:
    """M' = beta * M + G.

    «关于分布式Muon的想法整合及讨论» §1: Muon first keeps a momentum of the
    gradient.  The plainest form (no (1-beta) damping, no Nesterov term) is the
    reading taken.
    """
    return float(beta) * np.asarray(M, np.float64) + np.asarray(G, np.float64)


def nesterov_input(Mp: np.ndarray, G: np.ndarray, beta: float) -> np.ndarray:
    """U = G + beta * M', the Nesterov look-ahead of the momentum M'.

    The pages name no Nesterov variant; this is the reading taken for the
    option, the form that goes with undamped momentum M' = beta M + G: the
    gradient plus beta times the new momentum is orthogonalised instead of
    M' itself (M' is still the stored momentum).
    """
    return np.asarray(G, np.float64) + float(beta) * np.asarray(Mp, np.float64)


def step_coefficients(k: int, a: float, b: float, c: float, schedule=None):
    """The (a_s, b_s, c_s) of steps s = 0 .. k-1.

    With no schedule every step takes (a, b, c).  A schedule is a list of
    rows (a_s, b_s, c_s); past its last row the last row repeats (reading:
    the pages list 5-10 steps and give no per-step values).
    """
    if schedule is None:
        return [(float(a), float(b), float(c))] * int(k)
    rows = [tuple(float(v) for v in r) for r in schedule]
    if not rows or any(len(r) != 3 for r in rows):
        raise ValueError("a schedule is a non-empty list of (a, b, c) rows")
    return [rows[min(s, len(rows) - 1)] for s in range(int(k))]


def frobenius_normalize(M: np.ndarray, eps: float) -> np.ndarray:
    """X0 = M / (||M||_F + eps).

    «关于分布式Muon的想法整合及讨论» §2 (M is normalised before the iteration,
    which is why the whole M is needed) and §6 (the normaliser is a sum of
    squares, so sharded ranks only all-reduce the sum).  eps is added to the
    norm, not to its square (reading; the pages give no eps).
    """
    M = np.asarray(M, np.float64)
    return M / (math.sqrt(float(np.sum(M * M))) + float(eps))


def ns_polynomial(sigma, a: float, b: float, c: float):
    """p(s) = a s + b s^3 + c s^5, the scalar map one quintic step applies to
    each singular value (used by the pins, not by the oracle's update)."""
    s = np.asarray(sigma, np.float64)
    return a * s + b * s ** 3 + c * s ** 5


def newton_schulz(X: np.ndarray, k: int, a: float, b: float, c: float,
                  schedule=None) -> np.ndarray:
    """k quintic Newton-Schulz steps on a wide matrix X (rows <= cols).

    Each step forms the Gram matrix A = X X^T and then X <- aX + (bA + cA A)X
    («关于分布式Muon的想法整合及讨论» §2: the structure is a Gram matrix and a
    series of matrix products; §6: A changes with X every round, so it is
    recomputed each step).  «MindSpore HyperParallel X 盘古,Muon优化器实现6倍性能
    跃升», 三大性能挑战: typically 5-10 iterations.  Step s takes the
    coefficients step_coefficients(k, a, b, c, schedule)[s].
    """
    X = np.array(X, dtype=np.float64, copy=True)
    if X.ndim != 2:
        raise ValueError("newton_schulz acts on one matrix")
    if X.shape[0] > X.shape[1]:
        raise ValueError("newton_schulz expects rows <= cols; use orthogonalize")
    coeffs = step_coefficients(k, a, b, c, schedule)
    for a, b, c in coeffs:
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    return X


def newton_schulz_sharded(X: np.ndarray, k: int, a: float, b: float, c: float, shards: int,
                          schedule=None) -> np.ndarray:
    """The same k steps with X (rows <= cols) held as `shards` contiguous
    column blocks, as on ranks that each own a slice of the columns
    («关于分布式Muon的想法整合及讨论» §6: the Gram matrix is a sum of per-shard
    partial products, so each round needs one all-reduce of it).  Each step
    forms every shard's partial Gram, adds them in shard order (the
    all-reduce), and updates each shard with the same m x m polynomial."""
    X = np.array(X, dtype=np.float64, copy=True)
    if X.shape[0] > X.shape[1]:
        raise ValueError("newton_schulz_sharded expects rows <= cols")
    parts = [p.copy() for p in np.array_split(X, int(shards), axis=1)]
    for a_s, b_s, c_s in step_coefficients(k, a, b, c, schedule):
        A = np.zeros((X.shape[0], X.shape[0]))
        for p in parts:
            A = A + p @ p.T
        B = b_s * A + c_s * (A @ A)
        parts = [a_s * p + B @ p for p in parts]
    return np.concatenate(parts, axis=1)


def sharded_frobenius_normalize(M: np.ndarray, eps: float, shards: int) -> np.ndarray:
    """X0 = M / (||M||_F + eps) with ||M||_F^2 summed from per-shard sums of
    squares in shard order (the sharded normaliser of «关于分布式Muon的想法整合
    及讨论» §6)."""
    M = np.asarray(M, np.float64)
    ss = 0.0
    for p in np.array_split(M, int(shards), axis=1):
        ss += float(np.sum(p * p))
    return M / (math.sqrt(ss) + float(eps))


def orthogonalize(Mp: np.ndarray, k: int, a: float, b: float, c: float,
                  eps: float, schedule=None) -> np.ndarray:
    """O = NS_k(M' / (||M'||_F + eps)), iterating on the wide orientation.

    When rows > cols the normalised matrix is transposed before the iteration
    and the result transposed back (the m x m Gram with m = min(rows, cols) is
    the cheap side; reading of "X transposed when M > N").  Equal dims: no
    transpose.
    """
    X = frobenius_normalize(Mp, eps)
    transposed = X.shape[0] > X.shape[1]
    if transposed:
        X = X.T
    X = newton_schulz(X, k, a, b, c, schedule)
    return X.T if transposed else X


def scale_factor(rows: int, cols: int, mode: str = "sqrt_aspect") -> float:
    """Shape-dependent update scale s(rows, cols).

    The pages only say the update is scaled by shape (reading, parity
    unpinned): 'sqrt_aspect' s = sqrt(max(1, rows/cols)); 'rms_0_2'
    s = 0.2 * sqrt(max(rows, cols)); 'none' s = 1.
    """
    if mode == "sqrt_aspect":
        return math.sqrt(max(1.0, rows / cols))
    if mode == "rms_0_2":
        return 0.2 * math.sqrt(max(rows, cols))
    if mode == "none":
        return 1.0
    raise ValueError(f"unknown scale mode {mode!r}")


def muon_update_ref(P, G, M, beta, lr, wd, k, a, b, c, eps=1e-7,
                    scale_mode="sqrt_aspect", nesterov=False, schedule=None):
    """One Muon update of one matrix, in float64.

    Returns (P', M', O) with
      M' = beta M + G
      U  = G + beta M' with nesterov, else M'
      O  = orthogonalize(U, k, a, b, c, eps, schedule)
      P' = P (1 - lr wd) - lr s(rows, cols) O
    The decoupled, multiplicative weight decay and the scale are readings (the
    pages describe only momentum -> orthogonalised update direction).
    """
    P = np.asarray(P, np.float64)
    if P.ndim != 2:
        raise ValueError("muon_update_ref acts on one matrix")
    Mp = momentum(M, G, beta)
    U = nesterov_input(Mp, G, beta) if nesterov else Mp
    O = orthogonalize(U, k, a, b, c, eps, schedule)
    s = scale_factor(P.shape[0], P.shape[1], scale_mode)
    Pn = P * (1.0 - float(lr) * float(wd)) - float(lr) * s * O
    return Pn, Mp, O


def _members(shape: Sequence[int]) -> Tuple[int, int, int]:
    """(E, rows, cols) of a 2-D or 3-D parameter shape."""
    shape = tuple(int(d) for d in shape)
    if len(shape) == 2:
        return 1, shape[0], shape[1]
    if len(shape) == 3:
        return shape[0], shape[1], shape[2]
    raise ValueError(f"parameter must be 2-D or 3-D, got {shape}")


def bucket_shapes(shapes: Sequence[Sequence[int]], merge_transposed: bool = False) -> List[Dict]:
    """Group parameters by their exact trailing two dims, first-seen order.

    «MindSpore HyperParallel X 盘古,Muon优化器实现6倍性能跃升», 矩阵融合优化
    (Fig. 6): parameters whose trailing two dims agree are stacked into one
    [B, M, N] batch; Muon亲和的专家切分 (Fig. 4): a 3-D [E, M, N] tensor is E
    independent matrices.  Members keep parameter order, experts in E order.
    With merge_transposed the key is (min, max) of the two dims, so [r, c]
    and [c, r] share a group (a larger fused batch; each member keeps its
    orientation); the group's (rows, cols) are its first member's.
    Returns [{'rows', 'cols', 'members': [(param, expert), ...]}, ...].
    """
    groups: Dict[Tuple[int, int], Dict] = {}
    order: List[Tuple[int, int]] = []
    for pi, shp in enumerate(shapes):
        E, r, cl = _members(shp)
        if E < 1 or r < 1 or cl < 1:
            raise ValueError(f"parameter {pi} has an empty dim: {tuple(shp)}")
        key = (min(r, cl), max(r, cl)) if merge_transposed else (r, cl)
        if key not in groups:
            groups[key] = {"rows": r, "cols": cl, "members": []}
            order.append(key)
        groups[key]["members"].extend((pi, e) for e in range(E))
    return [groups[k] for k in order]


def muon_step_ref(params, grads, momenta, beta, lr, wd, k, a, b, c,
                  eps=1e-7, scale_mode="sqrt_aspect", nesterov=False, schedule=None):
    """Muon update of a list of 2-D / 3-D parameters, matrix by matrix.

    Bucketing changes nothing mathematically (each member is independent), so
    this loops over parameters and experts.  Returns lists (P', M', O) with the
    parameters' own shapes.
    """
    outP, outM, outO = [], [], []
    for P, G, M in zip(params, grads, momenta):
        P = np.asarray(P, np.float64)
        if P.ndim == 2:
            r = muon_update_ref(P, G, M, beta, lr, wd, k, a, b, c, eps, scale_mode, nesterov, schedule)
            outP.append(r[0]); outM.append(r[1]); outO.append(r[2])
        elif P.ndim == 3:
            rs = [muon_update_ref(P[e], np.asarray(G)[e], np.asarray(M)[e], beta, lr,
                                  wd, k, a, b, c, eps, scale_mode, nesterov, schedule)
                  for e in range(P.shape[0])]
            outP.append(np.stack([r[0] for r in rs]))
            outM.append(np.stack([r[1] for r in rs]))
            outO.append(np.stack([r[2] for r in rs]))
        else:
            raise ValueError("parameters must be 2-D or 3-D")
    return outP, outM, outO
