"""Shape-fused Muon update on one GB300 (sm_103a): Python binding of the C ABI.

Every step of the update runs in the library's CUDA kernels; this module only
marshals shapes, pointers and scalars (PyTorch supplies device memory and
streams).  See include/muon.h for the contract of each call.
"""
from __future__ import annotations

import ctypes as C
from typing import Dict, List, Sequence

from . import _capi as _c
from ._capi import MuonError  # noqa: F401

__all__ = ["MuonPlan", "describe", "assign_owners", "load_library", "MuonError", "QUINTIC"]

QUINTIC = (3.4445, -4.7750, 2.0315)

_MODES = {"bf16": _c.MUON_MODE_BF16, "fp32": _c.MUON_MODE_FP32}
_NS = {"fp16": _c.MUON_NS_FP16, "bf16": _c.MUON_NS_BF16}
_SCALES = {"sqrt_aspect": _c.MUON_SCALE_SQRT_ASPECT, "rms_0_2": _c.MUON_SCALE_RMS_0_2,
           "none": _c.MUON_SCALE_NONE}
_PATHS = {"auto": _c.MUON_PATH_AUTO, "skinny": _c.MUON_PATH_SKINNY,
          "tensor": _c.MUON_PATH_TENSOR, "simt": _c.MUON_PATH_SIMT,
          "resident": _c.MUON_PATH_RESIDENT}
PATH_NAMES = {v: k for k, v in _PATHS.items()}


def load_library():
    return _c.load()


def _shapes(shapes: Sequence[Sequence[int]]):
    arr = (_c.muon_shape_t * max(len(shapes), 1))()
    for i, s in enumerate(shapes):
        s = [int(d) for d in s]
        arr[i].ndim = len(s)
        for j, d in enumerate(s[:3]):
            arr[i].dims[j] = d
    return arr


def _options(mode="bf16", scale="sqrt_aspect", eps=1e-7, ns_dtype="fp16", skinny_threshold=0,
             path="auto", keep_update=False, no_graph=False, host_staging=False, max_streams=0,
             group_timing=False, nesterov=False, merge_transposed=False, column_shards=0):
    L = _c.load()
    o = _c.muon_plan_options()
    _c.check(L.muon_default_options(C.byref(o)), "muon_default_options")
    o.mode = _MODES[mode]
    o.scale = _SCALES[scale]
    o.eps = float(eps)
    o.ns_dtype = _NS[ns_dtype]
    o.skinny_threshold = int(skinny_threshold)
    o.path_override = _PATHS[path]
    o.flags = ((_c.MUON_FLAG_KEEP_UPDATE if keep_update else 0)
               | (_c.MUON_FLAG_NO_GRAPH if no_graph else 0)
               | (_c.MUON_FLAG_HOST_STAGING if host_staging else 0)
               | (_c.MUON_FLAG_GROUP_TIMING if group_timing else 0)
               | (_c.MUON_FLAG_NESTEROV if nesterov else 0)
               | (_c.MUON_FLAG_MERGE_TRANSPOSED if merge_transposed else 0))
    o.max_streams = int(max_streams)
    o.column_shards = int(column_shards)
    return o


def _group_dict(g) -> Dict:
    return {"rows": g.rows, "cols": g.cols, "batch": g.batch, "first_member": g.first_member,
            "transposed": {0: False, 1: True}.get(g.transposed, "mixed"),
            "path": PATH_NAMES.get(g.path, g.path),
            "workspace_bytes": g.workspace_bytes}


def describe(shapes: Sequence[Sequence[int]], **opts) -> Dict:
    """Host-only planning (no device): groups, members and workspace size."""
    L = _c.load()
    sh = _shapes(shapes)
    o = _options(**opts)
    ng, nm, ws = C.c_int32(), C.c_int64(), C.c_size_t()
    _c.check(L.muon_plan_describe(sh, len(shapes), C.byref(o), None, 0, C.byref(ng), None, None,
                                  0, C.byref(nm), C.byref(ws)), "muon_plan_describe")
    groups = (_c.muon_group_info_t * max(ng.value, 1))()
    mp = (C.c_int32 * max(nm.value, 1))()
    me = (C.c_int32 * max(nm.value, 1))()
    _c.check(L.muon_plan_describe(sh, len(shapes), C.byref(o), groups, ng.value, C.byref(ng), mp,
                                  me, nm.value, C.byref(nm), C.byref(ws)), "muon_plan_describe")
    return {"groups": [_group_dict(groups[i]) for i in range(ng.value)],
            "members": [(mp[i], me[i]) for i in range(nm.value)],
            "workspace_bytes": ws.value}


def assign_owners(shapes: Sequence[Sequence[int]], n_ranks: int, ns_steps: int = 5, **opts) -> Dict:
    """Host-only greedy, cost-balanced ownership of every member matrix over
    n_ranks data-parallel replicas (muon_plan_assign).  Returns the members
    (parameter, expert) in plan order, each member's owner rank and estimated
    cost (seconds), and each rank's summed cost."""
    L = _c.load()
    d = describe(shapes, **opts)
    nm = len(d["members"])
    sh = _shapes(shapes)
    o = _options(**opts)
    owner = (C.c_int32 * max(nm, 1))()
    mcost = (C.c_double * max(nm, 1))()
    rcost = (C.c_double * max(int(n_ranks), 1))()
    _c.check(L.muon_plan_assign(sh, len(shapes), C.byref(o), int(ns_steps), int(n_ranks), owner, nm,
                                mcost, rcost), "muon_plan_assign")
    return {"members": d["members"], "owner": [owner[i] for i in range(nm)],
            "member_cost": [mcost[i] for i in range(nm)],
            "rank_cost": [rcost[r] for r in range(int(n_ranks))]}


class MuonPlan:
    """A plan for one fixed list of parameter shapes (2-D or 3-D [E, rows, cols])."""

    def __init__(self, shapes: Sequence[Sequence[int]], device: int = 0, **opts):
        L = _c.load()
        self._L = L
        self._h = C.c_void_p()
        self.shapes = [list(map(int, s)) for s in shapes]
        self.mode = opts.get("mode", "bf16")
        self.keep_update = bool(opts.get("keep_update", False))
        o = _options(**opts)
        h = C.c_void_p()
        _c.check(L.muon_plan_create(_shapes(self.shapes), len(self.shapes), C.byref(o),
                                    int(device), C.byref(h)), "muon_plan_create")
        self._h = h
        self.device = int(device)

    # -- introspection --
    def groups(self) -> List[Dict]:
        out = []
        for g in range(self._L.muon_plan_num_groups(self._h)):
            info = _c.muon_group_info_t()
            _c.check(self._L.muon_plan_group_info(self._h, g, C.byref(info)), "group_info")
            out.append(_group_dict(info))
        return out

    def workspace_bytes(self) -> int:
        return int(self._L.muon_plan_workspace_bytes(self._h))

    # -- steps --
    def _ptrs(self, tensors, what, dtype, device_kind):
        if len(tensors) != len(self.shapes):
            raise ValueError(f"{what}: expected {len(self.shapes)} tensors, got {len(tensors)}")
        arr = (C.c_void_p * len(tensors))()
        for i, (t, s) in enumerate(zip(tensors, self.shapes)):
            if list(t.shape) != s:
                raise ValueError(f"{what}[{i}] has shape {list(t.shape)}, plan expects {s}")
            if t.dtype != dtype:
                raise ValueError(f"{what}[{i}] has dtype {t.dtype}, expected {dtype}")
            if not t.is_contiguous():
                raise ValueError(f"{what}[{i}] must be contiguous")
            if device_kind == "cuda" and (not t.is_cuda or t.device.index != self.device):
                raise ValueError(f"{what}[{i}] must live on cuda:{self.device}")
            if device_kind == "cpu" and t.is_cuda:
                raise ValueError(f"{what}[{i}] must be a host tensor")
            arr[i] = t.data_ptr()
        return arr

    def _pdtype(self):
        import torch
        return torch.float32 if self.mode == "fp32" else torch.bfloat16

    def _stream(self, stream):
        import torch
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)

    def _launch(self, P, G, M, beta, lr, wd, ns_steps, coeffs, stream):
        """muon_step for one (a, b, c) triple; muon_step_schedule for a list of
        per-step rows [(a_0, b_0, c_0), ...] (the last row repeats)."""
        st = C.c_void_p(self._stream(stream))
        if len(coeffs) and isinstance(coeffs[0], (tuple, list)):
            rows = [tuple(float(v) for v in r) for r in coeffs]
            flat = (C.c_float * (3 * max(len(rows), 1)))(*[v for r in rows for v in r])
            _c.check(self._L.muon_step_schedule(self._h, P, G, M, float(beta), float(lr), float(wd),
                                                int(ns_steps), flat, len(rows), st),
                     "muon_step_schedule")
            return
        a, b, c = coeffs
        _c.check(self._L.muon_step(self._h, P, G, M, float(beta), float(lr), float(wd),
                                   int(ns_steps), float(a), float(b), float(c), st), "muon_step")

    def step(self, params, grads, momenta, beta, lr, wd, ns_steps=5, coeffs=QUINTIC,
             stream=None) -> None:
        """One Muon step on device tensors (params / momenta updated in place).
        coeffs: (a, b, c), or a per-step schedule [(a_0, b_0, c_0), ...]."""
        import torch
        pd = self._pdtype()
        P = self._ptrs(params, "params", pd, "cuda")
        G = self._ptrs(grads, "grads", pd, "cuda")
        M = self._ptrs(momenta, "momenta", torch.float32, "cuda")
        self._launch(P, G, M, beta, lr, wd, ns_steps, coeffs, stream)

    def bind(self, params, grads, momenta):
        """Validate and marshal the tensors once; the returned handle feeds
        step_bound() (the tensors must stay alive and in place)."""
        import torch
        pd = self._pdtype()
        return (self._ptrs(params, "params", pd, "cuda"), self._ptrs(grads, "grads", pd, "cuda"),
                self._ptrs(momenta, "momenta", torch.float32, "cuda"))

    def step_bound(self, bound, beta, lr, wd, ns_steps=5, coeffs=QUINTIC, stream=None) -> None:
        """muon_step on pointer arrays prepared by bind()."""
        P, G, M = bound
        self._launch(P, G, M, beta, lr, wd, ns_steps, coeffs, stream)

    def step_host(self, params, grads, momenta, beta, lr, wd, ns_steps=5, coeffs=QUINTIC,
                  stream=None) -> None:
        """The same step on host tensors (copied in and out by the library),
        for one (a, b, c) triple."""
        import torch
        if len(coeffs) != 3 or isinstance(coeffs[0], (tuple, list)):
            raise ValueError("step_host takes one (a, b, c) triple; per-step schedules go "
                             "through step()")
        pd = self._pdtype()
        P = self._ptrs(params, "params", pd, "cpu")
        G = self._ptrs(grads, "grads", pd, "cpu")
        M = self._ptrs(momenta, "momenta", torch.float32, "cpu")
        a, b, c = coeffs
        _c.check(self._L.muon_step_host(self._h, P, G, M, float(beta), float(lr), float(wd),
                                        int(ns_steps), float(a), float(b), float(c),
                                        C.c_void_p(self._stream(stream))), "muon_step_host")

    def debug_update(self, param_index: int, expert: int = 0):
        """O = X_k of one member as a float32 numpy array (needs keep_update)."""
        import numpy as np
        r, c = self.shapes[param_index][-2:]
        out = np.empty((r, c), dtype=np.float32)
        _c.check(self._L.muon_debug_copy_update(self._h, int(param_index), int(expert),
                                                out.ctypes.data_as(C.c_void_p)),
                 "muon_debug_copy_update")
        return out

    def group_elapsed_ms(self, group: int) -> float:
        """Device time of one group's kernels in the last step (group_timing)."""
        ms = C.c_float()
        _c.check(self._L.muon_plan_group_elapsed_ms(self._h, int(group), C.byref(ms)),
                 "muon_plan_group_elapsed_ms")
        return float(ms.value)

    def kernels_per_step(self, ns_steps: int) -> int:
        """Number of this library's kernel launches in one step."""
        n = 0
        for g in self.groups():
            if g["path"] == "skinny":
                # one fused kernel in Gram space (up to 64 steps), else momentum + iteration
                n += 1 if ns_steps <= 64 else 2
            elif g["path"] == "resident":
                n += 1  # the whole step of the group in one kernel
            else:
                n += 4 + 3 * int(ns_steps)
        return n

    def check_error(self) -> None:
        _c.check(self._L.muon_plan_check_error(self._h), "muon_plan_check_error")

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            self._L.muon_plan_destroy(self._h)
            self._h = C.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
