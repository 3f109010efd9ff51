"""ctypes declarations of the C ABI in include/muon.h (argument marshalling only).

The library is the in-tree ``_lib/libmuon_gb300.so`` built by ``build.py``.
Loading fails loudly when it is missing: there is no fallback path.
"""
from __future__ import annotations

import ctypes as C
import os

from . import build as _build

MUON_OK = 0
MUON_ERR_INVALID_ARG = 1
MUON_ERR_UNSUPPORTED = 2
MUON_ERR_OOM = 3
MUON_ERR_CUDA = 4
MUON_ERR_TIMEOUT = 5

MUON_MODE_BF16 = 0
MUON_MODE_FP32 = 1
MUON_NS_FP16 = 0
MUON_NS_BF16 = 1
MUON_SCALE_SQRT_ASPECT = 0
MUON_SCALE_RMS_0_2 = 1
MUON_SCALE_NONE = 2
MUON_PATH_AUTO = 0
MUON_PATH_SKINNY = 1
MUON_PATH_TENSOR = 2
MUON_PATH_SIMT = 3
MUON_PATH_RESIDENT = 4
MUON_FLAG_KEEP_UPDATE = 1
MUON_FLAG_NO_GRAPH = 2
MUON_FLAG_HOST_STAGING = 4
MUON_FLAG_GROUP_TIMING = 8
MUON_FLAG_NESTEROV = 16
MUON_FLAG_MERGE_TRANSPOSED = 32
MUON_MAX_SCHEDULE_ROWS = 64


class muon_shape_t(C.Structure):
    _fields_ = [("ndim", C.c_int32), ("reserved_", C.c_int32), ("dims", C.c_int64 * 3)]


class muon_plan_options(C.Structure):
    _fields_ = [("mode", C.c_int32), ("scale", C.c_int32), ("eps", C.c_float),
                ("skinny_threshold", C.c_int32), ("ns_dtype", C.c_int32),
                ("flags", C.c_uint32), ("path_override", C.c_int32),
                ("max_streams", C.c_int32), ("column_shards", C.c_int32),
                ("reserved", C.c_int32 * 7)]


class muon_group_info_t(C.Structure):
    _fields_ = [("rows", C.c_int64), ("cols", C.c_int64), ("batch", C.c_int64),
                ("first_member", C.c_int64), ("transposed", C.c_int32), ("path", C.c_int32),
                ("workspace_bytes", C.c_int64)]


# test hooks declared in include/muon_testing.h
EXPORTED_TESTING = ["muon_testing_tc_gemm", "muon_testing_skinny_max_clusters",
                    "muon_testing_tile_walk", "muon_testing_tile_walk_pair",
                    "muon_testing_tc_pair_form", "muon_testing_wait_probe"]

# every symbol include/muon.h declares, for the export check
EXPORTED = ["muon_default_options", "muon_plan_describe", "muon_plan_create", "muon_step",
            "muon_step_schedule", "muon_step_host", "muon_plan_destroy", "muon_plan_num_groups",
            "muon_plan_group_info", "muon_plan_workspace_bytes", "muon_debug_copy_update",
            "muon_plan_assign",
            "muon_plan_check_error", "muon_plan_group_elapsed_ms", "muon_step_skinny_static",
            "muon_status_string",
            "muon_last_error", "muon_version"]

_lib = None


def lib_path() -> str:
    return _build.lib_path()


def load() -> C.CDLL:
    """Load the library; raises if the .so has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(
            f"CUDA library {path} is missing; build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = C.CDLL(path)
    vp, i32, i64, f32 = C.c_void_p, C.c_int32, C.c_int64, C.c_float
    L.muon_default_options.argtypes = [C.POINTER(muon_plan_options)]
    L.muon_plan_describe.argtypes = [C.POINTER(muon_shape_t), i32, C.POINTER(muon_plan_options),
                                     C.POINTER(muon_group_info_t), i32, C.POINTER(i32),
                                     C.POINTER(i32), C.POINTER(i32), i64, C.POINTER(i64),
                                     C.POINTER(C.c_size_t)]
    L.muon_plan_create.argtypes = [C.POINTER(muon_shape_t), i32, C.POINTER(muon_plan_options),
                                   C.c_int, C.POINTER(vp)]
    L.muon_step.argtypes = [vp, C.POINTER(vp), C.POINTER(vp), C.POINTER(vp), f32, f32, f32, i32,
                            f32, f32, f32, vp]
    L.muon_step_host.argtypes = L.muon_step.argtypes
    L.muon_step_schedule.argtypes = [vp, C.POINTER(vp), C.POINTER(vp), C.POINTER(vp), f32, f32, f32,
                                     i32, C.POINTER(f32), i32, vp]
    L.muon_plan_destroy.argtypes = [vp]
    L.muon_plan_assign.argtypes = [C.POINTER(muon_shape_t), i32, C.POINTER(muon_plan_options), i32, i32,
                                   C.POINTER(i32), i64, C.POINTER(C.c_double), C.POINTER(C.c_double)]
    L.muon_plan_num_groups.argtypes = [vp]
    L.muon_plan_num_groups.restype = i32
    L.muon_plan_group_info.argtypes = [vp, i32, C.POINTER(muon_group_info_t)]
    L.muon_plan_workspace_bytes.argtypes = [vp]
    L.muon_plan_workspace_bytes.restype = C.c_size_t
    L.muon_debug_copy_update.argtypes = [vp, i32, i64, vp]
    L.muon_plan_check_error.argtypes = [vp]
    L.muon_plan_group_elapsed_ms.argtypes = [vp, i32, C.POINTER(C.c_float)]
    L.muon_step_skinny_static.argtypes = [vp, vp, vp, i32, i64, i64, f32, f32, f32, i32, f32,
                                          f32, f32, f32, i32, vp]
    L.muon_step_skinny_static.restype = C.c_int
    L.muon_testing_tc_gemm.argtypes = [i32, i32, i32, i64, i64, vp, vp, vp, vp, f32, f32, f32,
                                       f32, vp]
    L.muon_testing_tc_gemm.restype = C.c_int
    L.muon_testing_skinny_max_clusters.argtypes = [i32, i64]
    L.muon_testing_skinny_max_clusters.restype = i32
    L.muon_testing_tile_walk.argtypes = [i32, i64, i64, i32, C.POINTER(i32), C.POINTER(i32), i32]
    L.muon_testing_tile_walk.restype = i32
    L.muon_testing_tile_walk_pair.argtypes = [i32, i64, i64, C.POINTER(i32), C.POINTER(i32), i32]
    L.muon_testing_tile_walk_pair.restype = i32
    L.muon_testing_tc_pair_form.argtypes = [i64]
    L.muon_testing_tc_pair_form.restype = i32
    L.muon_testing_wait_probe.argtypes = [i32, i64, vp]
    L.muon_testing_wait_probe.restype = C.c_int
    L.muon_status_string.argtypes = [C.c_int]
    L.muon_status_string.restype = C.c_char_p
    L.muon_last_error.argtypes = []
    L.muon_last_error.restype = C.c_char_p
    L.muon_version.argtypes = []
    L.muon_version.restype = C.c_char_p
    for name in ("muon_default_options", "muon_plan_describe", "muon_plan_create", "muon_step",
                 "muon_step_schedule", "muon_step_host", "muon_plan_destroy", "muon_plan_group_info",
                 "muon_debug_copy_update", "muon_plan_check_error",
                 "muon_plan_group_elapsed_ms"):
        getattr(L, name).restype = C.c_int
    _lib = L
    return L


class MuonError(RuntimeError):
    def __init__(self, status: int, where: str):
        L = load()
        msg = L.muon_last_error().decode(errors="replace")
        name = L.muon_status_string(status).decode()
        super().__init__(f"{where}: {name}: {msg}")
        self.status = status


def check(status: int, where: str) -> None:
    if status != MUON_OK:
        raise MuonError(status, where)
