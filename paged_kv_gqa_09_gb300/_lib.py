"""ctypes binding of libpkv (include/pkv.h): struct layouts and symbol types.

Loading fails loudly (``PkvLibraryError``) when libpkv.so has not been built;
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB

PKV_OK = 0
PKV_EINVAL = -1
PKV_EUNSUPPORTED = -2
PKV_ECUDA = -3
PKV_EDEVICE = -4
PKV_ETIMEOUT = -5
PKV_ECAPACITY = -6

PKV_PATH_BUCKETED_SPLIT = 0
PKV_PATH_WORKQUEUE = 1
PKV_PATH_SINGLE_PASS = 2

PKV_MERGE_SEPARATE = 0  # the split states are merged by a second kernel
PKV_MERGE_FUSED = 1     # merged on the decode kernel's tail
PKV_PLAN_SEPARATE = 0   # the workqueue's plan is its own launch (pkv_plan)
PKV_PLAN_IN_DECODE = 1  # the decode kernel builds the plan itself (B <= PKV_SELF_PLAN_MAX_B)
PKV_SELF_PLAN_MAX_B = 512
PATH_EXACT_BUCKETS = 3  # step-model only

NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024  # PKV_NOALLOC_SCRATCH_BYTES in include/pkv.h

STATUS_NAMES = {
    PKV_OK: "PKV_OK", PKV_EINVAL: "PKV_EINVAL", PKV_EUNSUPPORTED: "PKV_EUNSUPPORTED",
    PKV_ECUDA: "PKV_ECUDA", PKV_EDEVICE: "PKV_EDEVICE", PKV_ETIMEOUT: "PKV_ETIMEOUT",
    PKV_ECAPACITY: "PKV_ECAPACITY",
}

# every symbol include/pkv.h declares
EXPORTS = [
    "pkv_plan_workspace_size", "pkv_partials_size", "pkv_plan", "pkv_decode", "pkv_merge",
    "pkv_decode_merge",
    "pkv_single_pass", "pkv_decode_step", "pkv_decode_step_rows", "pkv_decode_step_noalloc",
    "pkv_decode_step_host", "pkv_append_decode_step_host",
    "pkv_append", "pkv_append_plan", "pkv_exact_length_groups", "pkv_policy_default", "pkv_policy",
    "pkv_cost_model_default", "pkv_policy_learned",
    "pkv_get_counters", "pkv_reset_counters", "pkv_step_model", "pkv_get_error",
    "pkv_test_starve_next_decodes", "pkv_last_error_string", "pkv_version",
]


class PkvLibraryError(RuntimeError):
    pass


class PkvError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {detail}")
        self.status = status


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("d", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("bt_stride", ctypes.c_int32),
                ("scale", ctypes.c_float)]


class PlanCfg(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("split_tokens", ctypes.c_int32),
                ("bucket_len", ctypes.c_int32), ("max_tasks", ctypes.c_int32),
                ("merge", ctypes.c_int32), ("plan", ctypes.c_int32)]


class PolicyCfg(ctypes.Structure):
    _fields_ = [("bucketed_min_tokens", ctypes.c_int32), ("bucketed_max_batch", ctypes.c_int32),
                ("workqueue_min_tokens", ctypes.c_int32), ("workqueue_min_batch", ctypes.c_int32),
                ("split_tokens", ctypes.c_int32), ("bucketed_split_tokens", ctypes.c_int32),
                ("workqueue_max_split_tokens", ctypes.c_int32),
                ("workqueue_target_splits", ctypes.c_int32),
                ("workqueue_min_long_splits", ctypes.c_int32)]


COST_FEATURES = 10
COST_MAX_ROUTES = 16


class CostRoute(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("split_tokens", ctypes.c_int32),
                ("w", ctypes.c_float * COST_FEATURES)]


class CostModel(ctypes.Structure):
    _fields_ = [("n_routes", ctypes.c_int32), ("route", CostRoute * COST_MAX_ROUTES)]


class Counters(ctypes.Structure):
    _fields_ = [("plan_launches", ctypes.c_int64), ("decode_launches", ctypes.c_int64),
                ("merge_launches", ctypes.c_int64), ("single_pass_launches", ctypes.c_int64),
                ("append_launches", ctypes.c_int64)]


class StepModel(ctypes.Structure):
    _fields_ = [("attn_launches", ctypes.c_int64), ("plan_launches", ctypes.c_int64),
                ("tasks", ctypes.c_int64), ("grid_tasks", ctypes.c_int64),
                ("states_written", ctypes.c_int64), ("states_read", ctypes.c_int64),
                ("merge_state_bytes", ctypes.c_int64), ("kv_bytes", ctypes.c_int64)]


_lib = None
_lock = threading.Lock()


def lib_path() -> str:
    return os.environ.get("PKV_LIB", LIB)


def load() -> ctypes.CDLL:
    """Load libpkv.so (built by ``paged_kv_gqa_09_gb300.build.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = lib_path()
        if not os.path.exists(path):
            raise PkvLibraryError(
                f"libpkv.so not found at {path}: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(path)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        S, C, PC = ctypes.POINTER(Shape), ctypes.POINTER(PlanCfg), ctypes.POINTER(PolicyCfg)
        sig = {
            "pkv_plan_workspace_size": (sz, [S, C]),
            "pkv_partials_size": (sz, [S, C]),
            "pkv_plan": (ctypes.c_int, [S, C, vp, vp, vp]),
            "pkv_decode": (ctypes.c_int, [S, C, vp, vp, vp, vp, vp, vp, vp, vp]),
            "pkv_decode_merge": (ctypes.c_int, [S, C, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
            "pkv_merge": (ctypes.c_int, [S, C, vp, vp, vp, vp, vp, vp]),
            "pkv_single_pass": (ctypes.c_int, [S, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
            "pkv_decode_step": (ctypes.c_int, [S, C, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
            "pkv_decode_step_noalloc": (ctypes.c_int, [S, C, vp, vp, vp, vp, vp, vp, vp, vp]),
            "pkv_decode_step_host": (ctypes.c_int, [S, C] + [vp] * 15),
            "pkv_append_decode_step_host": (ctypes.c_int, [S, C] + [vp] * 19),
            "pkv_decode_step_rows": (ctypes.c_int, [S, C, vp, vp, i32] + [vp] * 9),
            "pkv_append": (ctypes.c_int, [S, vp, vp, vp, vp, vp, vp, vp, vp]),
            "pkv_append_plan": (ctypes.c_int, [S, C] + [vp] * 10),
            "pkv_exact_length_groups": (ctypes.c_int, [vp, i32, vp, vp, vp, ctypes.POINTER(ctypes.c_int32)]),
            "pkv_policy_default": (None, [PC]),
            "pkv_policy": (ctypes.c_int, [i32, i32, PC, ctypes.POINTER(ctypes.c_int32),
                                          ctypes.POINTER(ctypes.c_int32)]),
            "pkv_cost_model_default": (None, [ctypes.POINTER(CostModel)]),
            "pkv_policy_learned": (ctypes.c_int, [i32, i32, ctypes.c_int64, ctypes.POINTER(CostModel),
                                                  ctypes.POINTER(ctypes.c_int32),
                                                  ctypes.POINTER(ctypes.c_int32)]),
            "pkv_get_counters": (ctypes.c_int, [ctypes.POINTER(Counters)]),
            "pkv_reset_counters": (ctypes.c_int, []),
            "pkv_step_model": (ctypes.c_int, [i32, S, i32, i32, vp, ctypes.POINTER(StepModel)]),
            "pkv_get_error": (ctypes.c_int, [vp, vp]),
            "pkv_test_starve_next_decodes": (ctypes.c_int, [i32]),
            "pkv_last_error_string": (ctypes.c_char_p, []),
            "pkv_version": (ctypes.c_int, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
        return L


def last_error() -> str:
    return load().pkv_last_error_string().decode(errors="replace")


def check(status: int, where: str) -> None:
    if status != PKV_OK:
        raise PkvError(status, where, last_error())
