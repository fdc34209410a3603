"""ctypes loader for ``liblamb_gb300.so`` (argument marshalling only).

The names mirror ``include/lamb.h``.  Loading never falls back to anything:
if the library is missing it is built from source, and if it cannot be built
or loaded an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

LAMB_OK = 0
LAMB_ERR_INVALID = -1
LAMB_ERR_ALIGN = -2
LAMB_ERR_CUDA = -3
LAMB_ERR_NOMEM = -4
LAMB_NOT_READY = 1
LAMB_GRAD_BF16 = 0
LAMB_GRAD_FP16 = 1

# Every symbol include/lamb.h declares.
EXPORTS = ("lamb_create", "lamb_step", "lamb_destroy", "lamb_last_error", "lamb_get_trust",
           "lamb_set_timing", "lamb_kernel_times", "lamb_plan", "lamb_plan_limits",
           "lamb_set_loss_scaler", "lamb_snapshot_async", "lamb_snapshot_wait",
           "lamb_grad_norm_noalloc", "lamb_step_async", "lamb_step_result", "lamb_set_step",
           "lamb_loss_scale_device", "lamb_step_kernel_times", "lamb_create_sharded",
           "lamb_split_norms", "lamb_split_moments", "lamb_split_apply",
           "lamb_get_info", "lamb_set_speculative", "lamb_state_buffers")


class LambHParams(ctypes.Structure):
    _fields_ = [("beta1", ctypes.c_float), ("beta2", ctypes.c_float), ("eps", ctypes.c_float),
                ("weight_decay", ctypes.c_float), ("grad_dtype", ctypes.c_int32)]


class LambResult(ctypes.Structure):
    _fields_ = [("skipped", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("grad_norm", ctypes.c_double), ("loss_scale", ctypes.c_float),
                ("next_loss_scale", ctypes.c_float), ("t", ctypes.c_int64)]


class LambLossScaler(ctypes.Structure):
    _fields_ = [("init_scale", ctypes.c_float), ("growth_factor", ctypes.c_float),
                ("backoff_factor", ctypes.c_float), ("growth_interval", ctypes.c_int32),
                ("min_scale", ctypes.c_float), ("max_scale", ctypes.c_float)]


class LambInfo(ctypes.Structure):
    _fields_ = [("n_params", ctypes.c_int64), ("one_pass_params", ctypes.c_int64),
                ("chunk_elems", ctypes.c_int64), ("n_items", ctypes.c_int64),
                ("fused", ctypes.c_int32), ("speculative", ctypes.c_int32)]


class LambWorkItem(ctypes.Structure):
    _fields_ = [("begin", ctypes.c_int64), ("count", ctypes.c_int32), ("tensor", ctypes.c_int32)]


class LambError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"lamb error {code}: {msg}")
        self.code = code


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load the in-tree library (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build_if_missing:
            _build.build()
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"{_build.LIB} is missing: build it with optimizer_step_gb300.build")
        lib = ctypes.CDLL(_build.LIB)
        P = ctypes.c_void_p
        i32, i64, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        lib.lamb_create.restype = ctypes.c_int
        lib.lamb_create.argtypes = [ctypes.POINTER(P), i32, P, P, P, P, P, P,
                                    ctypes.POINTER(LambHParams), P]
        lib.lamb_create_sharded.restype = ctypes.c_int
        lib.lamb_create_sharded.argtypes = [ctypes.POINTER(P), i32, P, P, P, P, P, P, P, i32, P,
                                            P, ctypes.POINTER(LambHParams), P]
        lib.lamb_split_norms.restype = ctypes.c_int
        lib.lamb_split_norms.argtypes = [P, P, f32]
        lib.lamb_split_moments.restype = ctypes.c_int
        lib.lamb_split_moments.argtypes = [P, f32, i64, f32]
        lib.lamb_split_apply.restype = ctypes.c_int
        lib.lamb_split_apply.argtypes = [P, ctypes.POINTER(i64)]
        lib.lamb_set_speculative.restype = ctypes.c_int
        lib.lamb_set_speculative.argtypes = [P, P, P]
        lib.lamb_state_buffers.restype = ctypes.c_int
        lib.lamb_state_buffers.argtypes = [P, ctypes.POINTER(i32)]
        lib.lamb_get_info.restype = ctypes.c_int
        lib.lamb_get_info.argtypes = [P, ctypes.POINTER(LambInfo)]
        lib.lamb_step.restype = ctypes.c_int
        lib.lamb_step.argtypes = [P, P, f32, i64, f32, f32, ctypes.POINTER(LambResult)]
        lib.lamb_step_async.restype = ctypes.c_int
        lib.lamb_step_async.argtypes = [P, P, f32, f32, f32, ctypes.POINTER(i64)]
        lib.lamb_step_result.restype = ctypes.c_int
        lib.lamb_step_result.argtypes = [P, i64, i32, ctypes.POINTER(LambResult)]
        lib.lamb_set_step.restype = ctypes.c_int
        lib.lamb_set_step.argtypes = [P, i64]
        lib.lamb_loss_scale_device.restype = ctypes.c_int
        lib.lamb_loss_scale_device.argtypes = [P, ctypes.POINTER(P)]
        lib.lamb_destroy.restype = ctypes.c_int
        lib.lamb_destroy.argtypes = [P]
        lib.lamb_last_error.restype = ctypes.c_char_p
        lib.lamb_last_error.argtypes = []
        lib.lamb_get_trust.restype = ctypes.c_int
        lib.lamb_get_trust.argtypes = [P, P, i32]
        lib.lamb_set_loss_scaler.restype = ctypes.c_int
        lib.lamb_set_loss_scaler.argtypes = [P, ctypes.POINTER(LambLossScaler)]
        lib.lamb_snapshot_async.restype = ctypes.c_int
        lib.lamb_snapshot_async.argtypes = [P, P, P, P, P]
        lib.lamb_snapshot_wait.restype = ctypes.c_int
        lib.lamb_snapshot_wait.argtypes = [P]
        lib.lamb_set_timing.restype = ctypes.c_int
        lib.lamb_set_timing.argtypes = [P, i32]
        lib.lamb_step_kernel_times.restype = ctypes.c_int
        lib.lamb_step_kernel_times.argtypes = [P, i64, P]
        lib.lamb_kernel_times.restype = ctypes.c_int
        lib.lamb_kernel_times.argtypes = [P, P]
        lib.lamb_plan.restype = ctypes.c_int
        lib.lamb_plan.argtypes = [i32, P, i64, P, i64, P, i64, ctypes.POINTER(i64),
                                  ctypes.POINTER(i64)]
        lib.lamb_grad_norm_noalloc.restype = ctypes.c_int
        lib.lamb_grad_norm_noalloc.argtypes = [i32, P, P, i32, f32, f32, P, P]
        lib.lamb_plan_limits.restype = None
        lib.lamb_plan_limits.argtypes = [ctypes.POINTER(i64)] * 4
        _lib = lib
        return lib


def check(rc: int) -> None:
    if rc != LAMB_OK:
        msg = load().lamb_last_error()
        raise LambError(rc, msg.decode() if msg else "")
