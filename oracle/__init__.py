"""CPU reference ("oracle") for one LAMB step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product library (``optimizer_step_gb300``)
never imports it, and the two share no code.

The arithmetic lives in ``lamb_oracle.cpp`` (plain C++17, fp64); this module
only builds it with g++ and marshals numpy arrays through ctypes.  The method
is LAMB (You et al., ICLR 2020) as adopted by MegaScale (guided-reading digest,
section 2), applied to one ZeRO-2 shard (digest, section 3); the step order is
listed in ``lamb_oracle.h``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lamb_oracle.cpp")
_HDR = os.path.join(_HERE, "lamb_oracle.h")
_LIB = os.path.join(_HERE, "liblamb_oracle.so")

GRAD_BF16 = 0
GRAD_FP16 = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (no FMA contraction, no fast-math)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest:
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread", "-Wall", "-Wextra", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            lib.oracle_lamb_step.restype = ctypes.c_int
            lib.oracle_lamb_step.argtypes = [
                ctypes.c_int32, P, P, P, P, P, P, P, ctypes.c_int32,
                ctypes.c_double, ctypes.c_double, ctypes.c_double, ctypes.c_double,
                ctypes.c_double, ctypes.c_int64, ctypes.c_double, ctypes.c_double,
                P, ctypes.c_int32, P, P, P]
            lib.oracle_decode_grad_n.restype = None
            lib.oracle_decode_grad_n.argtypes = [P, ctypes.c_int64, ctypes.c_int32, P]
            lib.oracle_loss_scale_update.restype = None
            lib.oracle_loss_scale_update.argtypes = [
                P, P, ctypes.c_int32, ctypes.c_float, ctypes.c_float, ctypes.c_int32,
                ctypes.c_float, ctypes.c_float]
            lib.oracle_bf16_rne_n.restype = None
            lib.oracle_bf16_rne_n.argtypes = [P, ctypes.c_int64, P]
            _lib = lib
    return _lib


def _ptr_array(arrays):
    out = (ctypes.c_void_p * max(1, len(arrays)))()
    for i, a in enumerate(arrays):
        out[i] = None if a is None else a.ctypes.data
    return out


def _check(a, dtype, name):
    if a is None:
        return
    if a.dtype != dtype or not a.flags["C_CONTIGUOUS"] or not a.flags["WRITEABLE"]:
        raise TypeError(f"{name}: need a writeable C-contiguous {np.dtype(dtype)} array")


def lamb_step(w, m, v, w16, g, wd_flags, *, grad_dtype, beta1, beta2, eps, weight_decay,
              lr, t, clip=0.0, loss_scale=1.0, update_mask=None, n_threads=0,
              want_trust=False):
    """One oracle LAMB step, in place on lists of numpy arrays.

    ``w, m, v``: float32 arrays; ``w16``: uint16 (bf16 bit patterns, written);
    ``g``: uint16 bit patterns of bf16 (``grad_dtype=GRAD_BF16``) or fp16
    grads.  Entries of unmasked tensors may be ``None`` in w/m/v/w16.
    Returns ``(skipped, grad_norm)`` or ``(skipped, grad_norm, trust)``.
    """
    lib = _load()
    n = len(g)
    for lst, dt, nm in ((w, np.float32, "w"), (m, np.float32, "m"),
                        (v, np.float32, "v"), (w16, np.uint16, "w16")):
        if len(lst) != n:
            raise ValueError(f"{nm}: expected {n} arrays")
        for a in lst:
            _check(a, dt, nm)
    for a in g:
        if a.dtype != np.uint16 or not a.flags["C_CONTIGUOUS"]:
            raise TypeError("g: need C-contiguous uint16 bit patterns")
    sizes = np.array([a.size for a in g], dtype=np.int64)
    wd = np.ascontiguousarray(np.asarray(wd_flags, dtype=np.uint8))
    mask = None if update_mask is None else np.ascontiguousarray(
        np.asarray(update_mask, dtype=np.uint8))
    for i in range(n):
        if mask is None or mask[i]:
            for lst in (w, m, v, w16):
                if lst[i] is None or lst[i].size != sizes[i]:
                    raise ValueError(f"tensor {i}: state size mismatch")
    trust = np.full(n, np.nan, dtype=np.float64)
    skipped = ctypes.c_int32(0)
    gn = ctypes.c_double(0.0)
    rc = lib.oracle_lamb_step(
        n, sizes.ctypes.data, wd.ctypes.data, _ptr_array(w), _ptr_array(m), _ptr_array(v),
        _ptr_array(w16), _ptr_array(g), grad_dtype, float(beta1), float(beta2), float(eps),
        float(weight_decay), float(lr), int(t), float(clip), float(loss_scale),
        None if mask is None else mask.ctypes.data, int(n_threads),
        ctypes.addressof(skipped), ctypes.addressof(gn), trust.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_lamb_step rejected its arguments")
    if want_trust:
        return int(skipped.value), float(gn.value), trust
    return int(skipped.value), float(gn.value)


def loss_scale_update(scale, good_steps, found_inf, *, growth=2.0, backoff=0.5,
                      growth_interval=2000, min_scale=0.0, max_scale=float("inf")):
    """One dynamic loss-scale update; returns the new (scale, good_steps)."""
    s = ctypes.c_float(scale)
    g = ctypes.c_int32(good_steps)
    _load().oracle_loss_scale_update(ctypes.addressof(s), ctypes.addressof(g),
                                     1 if found_inf else 0, growth, backoff,
                                     growth_interval, min_scale, max_scale)
    return float(s.value), int(g.value)


def decode_grad(bits: np.ndarray, grad_dtype: int) -> np.ndarray:
    """Decode bf16/fp16 bit patterns to float64."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().oracle_decode_grad_n(bits.ctypes.data, bits.size, grad_dtype, out.ctypes.data)
    return out


def bf16_rne(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 bit patterns (nearest, ties to even)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_bf16_rne_n(x.ctypes.data, x.size, out.ctypes.data)
    return out
