"""The allocation-free grad-norm entry point, lamb_grad_norm_noalloc.

It is for callers that cannot allocate device memory at the moment they need
the grad check (a framework allocator that has reserved nearly all of HBM, an
out-of-memory recovery path).  These tests call it through the C ABI and
compare what it writes with the grad norm, skip flag and clip factor that the
full step (lamb_step) reports for the same grads, twice in a row, since every
call reuses the same fixed scratch array.  The first call in this file also
exercises the per-device set-up when the file runs alone in a fresh process.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import workloads as W
from optimizer_step_gb300 import Lamb, _lib

pytestmark = pytest.mark.gpu

RTOL = 1e-5  # the one-step tolerance of the parity tests


def _noalloc(lib, sizes, grads, grad_dtype, loss_scale, clip, out):
    n = len(sizes)
    s = np.asarray(sizes, dtype=np.int64)
    ptrs = (ctypes.c_void_p * max(1, n))(*[g.data_ptr() if g.numel() else None for g in grads])
    stream = torch.cuda.current_stream().cuda_stream
    return lib.lamb_grad_norm_noalloc(n, s.ctypes.data, ptrs, grad_dtype, float(loss_scale),
                                      float(clip), ctypes.c_void_p(out.data_ptr()),
                                      ctypes.c_void_p(stream))


def _case(sizes, grad_dtype, S, clip, inject=None, seed=11):
    wl = W.Workload("noalloc", "noalloc", list(sizes), [1 if n > 4096 else 0 for n in sizes], [],
                    grad_dtype, t0=5, lr=1e-3, clip=clip, loss_scale=S, warm_state=True,
                    grad_kind="normal", grad_sigma=1e-3, seed=seed, inject=dict(inject or {}))
    return wl


def _reference(wl, gv):
    """grad norm, skip flag and step via the existing entry point (lamb_step)."""
    st = W.make_state(wl, "cuda")
    with Lamb(st.w, st.m, st.v, st.w16, wl.wd_flags, grad_dtype=wl.grad_dtype) as opt:
        return opt.step(wl.lr, wl.t0, wl.clip, wl.loss_scale, grads=gv)


@pytest.mark.parametrize("grad_dtype,S,clip", [(torch.bfloat16, 1.0, 0.05),
                                               (torch.float16, 1024.0, 0.0)])
def test_noalloc_grad_norm_matches_lamb_step_on_two_calls(grad_dtype, S, clip):
    lib = _lib.load()
    sizes = [1, 7, 300, 4097, 70001, 5000, 0, 1 << 20]
    wl = _case(sizes, grad_dtype, S, clip)
    _, gv = W.make_grads(wl, 1, "cuda")
    code = _lib.LAMB_GRAD_FP16 if grad_dtype == torch.float16 else _lib.LAMB_GRAD_BF16
    outs = []
    for _ in range(2):
        out = torch.full((3,), float("nan"), dtype=torch.float64, device="cuda")
        assert _noalloc(lib, sizes, gv, code, S, clip, out) == 0, lib.lamb_last_error()
        torch.cuda.synchronize()
        outs.append(out.tolist())
    skipped, gn = _reference(wl, gv)
    assert skipped is False
    for gn_na, c_na, nf_na in outs:
        assert nf_na == 0.0
        assert abs(gn_na - gn) <= RTOL * gn
        c_ref = clip / gn if (clip > 0 and gn > clip) else 1.0
        assert abs(c_na - c_ref) <= RTOL * c_ref
    assert outs[0] == outs[1]  # same grads, same fixed reduction order


def test_noalloc_flags_nonfinite_like_lamb_step_on_two_calls():
    lib = _lib.load()
    sizes = [40000, 300, 70001]
    wl = _case(sizes, torch.bfloat16, 1.0, 1.0, inject={1: "nan"})
    _, gv = W.make_grads(wl, 1, "cuda")
    for _ in range(2):
        out = torch.zeros(3, dtype=torch.float64, device="cuda")
        assert _noalloc(lib, sizes, gv, _lib.LAMB_GRAD_BF16, 1.0, 1.0, out) == 0
        torch.cuda.synchronize()
        gn_na, c_na, nf_na = out.tolist()
        assert nf_na == 1.0 and gn_na == math.inf and c_na == 0.0
    skipped, gn = _reference(wl, gv)
    assert skipped is True and gn == math.inf
    # A clean call afterwards starts from a cleared flag.
    _, gv2 = W.make_grads(wl, 2, "cuda")
    out = torch.zeros(3, dtype=torch.float64, device="cuda")
    assert _noalloc(lib, sizes, gv2, _lib.LAMB_GRAD_BF16, 1.0, 1.0, out) == 0
    torch.cuda.synchronize()
    assert out[2].item() == 0.0 and math.isfinite(out[0].item())


def test_noalloc_rejects_more_tensors_than_its_scratch_holds():
    lib = _lib.load()
    limit = 8192
    sizes = np.ones(limit + 1, dtype=np.int64)
    ptrs = (ctypes.c_void_p * (limit + 1))()
    out = torch.zeros(3, dtype=torch.float64, device="cuda")
    rc = lib.lamb_grad_norm_noalloc(limit + 1, sizes.ctypes.data, ptrs, 0, 1.0, 0.0,
                                    ctypes.c_void_p(out.data_ptr()), None)
    assert rc == _lib.LAMB_ERR_INVALID
    assert b"LAMB_NOALLOC_MAX_TENSORS" in lib.lamb_last_error()
