"""The allocation-free grad-norm entry point, lamb_grad_norm_noalloc.

It is for callers that cannot allocate device memory at the moment they need
the grad check (a framework allocator that has reserved nearly all of HBM, an
out-of-memory recovery path).  These tests call it through the C ABI and
compare what it writes with the CPU oracle's grad norm and with the grad
norm, skip flag and clip factor that the full step (lamb_step) reports for
the same grads, twice in a row, since every call reuses the same fixed
scratch array.  They also check that, after one warm-up call, further calls
leave the device's free memory and torch's reserved memory unchanged.  The
first call in this file also exercises the per-device set-up when the file
runs alone in a fresh process.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from optimizer_step_gb300 import Lamb, _lib

pytestmark = pytest.mark.gpu

RTOL = 1e-5  # the one-step tolerance of the parity tests


def f32c(x):
    return float(np.float32(x))


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


def _oracle_grad_norm(wl, gv):
    """The oracle's grad norm and skip flag for these grads (no state updated)."""
    g_host = [W.as_bits(x) for x in gv]
    n = len(g_host)
    none = [None] * n
    f32 = lambda x: float(np.float32(x))
    gd = oracle.GRAD_FP16 if wl.grad_dtype == torch.float16 else oracle.GRAD_BF16
    sk, gn = oracle.lamb_step(none, none, none, none, g_host, wl.wd_flags, grad_dtype=gd,
                              beta1=f32(wl.beta1), beta2=f32(wl.beta2), eps=f32(wl.eps),
                              weight_decay=f32(wl.weight_decay), lr=f32(wl.lr), t=wl.t0,
                              clip=f32(wl.clip), loss_scale=f32(wl.loss_scale),
                              update_mask=[0] * n)
    return sk, gn


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
    osk, ogn = _oracle_grad_norm(wl, gv)
    skipped, gn = _reference(wl, gv)
    assert skipped is False and osk == 0
    assert abs(gn - ogn) <= RTOL * ogn
    for gn_na, c_na, nf_na in outs:
        assert nf_na == 0.0
        assert abs(gn_na - ogn) <= RTOL * ogn  # against the oracle
        assert abs(gn_na - gn) <= RTOL * gn    # against lamb_step
        c_ref = f32c(clip) / ogn if (clip > 0 and ogn > f32c(clip)) else 1.0
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
    assert _oracle_grad_norm(wl, gv) == (1, math.inf)
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


def test_noalloc_calls_take_no_device_memory_after_a_warm_up_call():
    """After one warm-up call (which may load the library's module and its
    fixed array), ten more calls with both grad types leave the free device
    memory and torch's reserved memory exactly as they were."""
    lib = _lib.load()
    sizes = [300, 4097, 70001, 1 << 18]
    gvs = []
    for dt in (torch.bfloat16, torch.float16):
        _, gv = W.make_grads(_case(sizes, dt, 1.0, 0.0), 1, "cuda")
        gvs.append((dt, gv))
    out = torch.zeros(3, dtype=torch.float64, device="cuda")
    warm = torch.zeros(3, dtype=torch.float64, device="cuda")
    assert _noalloc(lib, [], [], _lib.LAMB_GRAD_BF16, 1.0, 0.0, warm) == 0, lib.lamb_last_error()
    torch.cuda.synchronize()
    assert warm.tolist() == [0.0, 1.0, 0.0]  # empty input: norm 0, no clip, finite
    torch.cuda.mem_get_info()  # the query itself sets nothing up after this
    free0 = torch.cuda.mem_get_info()[0]
    reserved0 = torch.cuda.memory_reserved()
    results = []
    for k in range(10):
        dt, gv = gvs[k % 2]
        code = _lib.LAMB_GRAD_FP16 if dt == torch.float16 else _lib.LAMB_GRAD_BF16
        assert _noalloc(lib, sizes, gv, code, 1.0, 0.0, out) == 0, lib.lamb_last_error()
        torch.cuda.synchronize()
        results.append(out[0].item())
        assert torch.cuda.mem_get_info()[0] == free0, f"call {k} changed free device memory"
        assert torch.cuda.memory_reserved() == reserved0
    assert all(math.isfinite(x) and x > 0 for x in results)
    assert results[0] == results[2] and results[1] == results[3]
