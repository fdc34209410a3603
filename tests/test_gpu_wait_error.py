"""The host's handling of a bounded wait that gives up inside the step's
apply pass (TMA copies from HBM that never arrive, or a tensor's trust ratio
that is never published to the fused moments-and-apply kernel).

No wait is ever made to run out here.  A test build of the library
(LAMB_TEST_APPLY_REPORTS_WAIT_ERROR) has CTA 0 of the kernel that applies the
update report a given-up wait after it has finished its work normally, with
nothing in flight; the test checks that lamb_step and lamb_step_result then
return LAMB_ERR_CUDA with the message that the state of the step is
undefined.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from optimizer_step_gb300 import _lib, build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def test_lib(tmp_path_factory):
    path = str(tmp_path_factory.mktemp("lamb_wait_error") / "liblamb_wait_error.so")
    build.build(defines=["LAMB_TEST_APPLY_REPORTS_WAIT_ERROR=1"], lib=path)
    lib = ctypes.CDLL(path)
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    lib.lamb_create.argtypes = [ctypes.POINTER(P), i32, P, P, P, P, P, P,
                                ctypes.POINTER(_lib.LambHParams), P]
    lib.lamb_step.argtypes = [P, P, f32, i64, f32, f32, ctypes.POINTER(_lib.LambResult)]
    lib.lamb_step_async.argtypes = [P, P, f32, f32, f32, ctypes.POINTER(i64)]
    lib.lamb_step_result.argtypes = [P, i64, i32, ctypes.POINTER(_lib.LambResult)]
    lib.lamb_destroy.argtypes = [P]
    lib.lamb_last_error.restype = ctypes.c_char_p
    return lib


def _ptrs(ts):
    return (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])


def test_a_reported_wait_error_fails_the_step(test_lib):
    sizes = [70001, 5000]
    wl = W.Workload("wait", "wait", sizes, [1, 0], [], torch.bfloat16, t0=1, lr=1e-3, clip=0.0,
                    loss_scale=1.0, warm_state=False, grad_kind="normal", grad_sigma=1e-3,
                    seed=5)
    st = W.make_state(wl, "cuda")
    _, gv = W.make_grads(wl, 1, "cuda")
    hp = _lib.LambHParams(0.9, 0.999, 1e-6, 0.01, _lib.LAMB_GRAD_BF16)
    s = np.asarray(sizes, np.int64)
    f = np.asarray(wl.wd_flags, np.uint8)
    h = ctypes.c_void_p()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert test_lib.lamb_create(ctypes.byref(h), 2, s.ctypes.data, f.ctypes.data, _ptrs(st.w),
                                _ptrs(st.m), _ptrs(st.v), _ptrs(st.w16), ctypes.byref(hp),
                                stream) == 0
    try:
        res = _lib.LambResult()
        rc = test_lib.lamb_step(h, _ptrs(gv), 1e-3, 1, 0.0, 1.0, ctypes.byref(res))
        assert rc == _lib.LAMB_ERR_CUDA
        assert b"bounded wait" in test_lib.lamb_last_error()
        seq = ctypes.c_int64()
        assert test_lib.lamb_step_async(h, _ptrs(gv), 1e-3, 0.0, 1.0, ctypes.byref(seq)) == 0
        rc = test_lib.lamb_step_result(h, seq.value, 1, ctypes.byref(res))
        assert rc == _lib.LAMB_ERR_CUDA
        assert b"state of this step is undefined" in test_lib.lamb_last_error()
    finally:
        assert test_lib.lamb_destroy(h) == 0
    # The context is still usable afterwards.
    assert torch.ones(4, device="cuda").sum().item() == 4.0
