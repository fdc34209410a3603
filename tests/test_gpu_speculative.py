"""Speculative mode: a second set of m and v buffers lets one persistent
kernel read the grads once, sum the grad norm on the way and write the new
moments into the other set, then apply the update once the step is known to
be neither skipped nor clipped (a clipped step is redone from the untouched
set).  LAMB as adopted by MegaScale (guided-reading digest, section 2) on one
ZeRO-2 shard (digest, section 3).

The results must equal an ordinary step's bit for bit (w, m, v, the bf16
copy, the trust ratios; the grad norm is summed in another order) and match
the oracle within the parity tolerances, whichever set holds the state.
"""
import math

import numpy as np
import pytest
import torch

import workloads as W
from optimizer_step_gb300 import Lamb, LambError

from parity import assert_close, run_parity

pytestmark = pytest.mark.gpu


def _wl(sizes, clip, inject=None, grad_dtype=torch.bfloat16, S=1.0, seed=31, t0=3):
    return W.Workload("spec", "spec", list(sizes), [1 if n > 4096 else 0 for n in sizes],
                      [len(sizes) - 1], grad_dtype, t0=t0, lr=1e-3, clip=clip, loss_scale=S,
                      warm_state=True, grad_kind="normal", grad_sigma=1e-3, seed=seed,
                      inject=dict(inject or {}))


SIZES = [1, 300, 4096, 4097, 20000, 32768, 70001, 200003, 17, 5000]


def test_bit_identical_to_ordinary_steps_without_clipping():
    """Clip off, an inf at step 3: every step of a speculative handle equals
    the same step of an ordinary handle bit for bit."""
    wl = _wl(SIZES, clip=0.0, inject={3: "inf"})
    a, b = W.make_state(wl, "cuda"), W.make_state(wl, "cuda")
    gflat, gviews = W.grad_buffer(wl, "cuda")
    oa = Lamb(a.w, a.m, a.v, a.w16, wl.wd_flags)
    ob = Lamb(b.w, b.m, b.v, b.w16, wl.wd_flags)
    m2, v2 = torch.empty_like(b.m_flat), torch.empty_like(b.v_flat)
    ob.set_speculative(b.views(m2), b.views(v2))
    try:
        sets = []
        for k in range(1, 7):
            W.fill_grads(wl, k, gflat)
            ska, gna = oa.step(wl.lr, wl.t0 + k, 0.0, 1.0, grads=gviews)
            skb, gnb = ob.step(wl.lr, wl.t0 + k, 0.0, 1.0, grads=gviews)
            assert ska == skb == (k == 3)
            if ska:
                assert gna == gnb == math.inf
            else:
                assert abs(gna - gnb) <= 1e-6 * gna
            mb, vb = ob.state_buffers()
            sets.append(mb[0].data_ptr() == b.m[0].data_ptr())
            torch.cuda.synchronize()
            assert torch.equal(a.w_flat, b.w_flat) and torch.equal(a.w16_flat, b.w16_flat)
            for ma, mb_, va, vb_ in zip(a.m, mb, a.v, vb):
                assert torch.equal(ma, mb_) and torch.equal(va, vb_)
            assert np.array_equal(oa.trust(), ob.trust())
        # the state moved to the other set on every step that was not skipped
        assert sets == [False, True, True, False, True, False]
    finally:
        oa.close()
        ob.close()


def test_dynamic_loss_scaler_equals_ordinary_steps_bit_for_bit():
    """fp16 grads under a device-resident loss scaler that starts at 2^24:
    the first steps overflow and are skipped while the scale backs off, then
    it grows again after 3 clean steps.  A speculative handle follows an
    ordinary one step by step: the same skip flags and scale sequence, and
    the same state bit for bit."""
    wl = _wl([1 << 18, 70001, 4096, 300, 17], clip=0.0, grad_dtype=torch.float16, t0=1)
    a, b = W.make_state(wl, "cuda"), W.make_state(wl, "cuda")
    gflat, gviews = W.grad_buffer(wl, "cuda")
    oa = Lamb(a.w, a.m, a.v, a.w16, wl.wd_flags, grad_dtype=torch.float16)
    ob = Lamb(b.w, b.m, b.v, b.w16, wl.wd_flags, grad_dtype=torch.float16)
    m2, v2 = torch.empty_like(b.m_flat), torch.empty_like(b.v_flat)
    ob.set_speculative(b.views(m2), b.views(v2))
    cfg = dict(init_scale=2.0 ** 24, growth_factor=2.0, backoff_factor=0.5, growth_interval=3,
               min_scale=1.0, max_scale=2.0 ** 24)
    try:
        oa.set_loss_scaler(**cfg)
        ob.set_loss_scaler(**cfg)
        skips, scales, t = [], [], wl.t0
        for k in range(1, 15):
            scale = oa.next_loss_scale
            assert ob.next_loss_scale == scale
            scales.append(scale)
            W.fill_grads(wl, k, gflat, loss_scale=scale)
            ska, _ = oa.step(wl.lr, t, 0.0, 1.0, grads=gviews)
            skb, _ = ob.step(wl.lr, t, 0.0, 1.0, grads=gviews)
            assert ska == skb and oa.next_loss_scale == ob.next_loss_scale
            skips.append(int(ska))
            t += 0 if ska else 1
            torch.cuda.synchronize()
            mb, vb = ob.state_buffers()
            assert torch.equal(a.w_flat, b.w_flat) and torch.equal(a.w16_flat, b.w16_flat)
            for ma, mb_, va, vb_ in zip(a.m, mb, a.v, vb):
                assert torch.equal(ma, mb_) and torch.equal(va, vb_)
        assert skips[0] == 1 and 0 in skips and sum(skips) >= 2
        assert max(scales[skips.index(0):]) > min(scales)  # it grew again
    finally:
        oa.close()
        ob.close()


@pytest.mark.parametrize("seed", range(8))
def test_random_shards_speculative_match_the_oracle(seed):
    """Seeded random shards in speculative mode (sizes from tiny to several
    chunks, wd flags, grad type and loss scale, clipping off, active or
    inactive, so that some steps are redone), three steps against the
    oracle."""
    rng = np.random.default_rng(700 + seed)
    sizes = [int(rng.choice([rng.integers(1, 40), rng.integers(4090, 4110),
                             rng.integers(5000, 60000), rng.integers(60000, 300000)]))
             for _ in range(int(rng.integers(1, 10)))]
    fp16 = bool(rng.integers(0, 2))
    wl = W.Workload(f"spec-random{seed}", "spec-random", sizes,
                    [int(x) for x in rng.integers(0, 2, len(sizes))], [],
                    torch.float16 if fp16 else torch.bfloat16, t0=int(rng.integers(1, 800)),
                    lr=1e-3, clip=float(rng.choice([0.0, 1e-3, 1e3])),
                    loss_scale=4096.0 if fp16 else 1.0, warm_state=bool(rng.integers(0, 2)),
                    grad_kind="normal", grad_sigma=1e-3, seed=800 + seed)
    run_parity(wl, 3, check_steps=(1, 3), speculative=True)


def test_clipped_steps_are_redone_and_match_the_oracle():
    """The clip threshold sits inside the range of the grad norms, so some
    steps are clipped (redone from the untouched set) and some are not; fp16
    grads with a loss scale; every step against the oracle."""
    wl = _wl(SIZES, clip=0.0, grad_dtype=torch.float16, S=512.0, seed=32)
    norms = []
    for k in range(1, 9):
        flat, _ = W.make_grads(wl, k, "cuda")
        norms.append(float(flat.double().div(512.0).norm()))
    wl.clip = float(np.median(norms))
    log = run_parity(wl, 8, check_steps=range(1, 9), speculative=True)
    assert log["skipped"] == [0] * 8


def test_config_tiny_ten_steps_speculative():
    log = run_parity(W.tiny(), 10, check_steps=(1, 10), speculative=True)
    assert log["skipped"] == [0] * 10


def test_config_fp16_twenty_steps_speculative():
    wl = W.fp16_24()
    site7, site15 = W.injection_site(wl, 7), W.injection_site(wl, 15)
    subset = sorted(set(list(range(6)) + [site7[0], site15[0], len(wl.sizes) - 1]))
    log = run_parity(wl, 20, check_steps=(1, 6, 7, 8, 15, 16, 20), subset=subset,
                     speculative=True)
    assert log["skipped"] == [1 if k in (7, 15) else 0 for k in range(1, 21)]


def test_config_ragged_ten_steps_speculative():
    wl = W.ragged()
    rng = np.random.default_rng(1)
    subset = sorted(set(wl.zero_w) | set(int(i) for i in rng.choice(len(wl.sizes), 120, False))
                    | {int(np.argmax(wl.sizes))})
    run_parity(wl, 10, check_steps=(1, 10), subset=subset, speculative=True)


def test_snapshot_and_turning_the_mode_off_follow_the_state():
    wl = _wl(SIZES, clip=0.0, seed=33)
    st = W.make_state(wl, "cuda")
    gflat, gviews = W.grad_buffer(wl, "cuda")
    opt = Lamb(st.w, st.m, st.v, st.w16, wl.wd_flags)
    m2, v2 = torch.empty_like(st.m_flat), torch.empty_like(st.v_flat)
    opt.set_speculative(st.views(m2), st.views(v2))
    try:
        for k in range(1, 4):  # three clean steps: the state ends in the second set
            W.fill_grads(wl, k, gflat)
            assert opt.step(wl.lr, wl.t0 + k, 0.0, 1.0, grads=gviews)[0] is False
        m_cur, v_cur = opt.state_buffers()
        assert m_cur[0].data_ptr() == m2.data_ptr()
        want_m = [x.cpu() for x in m_cur]
        want_v = [x.cpu() for x in v_cur]
        host = [[torch.empty(n, dtype=torch.float32).pin_memory() for n in wl.sizes]
                for _ in range(3)]
        opt.snapshot_async(*host)
        opt.snapshot_wait()
        for got, want in zip(host[1] + host[2], want_m + want_v):
            assert torch.equal(got, want)
        # Off: the state moves back into m and v.
        opt.set_speculative(None, None)
        assert opt.info()["speculative"] == 0
        for x, y in zip(st.m + st.v, want_m + want_v):
            assert torch.equal(x.cpu(), y)
        # Both sets or neither.
        import ctypes
        from optimizer_step_gb300 import _lib
        ptrs = (ctypes.c_void_p * len(wl.sizes))(*[x.data_ptr() for x in st.views(m2)])
        assert opt._lib.lamb_set_speculative(opt._h, ptrs, None) == _lib.LAMB_ERR_INVALID
    finally:
        opt.close()


def test_tensors_shared_with_other_ranks_refuse_the_mode():
    wl = _wl([5000, 300], clip=0.0, seed=34)
    st = W.make_state(wl, "cuda")
    xn = torch.zeros(2, dtype=torch.float64, device="cuda")
    xt = torch.zeros(2, dtype=torch.float64, device="cuda")
    opt = Lamb(st.w, st.m, st.v, st.w16, wl.wd_flags, exchange_slots=[0, -1],
               norm_exchange=xn, tensor_exchange=xt)
    try:
        m2, v2 = torch.empty_like(st.m_flat), torch.empty_like(st.v_flat)
        with pytest.raises(LambError):
            opt.set_speculative(st.views(m2), st.views(v2))
    finally:
        opt.close()
