"""Shared helpers of the GPU parity tests: run the CUDA library and the CPU
oracle on the same seeded inputs and compare element by element.

Tolerances: relative error <= 1e-5 after one step and <= 1e-4 after two or
more steps, with an absolute floor of 1e-9, for w, m, v and the grad norm.
Skip flags must match exactly.  The bf16 weight copy must be exactly the
bf16 rounding (nearest, ties to even) of the GPU's own fp32 weights, and may
differ from the oracle's copy by at most one bf16 ulp plus the fp32 weight
tolerance (rounding two fp32 values that differ within the weight tolerance
can land on bf16 neighbours, and near zero the weight tolerance itself can
exceed a bf16 ulp).  Hyperparameters cross the C ABI as
fp32, so the oracle is given those same fp32 values (widened to fp64).
"""
from __future__ import annotations

import math
from typing import Iterable, Optional, Sequence

import numpy as np
import torch

import oracle
import workloads as W
from optimizer_step_gb300 import Lamb

FLOOR = 1e-9


def f32(x: float) -> float:
    return float(np.float32(x))


def rtol_for(step_index: int) -> float:
    return 1e-5 if step_index <= 1 else 1e-4


def assert_close(got: np.ndarray, want: np.ndarray, rtol: float, what: str) -> None:
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    bound = np.maximum(FLOOR, rtol * np.abs(want))
    bad = ~(np.abs(got - want) <= bound)
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} of {got.size} elements off; first at "
                             f"{i}: got {got[i]!r} want {want[i]!r} (rtol {rtol})")


def check_bf16_copy(w16_gpu: np.ndarray, w_gpu: np.ndarray, w16_oracle: np.ndarray,
                    w_oracle: np.ndarray, rtol: float, what: str) -> int:
    """Returns the number of elements whose bf16 copy differs from the oracle's."""
    exact = oracle.bf16_rne(w_gpu)
    if not np.array_equal(w16_gpu, exact):
        i = int(np.flatnonzero(w16_gpu != exact)[0])
        raise AssertionError(f"{what}: w16 != bf16_rne(w) at {i}: {w16_gpu[i]:#06x} vs "
                             f"{exact[i]:#06x} (w {w_gpu[i]!r})")
    a = oracle.decode_grad(w16_gpu, oracle.GRAD_BF16)
    b = oracle.decode_grad(w16_oracle, oracle.GRAD_BF16)
    ulp = np.ldexp(1.0, np.frexp(np.maximum(np.abs(a), np.abs(b)))[1] - 8)
    wtol = np.maximum(FLOOR, rtol * np.abs(np.asarray(w_oracle, np.float64)))
    far = np.abs(a - b) > ulp + wtol
    if far.any():
        i = int(np.flatnonzero(far)[0])
        raise AssertionError(f"{what}: {int(far.sum())} bf16 copies too far from the oracle's; "
                             f"first at {i}: {a[i]!r} vs {b[i]!r} (w {w_gpu[i]!r} vs "
                             f"{w_oracle[i]!r})")
    return int(np.count_nonzero(w16_gpu != w16_oracle))


class HostState:
    """The oracle's own copy of (a subset of) the shard's state."""

    def __init__(self, st: W.State, subset: Optional[Sequence[int]]):
        n = len(st.wl.sizes)
        self.mask = np.ones(n, np.uint8) if subset is None else np.zeros(n, np.uint8)
        if subset is not None:
            self.mask[list(subset)] = 1
        self.w, self.m, self.v, self.w16 = [], [], [], []
        for i in range(n):
            if self.mask[i]:
                self.w.append(W.as_f32(st.w[i]).copy())
                self.m.append(W.as_f32(st.m[i]).copy())
                self.v.append(W.as_f32(st.v[i]).copy())
                self.w16.append(W.as_bits(st.w16[i]).copy())
            else:
                for lst in (self.w, self.m, self.v, self.w16):
                    lst.append(None)


def oracle_step(wl: W.Workload, hs: HostState, g_host, t: int):
    return oracle.lamb_step(
        hs.w, hs.m, hs.v, hs.w16, g_host, wl.wd_flags,
        grad_dtype=oracle.GRAD_FP16 if wl.grad_dtype == torch.float16 else oracle.GRAD_BF16,
        beta1=f32(wl.beta1), beta2=f32(wl.beta2), eps=f32(wl.eps),
        weight_decay=f32(wl.weight_decay), lr=f32(wl.lr), t=t, clip=f32(wl.clip),
        loss_scale=f32(wl.loss_scale), update_mask=hs.mask, want_trust=True)


def compare_state(st: W.State, hs: HostState, rtol: float, tag: str, opt: Lamb = None,
                  trust_oracle=None) -> dict:
    mism = 0
    count = 0
    for i, on in enumerate(hs.mask):
        if not on or st.wl.sizes[i] == 0:
            continue
        w_gpu = W.as_f32(st.w[i])
        assert_close(w_gpu, hs.w[i], rtol, f"{tag} w[{i}]")
        assert_close(W.as_f32(st.m[i]), hs.m[i], rtol, f"{tag} m[{i}]")
        assert_close(W.as_f32(st.v[i]), hs.v[i], rtol, f"{tag} v[{i}]")
        mism += check_bf16_copy(W.as_bits(st.w16[i]), w_gpu, hs.w16[i], hs.w[i], rtol,
                                f"{tag} w16[{i}]")
        count += st.wl.sizes[i]
    if opt is not None and trust_oracle is not None:
        tg = opt.trust()
        sel = [i for i, on in enumerate(hs.mask) if on and st.wl.sizes[i] > 0]
        assert_close(tg[sel], trust_oracle[sel], max(rtol, 1e-5), f"{tag} trust")
    return {"bf16_mismatch": mism, "checked": count}


class CurrentState:
    """A state whose m and v are the buffers that hold it now (speculative
    mode alternates between two sets)."""

    def __init__(self, st: W.State, opt: Lamb):
        self.wl, self.w, self.w16 = st.wl, st.w, st.w16
        self.m, self.v = opt.state_buffers()


def run_parity(wl: W.Workload, steps: int, check_steps: Iterable[int] = (),
               subset: Optional[Sequence[int]] = None, device: str = "cuda",
               speculative: bool = False) -> dict:
    """Runs ``steps`` steps of the GPU path and the oracle side by side.

    Every step compares the skip flag and the grad norm; the steps in
    ``check_steps`` also compare w, m, v, the bf16 copy and the trust ratios
    of the tensors in ``subset`` (all tensors if None).  ``speculative`` runs
    the library in speculative mode, with a second set of m and v buffers."""
    check_steps = set(check_steps)
    st = W.make_state(wl, device)
    hs = HostState(st, subset)
    gflat, gviews = W.grad_buffer(wl, device)
    opt = Lamb(st.w, st.m, st.v, st.w16, wl.wd_flags, beta1=wl.beta1, beta2=wl.beta2,
               eps=wl.eps, weight_decay=wl.weight_decay, grad_dtype=wl.grad_dtype)
    opt.set_grads(gviews)
    if speculative:
        m2, v2 = torch.empty_like(st.m_flat), torch.empty_like(st.v_flat)
        opt.set_speculative(st.views(m2), st.views(v2))
        assert opt.info()["speculative"] == 1
    t = wl.t0
    log = {"skipped": [], "bf16_mismatch": 0, "checked": 0}
    try:
        for k in range(1, steps + 1):
            W.fill_grads(wl, k, gflat)
            torch.cuda.synchronize()
            g_host = [W.as_bits(x) for x in gviews]
            sk, gn = opt.step(wl.lr, t, wl.clip, wl.loss_scale)
            osk, ogn, otrust = oracle_step(wl, hs, g_host, t)
            assert int(sk) == osk, f"step {k}: skip {sk} vs oracle {osk}"
            log["skipped"].append(int(sk))
            if osk:
                assert gn == math.inf
            else:
                assert_close(np.array([gn]), np.array([ogn]), rtol_for(k), f"step {k} grad_norm")
                t += 1
            if k in check_steps:
                cur = CurrentState(st, opt) if speculative else st
                r = compare_state(cur, hs, rtol_for(k), f"step {k}", opt,
                                  None if osk else otrust)
                log["bf16_mismatch"] += r["bf16_mismatch"]
                log["checked"] += r["checked"]
    finally:
        opt.close()
    return log


def run_parity_async(wl: W.Workload, phases: Sequence[int],
                     subset: Optional[Sequence[int]] = None, device: str = "cuda") -> dict:
    """Runs the GPU path with asynchronous steps (``step_async``: the step
    number on the GPU, no host wait between steps) against the oracle.

    ``phases`` lists step counts: each phase enqueues that many steps back to
    back, every step with its own grad buffer filled beforehand, then waits
    once, compares every step's outcome (skip flag, grad norm, the step number
    the GPU used) with the oracle's, and the state of ``subset`` (all tensors
    if None) at the end of the phase."""
    st = W.make_state(wl, device)
    hs = HostState(st, subset)
    opt = Lamb(st.w, st.m, st.v, st.w16, wl.wd_flags, beta1=wl.beta1, beta2=wl.beta2,
               eps=wl.eps, weight_decay=wl.weight_decay, grad_dtype=wl.grad_dtype)
    opt.set_step(wl.t0)
    t = wl.t0
    k = 0
    log = {"skipped": [], "bf16_mismatch": 0, "checked": 0, "t": []}
    try:
        for n_steps in phases:
            bufs = []
            for j in range(n_steps):
                flat, views = W.grad_buffer(wl, device)
                W.fill_grads(wl, k + j + 1, flat)
                bufs.append((flat, views, opt.prepare_grads(views)))
            torch.cuda.synchronize()
            seqs = [opt.step_async(wl.lr, wl.clip, wl.loss_scale, grads=b[2]) for b in bufs]
            outcomes = [opt.result(q) for q in seqs]
            for (flat, views, _), (sk, gn, t_gpu) in zip(bufs, outcomes):
                k += 1
                g_host = [W.as_bits(x) for x in views]
                osk, ogn, otrust = oracle_step(wl, hs, g_host, t)
                assert int(sk) == osk, f"step {k}: skip {sk} vs oracle {osk}"
                assert t_gpu == t, f"step {k}: the GPU used t={t_gpu}, the oracle t={t}"
                log["skipped"].append(int(sk))
                log["t"].append(t_gpu)
                if osk:
                    assert gn == math.inf
                else:
                    assert_close(np.array([gn]), np.array([ogn]), rtol_for(k),
                                 f"step {k} grad_norm")
                    t += 1
            r = compare_state(st, hs, rtol_for(k), f"after step {k}", opt,
                              None if osk else otrust)
            log["bf16_mismatch"] += r["bf16_mismatch"]
            log["checked"] += r["checked"]
            del bufs
    finally:
        opt.close()
    return log
