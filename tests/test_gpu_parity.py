"""GPU parity: the CUDA library against the CPU oracle on the same seeded
inputs (see tests/parity.py for the tolerances).  All of these need a GPU."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from optimizer_step_gb300 import Lamb, LambError

from parity import assert_close, check_bf16_copy, f32, run_parity, run_parity_async

pytestmark = pytest.mark.gpu


def custom(sizes, *, wd=None, zero=(), grad_dtype=torch.bfloat16, t0=1, clip=0.0, S=1.0,
           warm=True, seed=7, inject=None, kind="normal", sigma=1e-3):
    return W.Workload("custom", "custom", list(sizes),
                      list(wd) if wd is not None else [1 if n > 4096 else 0 for n in sizes],
                      list(zero), grad_dtype, t0=t0, lr=1e-3, clip=clip, loss_scale=S,
                      warm_state=warm, grad_kind=kind, grad_sigma=sigma, seed=seed,
                      inject=dict(inject or {}))


# -------------------------------------------------- small shapes, all paths
SHAPES = {
    "one": [1],
    "odd_tails": [1, 2, 3, 5, 7, 8, 9, 15, 17, 31, 33],
    "small_pack_edges": [4095, 4096, 4097, 1, 4096],
    "chunk_edges": [32767, 32768, 32769, 65536 + 3],
    "several_tiles_ragged_tail": [5 * 32768 + 1234, 300001],
    "many_small": [int(x) for x in np.random.default_rng(3).integers(1, 300, 700)],
    "empty_mixed": [0, 17, 0, 40000, 0],
    # one work item each (finished in one pass inside the moments kernel) up
    # to the chunk size, several items above it; ragged tails throughout
    "mid_sizes": [4097, 4103, 8191, 8200, 16385, 24577, 32767, 32768, 32769, 65535, 65543,
                  100003, 131071, 131072],
}


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("grad_dtype", [torch.bfloat16, torch.float16])
def test_small_shapes_one_and_ten_steps(name, grad_dtype):
    S = 1024.0 if grad_dtype == torch.float16 else 1.0
    wl = custom(SHAPES[name], grad_dtype=grad_dtype, S=S, zero=[0], t0=3, clip=0.05)
    run_parity(wl, 10, check_steps=(1, 10))


def _random_workload(seed):
    """A seeded random small shard: 1 to 12 tensors whose sizes mix tiny,
    pack-edge, one-chunk and several-chunk lengths; random wd flags and zero-
    weight tensors; random hyperparameters, step number, clip (active or not),
    grad type and loss scale; warm or zero moments."""
    rng = np.random.default_rng(seed)
    pools = [(1, 40), (4090, 4100), (4101, 40000), (40001, 300000)]
    sizes = []
    for _ in range(int(rng.integers(1, 13))):
        lo, hi = pools[int(rng.integers(0, len(pools)))]
        sizes.append(int(rng.integers(lo, hi + 1)))
    n = len(sizes)
    fp16 = bool(rng.integers(0, 2))
    return W.Workload(
        f"random{seed}", "random", sizes, [int(x) for x in rng.integers(0, 2, n)],
        sorted(set(int(x) for x in rng.integers(0, n, int(rng.integers(0, 2))))),
        torch.float16 if fp16 else torch.bfloat16, t0=int(rng.integers(1, 3000)),
        lr=float(rng.choice([1e-4, 1e-3, 1e-2])),
        clip=float(rng.choice([0.0, 1e-3, 0.05, 1e3])),
        loss_scale=float(rng.choice([256.0, 4096.0, 65536.0])) if fp16 else 1.0,
        warm_state=bool(rng.integers(0, 2)), grad_kind="normal",
        grad_sigma=float(rng.choice([1e-4, 1e-3, 1e-2])), seed=1000 + seed,
        beta1=float(rng.choice([0.0, 0.8, 0.9, 0.95])),
        beta2=float(rng.choice([0.95, 0.99, 0.999, 0.9999])),
        eps=float(rng.choice([1e-8, 1e-6, 1e-4])),
        weight_decay=float(rng.choice([0.0, 0.01, 0.1])))


@pytest.mark.parametrize("seed", range(32))
def test_random_small_shards_match_the_oracle(seed):
    """Thirty-two seeded random shards (mixed sizes, flags, hyperparameters, grad
    types, clipping, loss scales), three steps each against the oracle."""
    wl = _random_workload(seed)
    run_parity(wl, 3, check_steps=(1, 3))


@pytest.mark.parametrize("seed", range(6))
def test_random_small_shards_with_async_steps_match_the_oracle(seed):
    """Six more seeded random shards, stepped asynchronously (the step number
    on the GPU) in two batches of 3 and 4 steps, with an inf or a NaN planted
    in one step: outcomes, step numbers and state against the oracle."""
    wl = _random_workload(100 + seed)
    wl.inject = {int(2 + seed % 4): "inf" if seed % 2 else "nan"}
    run_parity_async(wl, [3, 4])


def test_first_step_from_zero_state_with_zero_weight_tensors():
    wl = custom([1000, 50000, 3, 8, 70000], zero=[1, 2], warm=False, t0=1)
    run_parity(wl, 1, check_steps=(1,))


def test_clip_active_and_inactive():
    for clip in (1e-3, 1e6):
        run_parity(custom([9000, 123457], clip=clip, t0=20), 2, check_steps=(1, 2))


def test_heavy_tailed_grads():
    run_parity(custom([200000, 77, 4096], kind="student_t3", sigma=1e-4, clip=1.0, t0=500), 3,
               check_steps=(1, 3))


@pytest.mark.parametrize("grad_dtype,kind", [(torch.bfloat16, "inf"), (torch.bfloat16, "nan"),
                                             (torch.float16, "inf"), (torch.float16, "nan")])
def test_nonfinite_grad_skips_bit_exactly(grad_dtype, kind):
    S = 65536.0 if grad_dtype == torch.float16 else 1.0
    wl = custom([5, 40000, 300, 70001], grad_dtype=grad_dtype, S=S, inject={2: kind})
    st = W.make_state(wl, "cuda")
    gflat, gv = W.grad_buffer(wl, "cuda")
    opt = Lamb(st.w, st.m, st.v, st.w16, wl.wd_flags, grad_dtype=grad_dtype)
    W.fill_grads(wl, 1, gflat)
    assert opt.step(1e-3, 1, 0.0, S, grads=gv)[0] is False
    before = [x.clone() for x in (st.w_flat, st.m_flat, st.v_flat, st.w16_flat)]
    W.fill_grads(wl, 2, gflat)
    sk, gn = opt.step(1e-3, 2, 1.0, S)
    assert sk is True and gn == math.inf
    for a, b in zip(before, (st.w_flat, st.m_flat, st.v_flat, st.w16_flat)):
        assert torch.equal(a.view(torch.int8), b.view(torch.int8))
    # The next clean step proceeds normally (no stale flag left on the device).
    W.fill_grads(wl, 3, gflat)
    assert opt.step(1e-3, 2, 0.0, S)[0] is False
    opt.close()


@pytest.mark.parametrize("grad_dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("clip", [0.0, 1e-3])
def test_power_of_two_loss_scale_is_bit_exact(grad_dtype, clip):
    """Grads multiplied by 2^4 and stepped with S = 2^4 give the same state,
    bit for bit, as the grads stepped with S = 1, clipped or not (the scaling
    is exact in bf16 and fp16 at these magnitudes, and so is every product
    with the grad factor); the grad norm is the same number too."""
    k = 16.0
    wl = custom([5000, 70001, 300, 131072, 7], grad_dtype=grad_dtype, t0=3, clip=clip)
    _, gv = W.make_grads(wl, 1, "cuda")
    gv2 = [(g.float() * k).to(grad_dtype) for g in gv]
    for a, b in zip(gv, gv2):
        assert torch.equal((b.float() / k).to(grad_dtype).view(torch.int16), a.view(torch.int16))
    outs = []
    for grads, S in ((gv, 1.0), (gv2, k)):
        st = W.make_state(wl, "cuda")
        with Lamb(st.w, st.m, st.v, st.w16, wl.wd_flags, grad_dtype=grad_dtype) as opt:
            sk, gn = opt.step(wl.lr, wl.t0, clip, S, grads=grads)
            sk2, gn2 = opt.step(wl.lr, wl.t0 + 1, clip, S, grads=grads)
        assert not sk and not sk2
        outs.append(((gn, gn2), [x.clone() for x in (st.w_flat, st.m_flat, st.v_flat,
                                                        st.w16_flat)]))
    (n1, s1), (n2, s2) = outs
    assert n1 == n2
    if clip:
        assert n1[0] > clip  # the clip factor is in play
    for a, b in zip(s1, s2):
        assert torch.equal(a.view(torch.int8), b.view(torch.int8))


def test_rotating_grad_buffers_match_the_oracle():
    """Steps that take their grads from 5 different buffers in turn (more
    buffers than the handle's grad-pointer slots) still match the oracle."""
    from parity import HostState, compare_state, oracle_step
    wl = custom([70001, 17, 5000, 40000], t0=4, clip=0.02)
    st = W.make_state(wl, "cuda")
    hs = HostState(st, None)
    bufs = [W.grad_buffer(wl, "cuda") for _ in range(5)]
    with Lamb(st.w, st.m, st.v, st.w16, wl.wd_flags) as opt:
        t = wl.t0
        for k in range(1, 9):
            flat, views = bufs[(k * 3) % 5]
            W.fill_grads(wl, k, flat)
            g_host = [W.as_bits(x) for x in views]
            sk, gn = opt.step(wl.lr, t, wl.clip, wl.loss_scale, grads=views)
            osk, ogn, otr = oracle_step(wl, hs, g_host, t)
            assert not sk and not osk
            assert_close(np.array([gn]), np.array([ogn]), 1e-4, f"step {k} grad_norm")
            t += 1
        compare_state(st, hs, 1e-4, "after 8 steps", opt, otr)


def test_dynamic_loss_scaler_matches_the_oracle():
    """Device-resident dynamic loss scaling: starting at 2^24, fp16 grads of
    N(0, 1e-3) overflow, the step skips and the scale backs off; after 3 clean
    steps it grows again.  Skip flags, the scale sequence (bit-exact) and the
    state follow the oracle's step and its own scaler rule."""
    from parity import HostState, compare_state, oracle_step
    wl = custom([1 << 20, 300000, 4096, 77, 700000], grad_dtype=torch.float16, t0=1, warm=False,
                S=1.0)
    st = W.make_state(wl, "cuda")
    hs = HostState(st, None)
    flat, views = W.grad_buffer(wl, "cuda")
    cfg = dict(growth=2.0, backoff=0.5, growth_interval=3, min_scale=1.0, max_scale=2.0 ** 24)
    with Lamb(st.w, st.m, st.v, st.w16, wl.wd_flags, grad_dtype=torch.float16) as opt:
        opt.set_grads(views)
        opt.set_loss_scaler(init_scale=2.0 ** 24, growth_factor=cfg["growth"],
                            backoff_factor=cfg["backoff"], growth_interval=3, min_scale=1.0,
                            max_scale=2.0 ** 24)
        scale, good, t, skips = 2.0 ** 24, 0, wl.t0, []
        for k in range(1, 17):
            assert opt.next_loss_scale == scale
            W.fill_grads(wl, k, flat, loss_scale=scale)
            g_host = [W.as_bits(x) for x in views]
            sk, gn = opt.step(wl.lr, t, 0.0, 12345.0)  # the argument is ignored
            wl.loss_scale = scale
            osk, ogn, otr = oracle_step(wl, hs, g_host, t)
            assert int(sk) == osk and opt.loss_scale == scale
            skips.append(osk)
            if not osk:
                assert_close(np.array([gn]), np.array([ogn]), 1e-4, f"step {k} grad_norm")
                t += 1
            scale, good = oracle.loss_scale_update(scale, good, osk, **cfg)
            assert opt.next_loss_scale == scale, (k, opt.next_loss_scale, scale)
            if k in (4, 16):
                compare_state(st, hs, 1e-4, f"step {k}", opt, None)
        assert skips[0] == 1 and sum(skips) >= 3 and 0 in skips
        opt.clear_loss_scaler()
        W.fill_grads(wl, 17, flat, loss_scale=1024.0)
        assert opt.step(wl.lr, t, 0.0, 1024.0)[0] is False and opt.loss_scale == 1024.0


class _DeviceFloat:
    """One fp32 at a device address, for torch.as_tensor (CUDA array interface)."""

    def __init__(self, ptr):
        self.__cuda_array_interface__ = {"shape": (1,), "typestr": "<f4", "data": (ptr, False),
                                         "version": 3}


def test_async_steps_with_the_loss_scale_read_on_the_device():
    """A caller that never waits: fp16 grads are scaled on the GPU by the
    scale lamb_loss_scale_device exposes (in stream order, before each
    step_async), the scale backs off after overflows and grows after clean
    steps; the outcomes read later follow the oracle's scaler rule."""
    wl = custom([300000, 4096, 77], grad_dtype=torch.float16, t0=1, warm=False, S=1.0)
    st = W.make_state(wl, "cuda")
    cfg = dict(growth=2.0, backoff=0.5, growth_interval=2, min_scale=1.0, max_scale=2.0 ** 24)
    with Lamb(st.w, st.m, st.v, st.w16, wl.wd_flags, grad_dtype=torch.float16) as opt:
        opt.set_loss_scaler(init_scale=2.0 ** 22, growth_factor=2.0, backoff_factor=0.5,
                            growth_interval=2, min_scale=1.0, max_scale=2.0 ** 24)
        opt.set_step(1)
        scale_dev = torch.as_tensor(_DeviceFloat(opt.loss_scale_device_ptr()), device="cuda")
        raw = [W.make_grads(custom([300000, 4096, 77], grad_dtype=torch.float32, seed=50 + k,
                                   sigma=1e-3), 1, "cuda")[1] for k in range(8)]
        bufs, seqs = [], []
        for k in range(8):  # every step's grads = raw * (the scale on the GPU), no host wait
            g = [(x * scale_dev).to(torch.float16) for x in raw[k]]
            bufs.append(g)
            seqs.append(opt.step_async(wl.lr, 0.0, 1.0, grads=opt.prepare_grads(g)))
        outs = [opt.result(q) for q in seqs]
        scale, good = 2.0 ** 22, 0
        for k, (sk, gn, t) in enumerate(outs):
            g_host = [W.as_bits(x) for x in bufs[k]]
            bad = any(not np.isfinite(oracle.decode_grad(b, oracle.GRAD_FP16)).all()
                      for b in g_host)
            assert sk == bad, (k, sk, bad)
            scale, good = oracle.loss_scale_update(scale, good, int(bad), **cfg)
        torch.cuda.synchronize()
        assert scale_dev.item() == scale and opt.next_loss_scale == scale
        assert sum(o[0] for o in outs) >= 1 and not all(o[0] for o in outs)


def test_info_reports_the_kernels_a_step_runs():
    """Few waves of work items: one fused moments-and-apply kernel; many: two."""
    for sizes, fused in (([70001, 5000, 300], 1), ([1 << 27, 5000], 0)):
        wl = custom(sizes)
        st = W.make_state(wl, "cuda")
        with Lamb(st.w, st.m, st.v, st.w16, wl.wd_flags) as opt:
            info = opt.info()
            assert info["fused"] == fused and info["speculative"] == 0
            assert info["n_params"] == sum(sizes)
            one_pass_max = max(4096, info["chunk_elems"])  # packed, or a single work item
            assert info["one_pass_params"] == sum(n for n in sizes if n <= one_pass_max)
            _, gv = W.make_grads(wl, 1, "cuda")
            opt.set_timing(True)
            assert opt.step(wl.lr, 1, 0.0, 1.0, grads=gv)[0] is False
            ms = opt.kernel_times()
            assert ms[0] > 0 and ms[1] > 0 and (ms[2] == pytest.approx(0.0, abs=0.02) if fused
                                                 else ms[2] > 0)


@pytest.mark.parametrize("pinned", [True, False])
def test_snapshot_captures_the_state_between_steps(pinned):
    """A snapshot taken after step 2 holds exactly the state after step 2, even
    though step 3 is enqueued at once; and step 3 is bit-identical to a run
    without a snapshot."""
    # 128M elements: 1.5 GB of state, many milliseconds of copies, far longer
    # than the next step's grad-norm kernel, so a step that did not wait would
    # be caught rewriting m and v under the copy.
    wl = custom([70001, 17, 5000, 1 << 27, 0, 300], t0=4, clip=0.02)
    st = W.make_state(wl, "cuda")
    ref = st.clone()
    flat, views = W.grad_buffer(wl, "cuda")

    def run(state, snapshot):
        with Lamb(state.w, state.m, state.v, state.w16, wl.wd_flags) as opt:
            opt.set_grads(views)
            for k in (1, 2):
                W.fill_grads(wl, k, flat)
                opt.step(wl.lr, wl.t0 + k - 1, wl.clip)
            if not snapshot:
                W.fill_grads(wl, 3, flat)
                opt.step(wl.lr, wl.t0 + 2, wl.clip)
                return None
            expect = [x.clone() for x in (state.w_flat, state.m_flat, state.v_flat)]
            host = [[torch.empty(n, dtype=torch.float32, pin_memory=pinned) for n in wl.sizes]
                    for _ in range(3)]
            opt.snapshot_async(*host)
            W.fill_grads(wl, 3, flat)
            opt.step(wl.lr, wl.t0 + 2, wl.clip)
            opt.snapshot_wait()
            return expect, host

    run(ref, False)
    expect, host = run(st, True)
    for flat_exp, views_host in zip(expect, host):
        for o, n, h in zip(W.offsets(wl.sizes)[0], wl.sizes, views_host):
            assert torch.equal(flat_exp[o:o + n].cpu().view(torch.int32), h.view(torch.int32))
    for a, b in ((st.w_flat, ref.w_flat), (st.m_flat, ref.m_flat), (st.v_flat, ref.v_flat),
                 (st.w16_flat, ref.w16_flat)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_bf16_copies_land_in_one_allgather_bucket():
    """The bf16 copies can be written straight into a ZeRO-2 all-gather bucket:
    one contiguous bf16 buffer with the tensors back to back at 16-byte
    aligned offsets.  After two steps the bucket holds exactly bf16(w) of every
    tensor, and the padding between tensors is untouched."""
    wl = custom([1000, 8, 4096, 70001, 3, 130], t0=2, clip=0.05)
    st = W.make_state(wl, "cuda")
    offs, at = [], 0
    for n in wl.sizes:
        offs.append(at)
        at += (n + 7) // 8 * 8
    sentinel = 0x7FC1  # a NaN pattern no weight rounds to
    bucket = torch.full((at,), sentinel, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    views16 = [bucket[o:o + n] for o, n in zip(offs, wl.sizes)]
    flat, gv = W.grad_buffer(wl, "cuda")
    with Lamb(st.w, st.m, st.v, views16, wl.wd_flags) as opt:
        for k in (1, 2):
            W.fill_grads(wl, k, flat)
            opt.step(wl.lr, wl.t0 + k - 1, wl.clip, grads=gv)
    bits = bucket.view(torch.int16).cpu().numpy().view(np.uint16)
    covered = np.zeros(at, bool)
    for o, n, w in zip(offs, wl.sizes, st.w):
        assert np.array_equal(bits[o:o + n], oracle.bf16_rne(W.as_f32(w)))
        covered[o:o + n] = True
    assert np.all(bits[~covered] == sentinel)


@pytest.mark.parametrize("case", [
    dict(beta1=0.0, beta2=0.0),            # m = g', v = g'^2 exactly
    dict(lr=0.0),                          # w unchanged, m and v still updated
    dict(t0=10_000_000),                   # b^t underflows: no bias correction
    dict(weight_decay=0.0),                # the decay term vanishes everywhere
    dict(beta1=0.5, beta2=0.75, eps=0.5),  # large eps dominates sqrt(v)
    dict(sigma=3.0e4),                     # bf16 grads near 1e5 (large squares)
    dict(sigma=1e-15),                     # tiny grads: squares near 1e-30
    # bf16 grads whose squares leave fp32's normal range: below 2^-126
    # (summed in fp64 instead of fp32) and, with clipping, so large that 128
    # of their squares would overflow fp32
    dict(sigma=1e-21),
    dict(sigma=3e19),
])
def test_hyperparameter_corner_cases(case):
    case = dict(case)
    hp = {k: case.pop(k) for k in ("beta1", "beta2", "eps", "weight_decay", "lr") if k in case}
    wl = custom([70001, 4096, 17, 300000], t0=case.pop("t0", 3), sigma=case.pop("sigma", 1e-3),
                clip=1.0)
    for k, v in hp.items():
        setattr(wl, k, v)
    run_parity(wl, 3, check_steps=(1, 3))


def test_two_snapshots_on_two_streams_both_precede_the_next_step():
    wl = custom([1 << 26, 5000, 17], t0=2)
    st = W.make_state(wl, "cuda")
    _, gv = W.make_grads(wl, 1, "cuda")
    with Lamb(st.w, st.m, st.v, st.w16, wl.wd_flags) as opt:
        opt.step(wl.lr, wl.t0, grads=gv)
        expect = [x.clone() for x in (st.w_flat, st.m_flat, st.v_flat)]
        sets = [[[torch.empty(n, dtype=torch.float32, pin_memory=True) for n in wl.sizes]
                 for _ in range(3)] for _ in range(2)]
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        opt.snapshot_async(*sets[0], stream=s1)
        opt.snapshot_async(*sets[1], stream=s2)
        opt.step(wl.lr, wl.t0 + 1, grads=gv)  # must wait for both
        opt.snapshot_wait()
    offs = W.offsets(wl.sizes)[0]
    for host in sets:
        for flat_exp, views_host in zip(expect, host):
            for o, n, h in zip(offs, wl.sizes, views_host):
                assert torch.equal(flat_exp[o:o + n].cpu().view(torch.int32), h.view(torch.int32))


def test_handle_on_a_side_stream():
    """A handle bound to a non-default stream: grads produced on that stream
    are consumed in order, and the results match the oracle."""
    from parity import HostState, compare_state, oracle_step
    wl = custom([70001, 300, 4096], t0=6, clip=0.05)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        st = W.make_state(wl, "cuda")
        hs = HostState(st, None)
        flat, views = W.grad_buffer(wl, "cuda")
        opt = Lamb(st.w, st.m, st.v, st.w16, wl.wd_flags)
        assert opt.stream.cuda_stream == side.cuda_stream
        W.fill_grads(wl, 1, flat)  # enqueued on the side stream
        sk, gn = opt.step(wl.lr, wl.t0, wl.clip, grads=views)
    g_host = [W.as_bits(x) for x in views]
    osk, ogn, otr = oracle_step(wl, hs, g_host, wl.t0)
    assert not sk and not osk
    assert_close(np.array([gn]), np.array([ogn]), 1e-5, "grad_norm")
    compare_state(st, hs, 1e-5, "side stream", opt, otr)
    opt.close()


def test_twenty_thousand_tiny_tensors():
    """The pack path and the pointer-write kernel at scale: 20,000 tensors of
    1 to 64 elements (313 packs, 42 pointer-write launches)."""
    sizes = [int(x) for x in np.random.default_rng(9).integers(1, 65, 20000)]
    run_parity(custom(sizes, t0=2, clip=0.01), 3, check_steps=(1, 3))


def test_deterministic_across_runs():
    wl = custom([300001, 17, 5000, 123])
    outs = []
    for _ in range(2):
        st = W.make_state(wl, "cuda")
        _, gv = W.make_grads(wl, 1, "cuda")
        with Lamb(st.w, st.m, st.v, st.w16, wl.wd_flags) as opt:
            r = opt.step(1e-3, 5, 0.1, 1.0, grads=gv)
            outs.append((r, st.w_flat.clone(), st.m_flat.clone(), opt.trust().copy()))
    assert outs[0][0] == outs[1][0]
    assert torch.equal(outs[0][1], outs[1][1]) and torch.equal(outs[0][2], outs[1][2])
    assert np.array_equal(outs[0][3], outs[1][3])


def test_concurrent_handles_on_their_own_streams_match_solo_runs():
    """Three handles on three streams -- a fused shard with clipping, a
    three-kernel one, and a speculative one -- step 8 times each with their
    steps interleaved and nothing waiting in between, so that their
    persistent grids share the GPU.  Every kernel's wait is on work that a
    running CTA holds, so none depends on its grid being resident at once;
    and every sum is taken in a fixed order.  So each handle ends bit for bit
    where it ends when it runs alone."""
    cases = [(custom([1 << 20, 70001, 300, 5000], seed=41, t0=2, clip=0.05), False),
             (custom([130 << 20, 4096, 17], seed=42, t0=5, clip=0.0), False),
             (custom([3 << 20, 12288, 9], seed=43, t0=9, clip=0.0, inject={3: "inf"}), True)]

    def run(concurrent):
        hs = []
        for wl, spec in cases:
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                st = W.make_state(wl, "cuda")
                flat, views = W.grad_buffer(wl, "cuda")
            opt = Lamb(st.w, st.m, st.v, st.w16, wl.wd_flags, stream=stream)
            opt.set_grads(views)
            if spec:
                opt.set_speculative(st.views(torch.empty_like(st.m_flat)),
                                    st.views(torch.empty_like(st.v_flat)))
            opt.set_step(wl.t0)
            hs.append([wl, st, flat, opt, stream, []])
        torch.cuda.synchronize()
        order = ([(k, h) for k in range(1, 9) for h in hs] if concurrent
                 else [(k, h) for h in hs for k in range(1, 9)])
        for k, (wl, st, flat, opt, stream, seqs) in order:
            with torch.cuda.stream(stream):
                W.fill_grads(wl, k, flat)
            seqs.append(opt.step_async(wl.lr, wl.clip, wl.loss_scale))
        torch.cuda.synchronize()
        out = []
        for wl, st, flat, opt, stream, seqs in hs:
            results = [opt.result(q) for q in seqs]
            m, v = opt.state_buffers()
            out.append((results, st.w_flat.clone(), torch.cat([x.flatten() for x in m]),
                        torch.cat([x.flatten() for x in v]), st.w16_flat.clone(),
                        opt.trust().copy(), opt.info()))
            opt.close()
        return out

    solo, together = run(False), run(True)
    assert [o[6]["fused"] for o in solo] == [1, 0, 1] and solo[2][6]["speculative"] == 1
    for a, b in zip(solo, together):
        assert a[0] == b[0]  # skip flags, grad norms and step numbers
        for x, y in zip(a[1:5], b[1:5]):
            assert torch.equal(x, y)
        assert np.array_equal(a[5], b[5])
    assert [r[0] for r in solo[2][0]].count(True) == 1  # the planted inf


def test_empty_handle_and_errors():
    with Lamb([], [], [], [], []) as opt:
        assert opt.step(1e-3, 1, grads=[]) == (False, 0.0)
    st = W.make_state(custom([64]), "cuda")
    _, gv = W.make_grads(custom([64]), 1, "cuda")
    with Lamb(st.w, st.m, st.v, st.w16, [1]) as opt:
        with pytest.raises(LambError):
            opt.step(1e-3, 0, grads=gv)
        with pytest.raises(LambError):
            opt.step(1e-3, 1, loss_scale=0.0, grads=gv)
        with pytest.raises(TypeError):
            opt.step(1e-3, 1, grads=[gv[0].float()])
        raw = torch.zeros(80, dtype=torch.bfloat16, device="cuda")
        with pytest.raises(LambError) as e:
            opt.step(1e-3, 1, grads=[raw[1:65]])
        assert e.value.code == -2
    w = torch.zeros(80, device="cuda")
    with pytest.raises(LambError) as e:
        Lamb([w[1:65]], [w[:64]], [w[:64]], [torch.zeros(64, dtype=torch.bfloat16, device="cuda")],
             [1])
    assert e.value.code == -2


def test_scaler_snapshot_and_monitor_argument_errors():
    import ctypes
    from optimizer_step_gb300 import _lib
    wl = custom([64, 5000])
    st = W.make_state(wl, "cuda")
    _, gv = W.make_grads(wl, 1, "cuda")
    with Lamb(st.w, st.m, st.v, st.w16, wl.wd_flags) as opt:
        with pytest.raises(LambError):
            opt.kernel_times()  # monitor off
        opt.set_timing(True)
        with pytest.raises(LambError):
            opt.kernel_times()  # no step timed yet
        opt.step(1e-3, 1, grads=gv)
        assert all(x > 0 for x in opt.kernel_times())
        for bad in (dict(init_scale=0.0), dict(init_scale=float("inf")), dict(growth_factor=0.5),
                    dict(backoff_factor=0.0), dict(backoff_factor=1.5), dict(growth_interval=0),
                    dict(min_scale=2.0 ** 20, init_scale=2.0 ** 10),
                    dict(max_scale=2.0, init_scale=4.0)):
            with pytest.raises(LambError) as e:
                opt.set_loss_scaler(**bad)
            assert e.value.code == _lib.LAMB_ERR_INVALID
        with pytest.raises(ValueError):
            opt.snapshot_async([torch.empty(3)], [torch.empty(3)], [torch.empty(3)])
        lib = _lib.load()
        null = (ctypes.c_void_p * 2)(None, None)
        assert lib.lamb_snapshot_async(opt._h, null, null, null, None) == _lib.LAMB_ERR_INVALID
        opt.snapshot_wait()  # nothing pending: returns at once


# ------------------------------------------------------- the named configs
def test_config_tiny_one_and_ten_steps():
    log = run_parity(W.tiny(), 10, check_steps=(1, 10))
    assert log["skipped"] == [0] * 10


def test_config_fp16_twenty_steps_with_injected_overflow():
    wl = W.fp16_24()
    first_block = list(range(6))
    site7, site15 = W.injection_site(wl, 7), W.injection_site(wl, 15)
    subset = sorted(set(first_block + [site7[0], site15[0], len(wl.sizes) - 1]))
    log = run_parity(wl, 20, check_steps=(1, 6, 7, 8, 10, 15, 16, 20), subset=subset)
    want = [1 if k in (7, 15) else 0 for k in range(1, 21)]
    assert log["skipped"] == want


def test_async_steps_fp16_twenty_with_injected_overflow():
    """Twenty fp16 steps of the fp16 config's tensor mix (every tensor cut to
    70,001 elements), enqueued asynchronously in phases of 6, 4 and 10 steps:
    steps 7 and 15 carry an inf / a NaN, so the GPU's step counter must stay
    put there.  Every outcome and the state after each phase match the oracle."""
    wl = W.scaled(W.fp16_24(), 70001)
    log = run_parity_async(wl, [6, 4, 10])
    assert log["skipped"] == [1 if k in (7, 15) else 0 for k in range(1, 21)]
    assert log["t"][-1] == 18  # t started at 1 and two steps were skipped


def test_step_result_without_waiting_and_sequence_bounds():
    """lamb_step_result with wait = 0 answers 'not ready' while the step is
    still queued behind other work on the handle's stream (a bounded sleep
    kernel), then the outcome once it has run; sequence numbers not yet
    given out, and those older than the last 64 steps, are refused."""
    wl = custom([1 << 20, 300], t0=2)
    st = W.make_state(wl, "cuda")
    _, gv = W.make_grads(wl, 1, "cuda")
    with Lamb(st.w, st.m, st.v, st.w16, wl.wd_flags) as opt:
        opt.set_grads(gv)
        opt.set_step(wl.t0)
        torch.cuda.synchronize()
        with torch.cuda.stream(opt.stream):
            torch.cuda._sleep(200_000_000)  # about 0.1 s of GPU time, then it ends
        q = opt.step_async(wl.lr)
        assert opt.result(q, wait=False) is None
        done = opt.result(q)
        assert done[0] is False and done[2] == wl.t0 and math.isfinite(done[1])
        assert opt.result(q, wait=False) == done
        with pytest.raises(LambError, match="no step"):
            opt.result(q + 1)
        seqs = [opt.step_async(wl.lr) for _ in range(70)]
        assert opt.result(seqs[-1])[2] == wl.t0 + 70
        with pytest.raises(LambError, match="only the last 64"):
            opt.result(q)
        assert opt.result(seqs[-64])[2] == wl.t0 + 7


def test_async_and_synchronous_steps_mix():
    """lamb_step with an explicit t leaves the GPU counter at t+1 (clean) or
    t (skipped), so asynchronous steps continue from there."""
    wl = custom([5000, 70001, 17], t0=4, clip=0.5, inject={2: "inf"})
    st = W.make_state(wl, "cuda")
    opt = Lamb(st.w, st.m, st.v, st.w16, wl.wd_flags)
    try:
        _, gv = W.make_grads(wl, 1, "cuda")
        assert opt.step(wl.lr, 9, wl.clip, 1.0, grads=gv)[0] is False
        q = opt.step_async(wl.lr, wl.clip, 1.0)
        assert opt.result(q)[2] == 10
        _, gbad = W.make_grads(wl, 2, "cuda")
        assert opt.step(wl.lr, 11, wl.clip, 1.0, grads=gbad)[0] is True
        q = opt.step_async(wl.lr, wl.clip, 1.0, grads=gv)
        assert opt.result(q)[2] == 11 and opt.result(q)[0] is False
        opt.set_step(3)
        q = opt.step_async(wl.lr, wl.clip, 1.0)
        assert opt.result(q)[2] == 3
        # Only the last 64 outcomes are kept; unknown sequence numbers are errors.
        for _ in range(64):
            last = opt.step_async(wl.lr, wl.clip, 1.0)
        opt.result(last)
        with pytest.raises(LambError):
            opt.result(q)
        with pytest.raises(LambError):
            opt.result(last + 1)
    finally:
        opt.close()


def test_config_ragged_full_step_then_ten_steps():
    wl = W.ragged()
    run_parity(wl, 1, check_steps=(1,))
    rng = np.random.default_rng(0)
    subset = sorted(set(wl.zero_w) | set(int(i) for i in rng.choice(len(wl.sizes), 150, False))
                    | {int(np.argmax(wl.sizes))})
    run_parity(wl, 10, check_steps=(1, 10), subset=subset)


def _large_one_step(wl, tensors):
    """One step of a large config; every tensor in ``tensors`` is checked in
    full against the oracle, one at a time (pre-step copies kept on the GPU)."""
    st = W.make_state(wl, "cuda")
    gflat, gv = W.make_grads(wl, 1, "cuda")
    pre = {i: (st.w[i].clone(), st.m[i].clone(), st.v[i].clone()) for i in tensors}
    with Lamb(st.w, st.m, st.v, st.w16, wl.wd_flags, grad_dtype=wl.grad_dtype) as opt:
        sk, gn = opt.step(wl.lr, wl.t0, wl.clip, wl.loss_scale, grads=gv)
        trust = opt.trust()
    assert sk is False
    g_host = [W.as_bits(x) for x in gv]
    for i in tensors:
        mask = np.zeros(len(wl.sizes), np.uint8)
        mask[i] = 1
        n = len(wl.sizes)
        w = [None] * n
        m = [None] * n
        v = [None] * n
        w16 = [None] * n
        w[i], m[i], v[i] = (W.as_f32(x).copy() for x in pre[i])
        w16[i] = np.zeros(wl.sizes[i], np.uint16)
        del pre[i]
        osk, ogn, otr = oracle.lamb_step(
            w, m, v, w16, g_host, wl.wd_flags, grad_dtype=oracle.GRAD_BF16,
            beta1=f32(wl.beta1), beta2=f32(wl.beta2), eps=f32(wl.eps),
            weight_decay=f32(wl.weight_decay), lr=f32(wl.lr), t=wl.t0, clip=f32(wl.clip),
            loss_scale=f32(wl.loss_scale), update_mask=mask, want_trust=True)
        assert osk == 0
        assert_close(np.array([gn]), np.array([ogn]), 1e-5, "grad_norm")
        assert_close(trust[i:i + 1], otr[i:i + 1], 1e-5, f"trust[{i}]")
        w_gpu = W.as_f32(st.w[i])
        assert_close(w_gpu, w[i], 1e-5, f"w[{i}]")
        assert_close(W.as_f32(st.m[i]), m[i], 1e-5, f"m[{i}]")
        assert_close(W.as_f32(st.v[i]), v[i], 1e-5, f"v[{i}]")
        check_bf16_copy(W.as_bits(st.w16[i]), w_gpu, w16[i], w[i], 1e-5, f"w16[{i}]")
        del w, m, v, w16, w_gpu


def test_config_175b_shard_full_step():
    wl = W.shard175b()
    _large_one_step(wl, list(range(len(wl.sizes))))


def test_config_175b_shard_ten_steps_subset():
    wl = W.shard175b()
    run_parity(wl, 10, check_steps=(1, 10), subset=[1, 4, 5])


def test_tensor_larger_than_2_to_the_31_elements():
    """64-bit element offsets: one tensor of 2^31 + 5 elements (plus a small one),
    checked in full against the oracle after one step."""
    wl = custom([(1 << 31) + 5, 1000], t0=7, clip=1.0, sigma=1e-4)
    _large_one_step(wl, [0, 1])


def test_config_7b_one_step_and_ten_steps_subset():
    wl = W.llama7b()
    n = len(wl.sizes)
    _large_one_step(wl, [0, 1, 2, 3, 4, 5, 6, n - 1])
    run_parity(wl, 10, check_steps=(1, 10), subset=[0, 2, 5, 6, n - 1])
