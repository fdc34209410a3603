"""The split step for a data-parallel (ZeRO-2) group whose shard boundaries
cut tensors, against the oracle stepping the whole, unsplit shard.

ZeRO-2 gives each data-parallel rank a contiguous slice of the flattened
optimizer state (MegaScale guided-reading digest, section 3, "Data parallelism
(ZeRO-2 style)"; the digest's "Terms" entry for ZeRO-2), so a rank's first and
last tensors can be pieces of tensors other ranks also hold.  Each rank runs
lamb_split_norms, the group sums the grad-norm partials, each runs
lamb_split_moments, the group sums the shared tensors' {sum w^2, sum r^2}, and
each runs lamb_split_apply.  Whatever the cut, the concatenated result must
match one step of the whole shard.

Here the ranks are handles on one GPU (their kernels never wait on one
another; the sums go through host memory), and in the second test two
processes on the same GPU that sum with a gloo all-reduce.  Runs of more than
one GPU are not measured.
"""
import math
import os
import socket

import numpy as np
import pytest
import torch

import workloads as W
from optimizer_step_gb300 import Lamb, LambError

from parity import HostState, assert_close, compare_state, oracle_step, rtol_for

pytestmark = pytest.mark.gpu

SIZES = [5000, 70001, 300, 200003, 17, 4096, 40000, 9]


def _workload(inject=None, clip=0.02, grad_dtype=torch.bfloat16, S=1.0):
    return W.Workload("split", "split", list(SIZES), [1, 1, 0, 1, 0, 0, 1, 0], [2],
                      grad_dtype, t0=5, lr=1e-3, clip=clip, loss_scale=S, warm_state=True,
                      grad_kind="normal", grad_sigma=1e-3, seed=77, inject=dict(inject or {}))


def _rank_handle(wl, st, gviews, mine, slots, n_slots, device):
    xn = torch.zeros(2, dtype=torch.float64, device=device)
    xt = torch.zeros(max(2, 2 * n_slots), dtype=torch.float64, device=device)
    take = lambda lst: [lst[i][b:e] for i, b, e in mine]
    opt = Lamb(take(st.w), take(st.m), take(st.v), take(st.w16),
               [wl.wd_flags[i] for i, _, _ in mine], grad_dtype=wl.grad_dtype,
               exchange_slots=slots, norm_exchange=xn, tensor_exchange=xt)
    return opt, xn, xt, opt.prepare_grads(take(gviews))


def _split_step(ranks, wl, t, sum_fn):
    """One split step over every rank; sum_fn sums a list of same-shaped
    tensors (one per rank) and writes the sum back into each."""
    for opt, xn, xt, g in ranks:
        opt.split_norms(g, wl.loss_scale)
    torch.cuda.synchronize()
    sum_fn([r[1] for r in ranks])
    for opt, xn, xt, g in ranks:
        xt.zero_()
        opt.split_moments(wl.lr, wl.clip, t)
    torch.cuda.synchronize()
    sum_fn([r[2] for r in ranks])
    return [opt.split_apply() for opt, _, _, _ in ranks]


def _host_sum(bufs):
    total = sum(b.double().cpu() for b in bufs)
    for b in bufs:
        b.copy_(total)


@pytest.mark.parametrize("n_ranks", [1, 2, 3, 5])
def test_split_step_matches_the_whole_shard(n_ranks):
    """n_ranks handles over the pieces of one shard, three steps (the second
    carries an inf), t from the host then from the GPU's counter."""
    wl = _workload(inject={2: "inf"})
    st = W.make_state(wl, "cuda")
    hs = HostState(st, None)
    gflat, gviews = W.grad_buffer(wl, "cuda")
    pieces, slots = W.zero2_pieces(wl.sizes, n_ranks)
    n_slots = 1 + max([k for sl in slots for k in sl] + [-1])
    ranks = [_rank_handle(wl, st, gviews, mine, sl, n_slots, "cuda")
             for mine, sl in zip(pieces, slots)]
    # Shards this small run the fused moments-and-apply kernel in the split
    # step too (whole tensors applied in lamb_split_moments).
    assert all(r[0].info()["fused"] == 1 for r in ranks)
    try:
        t = wl.t0
        for k in (1, 2, 3):
            W.fill_grads(wl, k, gflat)
            torch.cuda.synchronize()
            g_host = [W.as_bits(x) for x in gviews]
            seqs = _split_step(ranks, wl, t if k == 1 else 0, _host_sum)
            if k == 1:
                for opt, _, _, _ in ranks:
                    opt.set_step(t + 1)  # later steps take the GPU's counter
            outs = [opt.result(q) for (opt, _, _, _), q in zip(ranks, seqs)]
            osk, ogn, otrust = oracle_step(wl, hs, g_host, t)
            for sk, gn, t_used in outs:
                assert int(sk) == osk and t_used == t
                if osk:
                    assert gn == math.inf
                else:
                    assert_close(np.array([gn]), np.array([ogn]), 1e-5, f"step {k} grad_norm")
            if not osk:
                t += 1
            compare_state(st, hs, rtol_for(k), f"{n_ranks} ranks, step {k}")
            if not osk:
                for (opt, _, _, _), mine in zip(ranks, pieces):
                    tr = opt.trust()
                    want = np.array([otrust[i] for i, _, _ in mine])
                    assert_close(tr, want, 1e-5, f"{n_ranks} ranks, step {k} trust")
        assert [int(o[0]) for o in outs] == [0] * n_ranks
    finally:
        for opt, _, _, _ in ranks:
            opt.close()


@pytest.mark.parametrize("seed", range(8))
def test_random_shards_cut_over_random_groups(seed):
    """Seeded random tensor lists cut over 2 to 6 ranks (shared tensors
    wherever the cuts fall; fp16 or bf16 grads; clipping active or not), two
    split steps each, against the oracle stepping the unsplit shard."""
    rng = np.random.default_rng(500 + seed)
    sizes = [int(rng.choice([rng.integers(1, 50), rng.integers(4090, 4110),
                             rng.integers(5000, 90000), rng.integers(90000, 400000)]))
             for _ in range(int(rng.integers(2, 12)))]
    fp16 = bool(rng.integers(0, 2))
    wl = W.Workload(f"split-random{seed}", "split-random", sizes,
                    [int(x) for x in rng.integers(0, 2, len(sizes))], [],
                    torch.float16 if fp16 else torch.bfloat16, t0=int(rng.integers(1, 500)),
                    lr=1e-3, clip=float(rng.choice([0.0, 0.01, 100.0])),
                    loss_scale=1024.0 if fp16 else 1.0, warm_state=True, grad_kind="normal",
                    grad_sigma=1e-3, seed=900 + seed)
    n_ranks = int(rng.integers(2, 7))
    st = W.make_state(wl, "cuda")
    hs = HostState(st, None)
    gflat, gviews = W.grad_buffer(wl, "cuda")
    pieces, slots = W.zero2_pieces(wl.sizes, n_ranks)
    n_slots = 1 + max([k for sl in slots for k in sl] + [-1])
    ranks = [_rank_handle(wl, st, gviews, mine, sl, n_slots, "cuda")
             for mine, sl in zip(pieces, slots) if mine]
    try:
        for k in (1, 2):
            W.fill_grads(wl, k, gflat)
            torch.cuda.synchronize()
            g_host = [W.as_bits(x) for x in gviews]
            seqs = _split_step(ranks, wl, wl.t0 + k - 1, _host_sum)
            osk, ogn, otrust = oracle_step(wl, hs, g_host, wl.t0 + k - 1)
            assert osk == 0
            for (opt, _, _, _), q in zip(ranks, seqs):
                sk, gn, _ = opt.result(q)
                assert sk is False
                assert_close(np.array([gn]), np.array([ogn]), 1e-5, f"step {k} grad_norm")
            compare_state(st, hs, rtol_for(k), f"seed {seed}, {n_ranks} ranks, step {k}")
    finally:
        for opt, _, _, _ in ranks:
            opt.close()


def test_split_step_on_shards_of_many_waves():
    """Two ranks of about 125 M params each: shards of more than 8 waves of
    work items, so the split step runs the separate moments and apply kernels.
    One step with clipping active, against the oracle on the unsplit shard."""
    sizes = [100_000_000, 90_000_003, 60_000_000, 4097, 300, 17]
    wl = W.Workload("split-large", "split-large", sizes, [1, 1, 1, 1, 0, 0], [], torch.bfloat16,
                    t0=7, lr=1e-3, clip=0.05, loss_scale=1.0, warm_state=True,
                    grad_kind="normal", grad_sigma=1e-3, seed=79)
    st = W.make_state(wl, "cuda")
    hs = HostState(st, None)
    gflat, gviews = W.make_grads(wl, 1, "cuda")
    pieces, slots = W.zero2_pieces(wl.sizes, 2)
    n_slots = 1 + max([k for sl in slots for k in sl] + [-1])
    assert n_slots == 1
    ranks = [_rank_handle(wl, st, gviews, mine, sl, n_slots, "cuda")
             for mine, sl in zip(pieces, slots)]
    assert all(r[0].info()["fused"] == 0 for r in ranks)
    try:
        g_host = [W.as_bits(x) for x in gviews]
        seqs = _split_step(ranks, wl, wl.t0, _host_sum)
        osk, ogn, otrust = oracle_step(wl, hs, g_host, wl.t0)
        assert osk == 0 and ogn > wl.clip
        for (opt, _, _, _), q in zip(ranks, seqs):
            sk, gn, _ = opt.result(q)
            assert sk is False
            assert_close(np.array([gn]), np.array([ogn]), 1e-5, "grad_norm")
        compare_state(st, hs, 1e-5, "two ranks of many waves")
        for (opt, _, _, _), mine in zip(ranks, pieces):
            want = np.array([otrust[i] for i, _, _ in mine])
            assert_close(opt.trust(), want, 1e-5, "trust")
    finally:
        for opt, _, _, _ in ranks:
            opt.close()


def test_split_step_with_a_tensor_over_three_ranks_and_fp16_scale():
    """One tensor cut across three ranks (the middle rank holds only a piece of
    it), fp16 grads with a loss scale, clipping active."""
    wl = W.Workload("split3", "split3", [3000, 300000, 5000], [1, 1, 0], [], torch.float16,
                    t0=3, lr=1e-3, clip=1e-4, loss_scale=1024.0, warm_state=True,
                    grad_kind="normal", grad_sigma=1e-3, seed=78)
    st = W.make_state(wl, "cuda")
    hs = HostState(st, None)
    gflat, gviews = W.make_grads(wl, 1, "cuda")
    pieces, slots = W.zero2_pieces(wl.sizes, 4)
    assert pieces[1] == [(1, pieces[1][0][1], pieces[1][0][2])] and slots[1] == [0]
    n_slots = 1
    ranks = [_rank_handle(wl, st, gviews, mine, sl, n_slots, "cuda")
             for mine, sl in zip(pieces, slots)]
    try:
        g_host = [W.as_bits(x) for x in gviews]
        seqs = _split_step(ranks, wl, wl.t0, _host_sum)
        osk, ogn, otrust = oracle_step(wl, hs, g_host, wl.t0)
        assert osk == 0 and ogn * 1.0 > wl.clip  # clipping is active
        for (opt, _, _, _), q in zip(ranks, seqs):
            sk, gn, _ = opt.result(q)
            assert sk is False
            assert_close(np.array([gn]), np.array([ogn]), 1e-5, "grad_norm")
        compare_state(st, hs, 1e-5, "three-rank tensor")
    finally:
        for opt, _, _, _ in ranks:
            opt.close()


def test_split_steps_with_a_dynamic_loss_scaler_follow_an_ordinary_handle():
    """Two ranks, fp16 grads, each rank's handle with the same device-resident
    loss scaler starting at 2^24 (the first steps overflow), clipping off.
    Every rank takes the group's skip decision, so both ranks and an ordinary
    handle over the whole shard give the same skip flags and scale sequence;
    tensors no rank shares come out bit for bit equal to the ordinary
    handle's, and the shared one within 1e-6 (its norms are summed in another
    order)."""
    wl = _workload(clip=0.0, grad_dtype=torch.float16)
    st = W.make_state(wl, "cuda")
    ref = W.make_state(wl, "cuda")
    gflat, gviews = W.grad_buffer(wl, "cuda")
    pieces, slots = W.zero2_pieces(wl.sizes, 2)
    n_slots = 1 + max([k for sl in slots for k in sl] + [-1])
    ranks = [_rank_handle(wl, st, gviews, mine, sl, n_slots, "cuda")
             for mine, sl in zip(pieces, slots)]
    whole = Lamb(ref.w, ref.m, ref.v, ref.w16, wl.wd_flags, grad_dtype=torch.float16)
    cfg = dict(init_scale=2.0 ** 24, growth_factor=2.0, backoff_factor=0.5, growth_interval=3,
               min_scale=1.0, max_scale=2.0 ** 24)
    shared = {i for mine, sl in zip(pieces, slots) for (i, _, _), k in zip(mine, sl) if k >= 0}
    try:
        for opt, _, _, _ in ranks:
            opt.set_loss_scaler(**cfg)
        whole.set_loss_scaler(**cfg)
        skips = []
        for k in range(1, 11):
            scale = whole.next_loss_scale
            W.fill_grads(wl, k, gflat, loss_scale=scale)
            torch.cuda.synchronize()
            seqs = _split_step(ranks, wl, wl.t0 + k, _host_sum)
            sk_w, _ = whole.step(wl.lr, wl.t0 + k, 0.0, 1.0, grads=gviews)
            for (opt, _, _, _), q in zip(ranks, seqs):
                sk, _, _ = opt.result(q)
                assert sk == sk_w and opt.next_loss_scale == whole.next_loss_scale
            skips.append(int(sk_w))
            torch.cuda.synchronize()
            for i in range(len(wl.sizes)):
                for name in ("w", "m", "v", "w16"):
                    got, want = getattr(st, name)[i], getattr(ref, name)[i]
                    if i in shared and name in ("w", "w16"):  # the trust ratio differs
                        rtol = 1e-6 if name == "w" else 2.0 ** -7  # w16: one bf16 ulp
                        assert torch.allclose(got.float(), want.float(), rtol=rtol, atol=0), \
                            (k, i, name)
                    else:
                        assert torch.equal(got, want), (k, i, name)
        assert skips[0] == 1 and 0 in skips and shared
    finally:
        for opt, _, _, _ in ranks:
            opt.close()
        whole.close()


def test_split_step_of_a_group_of_one_equals_lamb_step():
    """The binding's whole split step (Lamb.split_step) on a group of one,
    with no exchange at all, gives lamb_step's result bit for bit, three
    steps in a row with clipping active."""
    wl = _workload(clip=0.02)
    a, b = W.make_state(wl, "cuda"), W.make_state(wl, "cuda")
    gflat, gviews = W.grad_buffer(wl, "cuda")
    whole = [(i, 0, n) for i, n in enumerate(wl.sizes)]
    opt_s, _, _, g = _rank_handle(wl, a, gviews, whole, [-1] * len(whole), 0, "cuda")
    opt_o = Lamb(b.w, b.m, b.v, b.w16, wl.wd_flags)
    try:
        for k in range(1, 4):
            W.fill_grads(wl, k, gflat)
            q = opt_s.split_step(wl.lr, wl.clip, wl.t0 + k, grads=g, loss_scale=1.0)
            sk, gn = opt_o.step(wl.lr, wl.t0 + k, wl.clip, 1.0, grads=gviews)
            assert opt_s.result(q)[:2] == (sk, gn)
            torch.cuda.synchronize()
            for x, y in ((a.w_flat, b.w_flat), (a.m_flat, b.m_flat), (a.v_flat, b.v_flat),
                         (a.w16_flat, b.w16_flat)):
                assert torch.equal(x, y)
    finally:
        opt_s.close()
        opt_o.close()


def test_ordinary_steps_are_refused_while_a_tensor_is_shared():
    """A shared tensor's trust ratio needs the group's sums, so lamb_step and
    lamb_step_async refuse such a shard (before enqueueing anything); a shard
    of the same kind whose tensors are all whole still takes them."""
    wl = _workload()
    st = W.make_state(wl, "cuda")
    _, gviews = W.make_grads(wl, 1, "cuda")
    pieces, slots = W.zero2_pieces(wl.sizes, 2)
    opt, _, _, g = _rank_handle(wl, st, gviews, pieces[0], slots[0], 1, "cuda")
    before = [x.clone() for x in (st.w_flat, st.m_flat, st.v_flat)]
    try:
        assert any(k >= 0 for k in slots[0])
        with pytest.raises(LambError, match="shared with other ranks"):
            opt.step(wl.lr, wl.t0, wl.clip, wl.loss_scale, grads=g)
        with pytest.raises(LambError, match="shared with other ranks"):
            opt.step_async(wl.lr, wl.clip, grads=g)
    finally:
        opt.close()
    torch.cuda.synchronize()
    for a, b in zip(before, (st.w_flat, st.m_flat, st.v_flat)):
        assert torch.equal(a, b)
    whole = [(i, 0, n) for i, n in enumerate(wl.sizes)]
    opt, _, _, g = _rank_handle(wl, st, gviews, whole, [-1] * len(whole), 0, "cuda")
    try:
        assert opt.step(wl.lr, wl.t0, wl.clip, wl.loss_scale, grads=g)[0] is False
    finally:
        opt.close()


def test_calls_between_the_phases_are_refused():
    """Between lamb_split_norms and lamb_split_apply the handle refuses
    another step, a new step number or loss scaler, speculative mode and a
    snapshot (the state is half-updated there); the split step then finishes
    normally."""
    wl = _workload(clip=0.0)
    st = W.make_state(wl, "cuda")
    _, gviews = W.make_grads(wl, 1, "cuda")
    pieces, slots = W.zero2_pieces(wl.sizes, 1)
    opt, xn, xt, g = _rank_handle(wl, st, gviews, pieces[0], slots[0], 1, "cuda")
    host = [torch.empty(n, dtype=torch.float32).pin_memory() for n in wl.sizes]
    m2 = [torch.zeros_like(x) for x in st.m]
    v2 = [torch.zeros_like(x) for x in st.v]
    refused = {
        "step": lambda: opt.step(wl.lr, wl.t0, 0.0, 1.0, grads=g),
        "step_async": lambda: opt.step_async(wl.lr, 0.0, grads=g),
        "set_step": lambda: opt.set_step(7),
        "set_loss_scaler": lambda: opt.set_loss_scaler(),
        "set_speculative": lambda: opt.set_speculative(m2, v2),
        "snapshot_async": lambda: opt.snapshot_async(host, host, host),
    }
    try:
        for phase in ("norms", "moments"):
            if phase == "norms":
                opt.split_norms(g, wl.loss_scale)
            else:
                opt.split_moments(wl.lr, 0.0, wl.t0)
            for name, call in refused.items():
                with pytest.raises(LambError, match="split step"):
                    call()
        seq = opt.split_apply()
        sk, gn, t = opt.result(seq)
        assert sk is False and math.isfinite(gn) and t == wl.t0
    finally:
        opt.close()


# ------------------------------------------------ two processes, gloo sums
def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, result_dir):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        torch.cuda.set_device(0)
        wl = _workload(inject={2: "nan"})
        st = W.make_state(wl, "cuda")  # every rank builds the same seeded shard
        hs = HostState(st, None)
        gflat, gviews = W.grad_buffer(wl, "cuda")
        pieces, slots = W.zero2_pieces(wl.sizes, world)
        n_slots = 1 + max([k for sl in slots for k in sl] + [-1])
        ranks = [_rank_handle(wl, st, gviews, pieces[rank], slots[rank], n_slots, "cuda")]

        def gloo_sum(bufs):
            (b,) = bufs
            h = b.cpu()
            dist.all_reduce(h)
            b.copy_(h)

        t = wl.t0
        skipped = []
        opt = ranks[0][0]
        for k in (1, 2, 3):
            W.fill_grads(wl, k, gflat)
            torch.cuda.synchronize()
            g_host = [W.as_bits(x) for x in gviews]
            # the binding's whole split step, with the group's sums by gloo
            q = opt.split_step(wl.lr, wl.clip, t, grads=ranks[0][3], loss_scale=wl.loss_scale,
                               all_reduce=lambda b: gloo_sum([b]))
            sk, gn, _ = ranks[0][0].result(q)
            osk, ogn, _ = oracle_step(wl, hs, g_host, t)
            assert int(sk) == osk
            if not osk:
                assert_close(np.array([gn]), np.array([ogn]), 1e-5, "grad_norm")
                t += 1
            skipped.append(int(sk))
            # this rank's pieces against the oracle's whole tensors
            for i, b, e in pieces[rank]:
                for name, got, want in (("w", st.w, hs.w), ("m", st.m, hs.m), ("v", st.v, hs.v)):
                    assert_close(W.as_f32(got[i][b:e]), want[i][b:e], rtol_for(k),
                                 f"rank {rank} step {k} {name}[{i}][{b}:{e}]")
        ranks[0][0].close()
        with open(os.path.join(result_dir, f"rank{rank}.ok"), "w") as f:
            f.write(" ".join(map(str, skipped)))
    finally:
        dist.destroy_process_group()


def test_two_processes_sum_the_partials_with_gloo(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        assert (tmp_path / f"rank{r}.ok").read_text() == "0 1 0"
