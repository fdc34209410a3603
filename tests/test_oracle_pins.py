"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test fixes one part of the LAMB step (You et al., ICLR 2020, as adopted
by MegaScale -- guided-reading digest, section 2, per-layer learning-rate
adaptation; applied to one ZeRO-2 shard, digest section 3) by a closed form,
an invariant, a special case or a library routine, chosen so that a dropped
term, a wrong sign, a wrong exponent or a swapped operand fails one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "lamb_closed_forms.json")
B1, B2 = np.float32(0.9), np.float32(0.999)


# ----------------------------------------------------------------- helpers
def to_bits(values, dtype):
    """Float values -> bf16 / fp16 bit patterns via library conversions."""
    vals = [float(x) if not isinstance(x, str) else float(x) for x in values]
    if dtype == oracle.GRAD_FP16:
        return np.asarray(vals, dtype=np.float16).view(np.uint16).copy()
    t = torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_of(x32):
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def rand_state(rng, sizes, grad_dtype=oracle.GRAD_BF16, gscale=1e-3, zero_mv=True):
    w = [rng.normal(0, 0.02, n).astype(np.float32) for n in sizes]
    if zero_mv:
        m = [np.zeros(n, np.float32) for n in sizes]
        v = [np.zeros(n, np.float32) for n in sizes]
    else:
        m = [rng.normal(0, 1e-5, n).astype(np.float32) for n in sizes]
        v = [(1e-8 * rng.normal(0, 1, n) ** 2).astype(np.float32) for n in sizes]
    w16 = [np.zeros(n, np.uint16) for n in sizes]
    g = [to_bits(rng.normal(0, gscale, n), grad_dtype) for n in sizes]
    return w, m, v, w16, g


def copy_state(st):
    return [[None if a is None else a.copy() for a in lst] for lst in st]


def run(st, wd, **kw):
    w, m, v, w16, g = st
    base = dict(grad_dtype=oracle.GRAD_BF16, beta1=float(B1), beta2=float(B2), eps=1e-6,
                weight_decay=0.01, lr=1e-3, t=1)
    base.update(kw)
    return oracle.lamb_step(w, m, v, w16, g, wd, want_trust=True, **base)


def ev(expr):
    if isinstance(expr, (int, float)):
        return float(expr)
    return float(eval(expr, {"__builtins__": {}}, {"sqrt": math.sqrt, "inf": math.inf}))


def close(a, b, rtol, floor=1e-12):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.all(np.abs(a - b) <= np.maximum(floor, rtol * np.abs(b)))


# ------------------------------------------------------ hand closed forms
with open(GOLDEN) as f:
    CASES = json.load(f)["cases"]


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_closed_form_cases(case):
    gd = oracle.GRAD_FP16 if case["grad_dtype"] == "fp16" else oracle.GRAD_BF16
    ts = case["tensors"]
    w = [np.array([ev(x) for x in t["w"]], np.float32) for t in ts]
    m = [np.array([ev(x) for x in t["m"]], np.float32) for t in ts]
    v = [np.array([ev(x) for x in t["v"]], np.float32) for t in ts]
    g = [to_bits([float(x) for x in t["g"]], gd) for t in ts]
    w16 = [np.full(len(t["w"]), 0xABCD, np.uint16) for t in ts]
    wd = [t["wd"] for t in ts]
    before = copy_state((w, m, v, w16, g))
    sk, gn, trust = oracle.lamb_step(
        w, m, v, w16, g, wd, grad_dtype=gd, beta1=case["beta1"], beta2=case["beta2"],
        eps=case["eps"], weight_decay=case["weight_decay"], lr=case["lr"], t=case["t"],
        clip=case["clip"], loss_scale=case["loss_scale"], want_trust=True)
    ex = case["expect"]
    assert sk == ex["skipped"]
    if ex.get("unchanged"):
        assert gn == math.inf
        for a_list, b_list in zip((w, m, v, w16), before[:4]):
            for a, b in zip(a_list, b_list):
                assert a.tobytes() == b.tobytes()
        return
    rtol = case["rtol"]
    assert close(gn, ev(ex["grad_norm"]), 1e-14)
    assert close(trust, [ev(x) for x in ex["trust"]], max(rtol, 1e-14))
    for key, arrs in (("w", w), ("m", m), ("v", v)):
        for a, exprs in zip(arrs, ex[key]):
            want = np.array([ev(x) for x in exprs])
            if rtol == 0.0:
                assert np.array_equal(a.astype(np.float64), want), (key, a, want)
            else:
                assert close(a, want, rtol), (key, a, want)
    for a, b in zip(w16, w):
        assert np.array_equal(a, bf16_bits_of(b))


# -------------------------------------------- conversions vs libraries
def test_decode_bf16_every_pattern_matches_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = oracle.decode_grad(bits, oracle.GRAD_BF16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])


def test_decode_fp16_every_pattern_matches_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = oracle.decode_grad(bits, oracle.GRAD_FP16)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])


def test_bf16_round_nearest_even_matches_torch():
    rng = np.random.default_rng(7)
    pats = rng.integers(0, 2**32, 1 << 20, dtype=np.uint64).astype(np.uint32)
    special = []
    for hi in (0x0000, 0x0001, 0x3F80, 0x3F81, 0x7F7F, 0x7F7E, 0x007F, 0x8000, 0xBF80, 0xFF7F):
        for lo in (0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF):
            special.append((hi << 16) | lo)
    special += [0x7F800000, 0xFF800000, 0x00000001, 0x80000001, 0x7F7FFFFF]
    pats = np.concatenate([pats, np.array(special, np.uint32)])
    x = pats.view(np.float32)
    mine = oracle.bf16_rne(x)
    ref = bf16_bits_of(x)
    nan = np.isnan(x)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.all((mine[nan] & 0x7F80) == 0x7F80) and np.all((mine[nan] & 0x7F) != 0)


# ----------------------------------------------- closed forms at t = 1
@pytest.mark.parametrize("grad_dtype", [oracle.GRAD_BF16, oracle.GRAD_FP16])
def test_first_step_closed_form_random(grad_dtype):
    """t=1, m=v=0, wd=0, eps=0: r = sign(g), ||r|| = sqrt(n), trust = ||w||/sqrt(n)."""
    rng = np.random.default_rng(1)
    sizes = [1, 7, 8, 9, 300, 4099]
    st = rand_state(rng, sizes, grad_dtype)
    w0 = [a.copy() for a in st[0]]
    S = 1024.0 if grad_dtype == oracle.GRAD_FP16 else 1.0
    if grad_dtype == oracle.GRAD_FP16:
        st[4][:] = [to_bits(rng.normal(0, 1e-3, n) * S, grad_dtype) for n in sizes]
    ghat = [oracle.decode_grad(g, grad_dtype) / S for g in st[4]]
    assert all(np.all(x != 0) for x in ghat)
    lr = 0.01
    sk, gn, trust = run(st, [0] * len(sizes), eps=0.0, weight_decay=0.25, lr=lr,
                        grad_dtype=grad_dtype, loss_scale=S)
    assert sk == 0
    assert close(gn, np.linalg.norm(np.concatenate(ghat)), 1e-13)
    for i, n in enumerate(sizes):
        tr = np.linalg.norm(w0[i].astype(np.float64)) / math.sqrt(n)
        assert close(trust[i], tr, 1e-13)
        want_w = (w0[i] - lr * tr * np.sign(ghat[i])).astype(np.float32)
        assert np.array_equal(st[0][i], want_w) or close(st[0][i], want_w, 1.2e-7)
        assert close(st[1][i], (1 - float(B1)) * ghat[i], 1.2e-7)
        assert close(st[2][i], (1 - float(B2)) * ghat[i] ** 2, 1.2e-7)
        assert np.array_equal(st[3][i], bf16_bits_of(st[0][i]))


def test_first_step_closed_form_with_decay():
    """t=1, m=v=0, eps=0, wd>0: r = sign(g) + wd*w exactly."""
    rng = np.random.default_rng(2)
    sizes = [5, 64, 1000]
    st = rand_state(rng, sizes)
    w0 = [a.astype(np.float64) for a in st[0]]
    ghat = [oracle.decode_grad(g, oracle.GRAD_BF16) for g in st[4]]
    wd, lr = 0.5, 0.02
    sk, gn, trust = run(st, [1, 0, 1], eps=0.0, weight_decay=wd, lr=lr)
    for i, flag in enumerate([1, 0, 1]):
        r = np.sign(ghat[i]) + flag * wd * w0[i]
        tr = np.linalg.norm(w0[i]) / np.linalg.norm(r)
        assert close(trust[i], tr, 1e-13)
        assert close(st[0][i], (w0[i] - lr * tr * r), 1.2e-7)


# ----------------------------------------------------------- invariants
def test_scale_invariance_of_direction_and_update():
    """(g, m, v) -> (c g, c m, c^2 v) with eps=0 leaves r, trust and w' unchanged."""
    rng = np.random.default_rng(3)
    sizes = [33, 500]
    c = 4.0
    ks = [rng.integers(-60, 61, n) for n in sizes]
    for k in ks:
        k[k == 0] = 1
    g1 = [to_bits(k / 64.0, oracle.GRAD_BF16) for k in ks]
    gc = [to_bits(c * k / 64.0, oracle.GRAD_BF16) for k in ks]
    w = [rng.normal(0, 0.02, n).astype(np.float32) for n in sizes]
    m = [rng.normal(0, 0.1, n).astype(np.float32) for n in sizes]
    v = [rng.uniform(0.01, 0.2, n).astype(np.float32) for n in sizes]
    a = ([x.copy() for x in w], [x.copy() for x in m], [x.copy() for x in v],
         [np.zeros(n, np.uint16) for n in sizes], g1)
    b = ([x.copy() for x in w], [(c * x).astype(np.float32) for x in m],
         [(c * c * x).astype(np.float32) for x in v], [np.zeros(n, np.uint16) for n in sizes], gc)
    _, gna, ta = run(a, [1, 0], eps=0.0, t=5, lr=0.05)
    _, gnb, tb = run(b, [1, 0], eps=0.0, t=5, lr=0.05)
    assert close(gnb, c * gna, 1e-15)
    assert close(ta, tb, 1e-12)
    for i in range(2):
        assert close(a[0][i], b[0][i], 1.2e-7)
        assert close(c * a[1][i].astype(np.float64), b[1][i], 1e-15)
        assert close(c * c * a[2][i].astype(np.float64), b[2][i], 1e-15)


@pytest.mark.parametrize("k", [0, 4, 10, 16])
def test_power_of_two_loss_scale_is_bit_exact(k):
    rng = np.random.default_rng(4 + k)
    sizes = [3, 100, 2049]
    mags = [rng.uniform(-8, -1, n) for n in sizes]
    signs = [rng.choice([-1.0, 1.0], n) for n in sizes]
    g_true = [np.asarray(s * 2.0 ** e, np.float16) for s, e in zip(signs, mags)]
    S = 2.0 ** k
    base = rand_state(rng, sizes, zero_mv=False)
    a = copy_state(base)
    b = copy_state(base)
    a[4][:] = [x.view(np.uint16).copy() for x in g_true]
    b[4][:] = [(x.astype(np.float32) * np.float32(S)).astype(np.float16).view(np.uint16).copy()
               for x in g_true]
    ra = run(a, [1, 0, 1], grad_dtype=oracle.GRAD_FP16, loss_scale=1.0, t=4, clip=0.5)
    rb = run(b, [1, 0, 1], grad_dtype=oracle.GRAD_FP16, loss_scale=S, t=4, clip=0.5)
    assert ra[0] == rb[0] == 0 and ra[1] == rb[1]
    for la, lb in zip(a[:4], b[:4]):
        for x, y in zip(la, lb):
            assert x.tobytes() == y.tobytes()


@pytest.mark.parametrize("grad_dtype,bad", [(oracle.GRAD_BF16, 0x7F80), (oracle.GRAD_BF16, 0xFF80),
                                            (oracle.GRAD_BF16, 0x7FC1), (oracle.GRAD_FP16, 0x7C00),
                                            (oracle.GRAD_FP16, 0xFE01)])
def test_nonfinite_grad_skips_with_state_untouched(grad_dtype, bad):
    rng = np.random.default_rng(5)
    sizes = [10, 4096, 70000]
    st = rand_state(rng, sizes, grad_dtype, zero_mv=False)
    st[3][:] = [rng.integers(0, 65536, n, dtype=np.uint32).astype(np.uint16) for n in sizes]
    st[4][2][rng.integers(0, sizes[2])] = bad
    before = copy_state(st)
    sk, gn, _ = run(st, [1, 1, 0], grad_dtype=grad_dtype, t=9, clip=1.0)
    assert sk == 1 and gn == math.inf
    for la, lb in zip(st, before):
        for x, y in zip(la, lb):
            assert x.tobytes() == y.tobytes()


def test_finite_extremes_do_not_skip():
    """The largest finite bf16 and subnormals are finite: no skip."""
    st = rand_state(np.random.default_rng(6), [4])
    st[4][0][:] = np.array([0x7F7F, 0xFF7F, 0x0001, 0x8001], np.uint16)
    sk, gn, _ = run(st, [1])
    assert sk == 0 and math.isfinite(gn)


def test_clip_at_or_above_norm_is_no_clip():
    rng = np.random.default_rng(8)
    sizes = [17, 3000]
    base = rand_state(rng, sizes, zero_mv=False)
    ref = copy_state(base)
    _, gn, _ = run(ref, [1, 0], t=20, clip=0.0)
    for clip in (gn, 2 * gn, 1e30):
        st = copy_state(base)
        _, gn2, _ = run(st, [1, 0], t=20, clip=clip)
        assert gn2 == gn
        for la, lb in zip(st[:4], ref[:4]):
            for x, y in zip(la, lb):
                assert x.tobytes() == y.tobytes()


def test_clip_equals_feeding_scaled_grads():
    """Clipping by c = clip/G equals no clip with loss scale S/c."""
    rng = np.random.default_rng(9)
    sizes = [12, 5000]
    base = rand_state(rng, sizes, zero_mv=False, gscale=1e-2)
    a = copy_state(base)
    _, G, ta = run(a, [1, 0], t=7, clip=0.05)
    c = 0.05 / G
    assert c < 1
    b = copy_state(base)
    _, G2, tb = run(b, [1, 0], t=7, clip=0.0, loss_scale=1.0 / c)
    assert close(G2, G * c, 1e-13)
    assert close(ta, tb, 1e-12)
    for la, lb in zip(a[:3], b[:3]):
        for x, y in zip(la, lb):
            assert close(x, y, 2.4e-7, floor=1e-30)


def test_trust_is_per_tensor():
    """With clipping off, a joint step over [A, B] equals separate steps."""
    rng = np.random.default_rng(10)
    sizes = [77, 70001]
    base = rand_state(rng, sizes, zero_mv=False)
    joint = copy_state(base)
    run(joint, [1, 0], t=3)
    for i, flag in enumerate([1, 0]):
        one = [[lst[i].copy()] for lst in base]
        run(one, [flag], t=3)
        for la, lb in zip(one[:4], joint[:4]):
            assert la[0].tobytes() == lb[i].tobytes()


def test_zero_direction_keeps_weights():
    """g = 0, m = v = 0, no decay: r = 0, trust = 1, w unchanged, w16 = bf16(w)."""
    rng = np.random.default_rng(11)
    st = rand_state(rng, [50])
    st[4][0][:] = 0
    w0 = st[0][0].copy()
    sk, gn, tr = run(st, [0])
    assert sk == 0 and gn == 0.0 and tr[0] == 1.0
    assert st[0][0].tobytes() == w0.tobytes()
    assert np.array_equal(st[3][0], bf16_bits_of(w0))


def test_update_mask_matches_full_step():
    rng = np.random.default_rng(12)
    sizes = [9, 2000, 66000]
    base = rand_state(rng, sizes, zero_mv=False)
    full = copy_state(base)
    _, gfull, tfull = run(full, [1, 0, 1], t=11, clip=0.01)
    part = copy_state(base)
    for lst in part[:4]:
        lst[0] = None
        lst[2] = None
    _, gpart, tpart = run(part, [1, 0, 1], t=11, clip=0.01, update_mask=[0, 1, 0])
    assert gpart == gfull and tpart[1] == tfull[1]
    for la, lb in zip(part[:4], full[:4]):
        assert la[1].tobytes() == lb[1].tobytes()


def test_thread_count_does_not_change_results():
    rng = np.random.default_rng(13)
    sizes = [5, 200000, 131072]
    base = rand_state(rng, sizes, zero_mv=False)
    a, b = copy_state(base), copy_state(base)
    ra = run(a, [1, 0, 1], t=2, clip=0.02, n_threads=1)
    rb = run(b, [1, 0, 1], t=2, clip=0.02, n_threads=7)
    assert ra[1] == rb[1] and np.array_equal(ra[2], rb[2])
    for la, lb in zip(a[:4], b[:4]):
        for x, y in zip(la, lb):
            assert x.tobytes() == y.tobytes()


def test_empty_inputs():
    sk, gn = oracle.lamb_step([], [], [], [], [], [], grad_dtype=0, beta1=0.9, beta2=0.999,
                              eps=1e-6, weight_decay=0.01, lr=1e-3, t=1)
    assert sk == 0 and gn == 0.0
    st = rand_state(np.random.default_rng(14), [0, 3, 0])
    sk, gn, tr = run(st, [1, 1, 0])
    assert sk == 0 and gn > 0 and np.isnan(tr[0]) and np.isfinite(tr[1])


def test_rejects_bad_arguments():
    st = rand_state(np.random.default_rng(15), [4])
    for kw in (dict(t=0), dict(loss_scale=0.0), dict(loss_scale=-1.0), dict(grad_dtype=3),
               dict(loss_scale=math.inf)):
        with pytest.raises(ValueError):
            run(copy_state(st), [1], **kw)


# ------------------------------------------------- dynamic loss scaling
@pytest.mark.parametrize("growth,backoff,interval", [(2.0, 0.5, 3), (2.0, 0.5, 1), (1.5, 0.25, 5),
                                                     (4.0, 0.5, 2000)])
def test_loss_scale_update_matches_torch(growth, backoff, interval):
    """The oracle's scaler agrees with torch's own update routine (no clamps)."""
    rng = np.random.default_rng(int(growth * 10 + interval))
    flags = (rng.random(400) < 0.15).astype(int)
    flags[50:80] = 0
    s_t = torch.tensor([65536.0])
    g_t = torch.tensor([0], dtype=torch.int32)
    f_t = torch.tensor([0.0])
    s, g = 65536.0, 0
    for f in flags:
        f_t.fill_(float(f))
        torch._amp_update_scale_(s_t, g_t, f_t, growth, backoff, interval)
        s, g = oracle.loss_scale_update(s, g, f, growth=growth, backoff=backoff,
                                        growth_interval=interval)
        assert s == s_t.item() and g == g_t.item()


def test_loss_scale_update_hand_sequence_with_clamps():
    """Interval 2, x2 / x0.5, clamped to [1, 8]; written out by hand."""
    flags = [0, 0, 0, 0, 0, 0, 1, 1, 1, 1, 0, 0]
    want = [(2.0, 1), (4.0, 0), (4.0, 1), (8.0, 0), (8.0, 1), (8.0, 0),
            (4.0, 0), (2.0, 0), (1.0, 0), (1.0, 0), (1.0, 1), (2.0, 0)]
    s, g = 2.0, 0
    for f, w in zip(flags, want):
        s, g = oracle.loss_scale_update(s, g, f, growth=2.0, backoff=0.5, growth_interval=2,
                                        min_scale=1.0, max_scale=8.0)
        assert (s, g) == w


def test_loss_scale_growth_never_overflows():
    s, g = 3.0e38, 0
    s, g = oracle.loss_scale_update(s, g, 0, growth=2.0, backoff=0.5, growth_interval=1)
    assert s == np.float32(3.0e38) and g == 0


# ------------------------------------- tensors of more than one block
# The oracle walks tensors of more than 65,536 elements block by block (one
# block of direction values per thread, block partials of the norms added in
# block order).  These pins repeat the closed forms on tensors that take that
# path -- one element past a block, several full blocks plus a ragged tail --
# with weight-decay flags mixed, so that a partial sum dropped, a block's r
# applied at the wrong offset or a flag ignored there fails a pin.
BIG = [65537, 200003, 3 * 65536 + 5, 300]
BIG_WD = [1, 0, 1, 0]


def decoded(bits, grad_dtype):
    """bf16 / fp16 bit patterns -> float64 with numpy and torch (not the oracle)."""
    if grad_dtype == oracle.GRAD_FP16:
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_multi_block_first_step_closed_form():
    """t=1, m=v=0, eps=0: r = sign(g) + wd*w, trust = ||w||/||r||, w' = w - lr*trust*r,
    element by element over every block of every tensor."""
    rng = np.random.default_rng(21)
    st = rand_state(rng, BIG)
    w0 = [a.astype(np.float64) for a in st[0]]
    ghat = [decoded(g, oracle.GRAD_BF16) for g in st[4]]
    assert all(np.all(x != 0) for x in ghat)
    wd, lr = 0.25, 0.01
    sk, gn, trust = run(st, BIG_WD, eps=0.0, weight_decay=wd, lr=lr)
    assert sk == 0
    assert close(gn, np.linalg.norm(np.concatenate(ghat)), 1e-13)
    for i, flag in enumerate(BIG_WD):
        r = np.sign(ghat[i]) + flag * wd * w0[i]
        tr = np.linalg.norm(w0[i]) / np.linalg.norm(r)
        assert close(trust[i], tr, 1e-12), (i, trust[i], tr)
        assert close(st[0][i], w0[i] - lr * tr * r, 1.2e-7, floor=1e-30), i
        assert close(st[1][i], (1 - float(B1)) * ghat[i], 1.2e-7, floor=1e-30), i
        assert close(st[2][i], (1 - float(B2)) * ghat[i] ** 2, 1.2e-7, floor=1e-30), i
        assert np.array_equal(st[3][i], bf16_bits_of(st[0][i])), i


@pytest.mark.parametrize("grad_dtype", [oracle.GRAD_BF16, oracle.GRAD_FP16])
def test_multi_block_grad_norm_and_active_clip(grad_dtype):
    """G = ||g/S|| over all blocks of all tensors (numpy), and the clip factor
    clip/G reaches every block: m' = (1-b1)*(clip/G)*g^ at t=1."""
    rng = np.random.default_rng(22)
    S = 256.0
    st = rand_state(rng, BIG, grad_dtype)
    st[4][:] = [to_bits(rng.normal(0, 1e-3, n) * S, grad_dtype) for n in BIG]
    ghat = [decoded(g, grad_dtype) / S for g in st[4]]
    G = np.linalg.norm(np.concatenate(ghat))
    clip = 0.3 * G
    w0 = [a.astype(np.float64) for a in st[0]]
    lr = 0.02
    sk, gn, trust = run(st, BIG_WD, eps=0.0, weight_decay=0.0, lr=lr, clip=clip,
                        loss_scale=S, grad_dtype=grad_dtype)
    assert sk == 0
    assert close(gn, G, 1e-13)
    c = clip / G
    for i, n in enumerate(BIG):
        assert close(st[1][i], (1 - float(B1)) * c * ghat[i], 1.2e-7, floor=1e-30), i
        assert close(st[2][i], (1 - float(B2)) * (c * ghat[i]) ** 2, 1.2e-7, floor=1e-30), i
        tr = np.linalg.norm(w0[i]) / math.sqrt(n)  # r = sign(c g) = sign(g)
        assert close(trust[i], tr, 1e-12), i
        assert close(st[0][i], w0[i] - lr * tr * np.sign(ghat[i]), 1.2e-7, floor=1e-30), i


@pytest.mark.parametrize("k", [3, 12])
def test_multi_block_power_of_two_loss_scale_is_bit_exact(k):
    rng = np.random.default_rng(23 + k)
    mags = [rng.uniform(-8, -1, n) for n in BIG]
    signs = [rng.choice([-1.0, 1.0], n) for n in BIG]
    g_true = [np.asarray(s * 2.0 ** e, np.float16) for s, e in zip(signs, mags)]
    base = rand_state(rng, BIG, zero_mv=False)
    a, b = copy_state(base), copy_state(base)
    a[4][:] = [x.view(np.uint16).copy() for x in g_true]
    b[4][:] = [(x.astype(np.float32) * np.float32(2.0 ** k)).astype(np.float16)
               .view(np.uint16).copy() for x in g_true]
    ra = run(a, BIG_WD, grad_dtype=oracle.GRAD_FP16, loss_scale=1.0, t=6, clip=0.5)
    rb = run(b, BIG_WD, grad_dtype=oracle.GRAD_FP16, loss_scale=2.0 ** k, t=6, clip=0.5)
    assert ra[0] == rb[0] == 0 and ra[1] == rb[1]
    for la, lb in zip(a[:4], b[:4]):
        for x, y in zip(la, lb):
            assert x.tobytes() == y.tobytes()


@pytest.mark.parametrize("where", ["first", "middle", "last"])
def test_multi_block_nonfinite_anywhere_skips(where):
    """An inf/NaN in any block of a multi-block tensor skips the whole step."""
    rng = np.random.default_rng(24)
    st = rand_state(rng, BIG, zero_mv=False)
    n = BIG[1]
    idx = {"first": 0, "middle": 2 * 65536 + 17, "last": n - 1}[where]
    st[4][1][idx] = 0x7FC0 if where == "middle" else 0x7F80
    before = copy_state(st)
    sk, gn, _ = run(st, BIG_WD, t=3, clip=1.0)
    assert sk == 1 and gn == math.inf
    for la, lb in zip(st, before):
        for x, y in zip(la, lb):
            assert x.tobytes() == y.tobytes()
