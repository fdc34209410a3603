"""The oracle against a 50-digit decimal evaluation of the LAMB step (no GPU).

Hand-sized cases -- at most 8 elements per tensor, several tensors in one
step, mixed weight-decay flags, a zero-weight tensor, a one-element tensor,
active and inactive clipping, a loss scale, t > 1 with non-zero moments, bf16
and fp16 grads -- are evaluated in Python's ``decimal`` at 50 significant
digits, straight from the definition of the step: LAMB (You et al., ICLR
2020; per-layer trust ratio, MegaScale guided-reading digest, section 2) with
global clipping and loss-scale unscaling, on one ZeRO-2 shard (digest,
section 3).

This checks the oracle's precision handling rather than its formula (the
closed forms and invariants in test_oracle_pins.py pin the formula): every
quantity the oracle carries in fp64 must agree with the 50-digit value to
fp64 accuracy, and every stored fp32 value (m, v, w) must be the 50-digit
value rounded once, so within half an fp32 ulp.  The inputs are decoded with
numpy and torch, not with the oracle's own decoder.
"""
from decimal import Decimal, localcontext

import numpy as np
import pytest
import torch

import oracle

F32 = np.float32


def bits_of(values, grad_dtype):
    if grad_dtype == oracle.GRAD_FP16:
        return np.asarray(values, dtype=np.float16).view(np.uint16).copy()
    t = torch.tensor(np.asarray(values, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def values_of(bits, grad_dtype):
    if grad_dtype == oracle.GRAD_FP16:
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def decimal_step(w, m, v, g, wd_flags, *, beta1, beta2, eps, weight_decay, lr, t, clip,
                 loss_scale):
    """One LAMB step at 50 digits: (G, trust, m', v', w') as Decimals."""
    with localcontext() as ctx:
        ctx.prec = 50
        D = lambda x: Decimal(float(x))  # exact value of a binary float
        b1, b2, ep, wd, lr_, S = map(D, (beta1, beta2, eps, weight_decay, lr, loss_scale))
        ghat = [[D(x) / S for x in gi] for gi in g]
        G = sum((x * x for gi in ghat for x in gi), Decimal(0)).sqrt()
        c = D(clip) / G if clip > 0 and G > D(clip) else Decimal(1)
        bc1 = 1 - b1 ** t
        bc2 = 1 - b2 ** t
        trust, m_new, v_new, w_new = [], [], [], []
        for i in range(len(g)):
            gp = [c * x for x in ghat[i]]
            mi = [b1 * D(a) + (1 - b1) * x for a, x in zip(m[i], gp)]
            vi = [b2 * D(a) + (1 - b2) * x * x for a, x in zip(v[i], gp)]
            decay = wd if wd_flags[i] else Decimal(0)
            ri = [(a / bc1) / ((b / bc2).sqrt() + ep) + decay * D(x)
                  for a, b, x in zip(mi, vi, w[i])]
            wn = sum((D(x) * D(x) for x in w[i]), Decimal(0)).sqrt()
            rn = sum((x * x for x in ri), Decimal(0)).sqrt()
            tr = wn / rn if wn > 0 and rn > 0 else Decimal(1)
            trust.append(tr)
            m_new.append(mi)
            v_new.append(vi)
            w_new.append([D(x) - lr_ * tr * r for x, r in zip(w[i], ri)])
        return G, trust, m_new, v_new, w_new


def half_ulp_ok(got32, exact):
    """|got - exact| <= half an fp32 ulp of exact (plus fp64-level slack)."""
    got = np.asarray(got32, np.float32)
    ex = np.array([float(x) for x in exact], np.float64)
    ulp = np.spacing(np.abs(ex).astype(np.float32)).astype(np.float64)
    err = np.abs(got.astype(np.float64) - ex)
    return np.all(err <= 0.5 * ulp * (1 + 1e-9) + 1e-15 * np.abs(ex)), err / ulp


def make_case(seed, sizes, *, grad_dtype, t, m_scale, g_scale, zero_w=(), v_scale=None):
    rng = np.random.default_rng(seed)
    w = [rng.normal(0, 0.02, n).astype(F32) for n in sizes]
    for i in zero_w:
        w[i][:] = 0
    m = [(rng.normal(0, m_scale, n) if m_scale else np.zeros(n)).astype(F32) for n in sizes]
    vs = v_scale if v_scale is not None else m_scale
    v = [(vs * vs * rng.chisquare(1, n) if vs else np.zeros(n)).astype(F32) for n in sizes]
    g = [bits_of(rng.normal(0, g_scale, n), grad_dtype) for n in sizes]
    return w, m, v, g


CASES = {
    # several tensors, mixed flags, a zero-weight tensor, clipping active,
    # loss scale 4, t = 3 with non-zero moments
    "mixed_clip_scale4_t3": dict(
        seed=11, sizes=[8, 5, 1, 3], wd_flags=[1, 0, 1, 1], zero_w=(3,),
        grad_dtype=oracle.GRAD_BF16, t=3, m_scale=1e-4, g_scale=4e-3,
        hp=dict(beta1=0.9, beta2=0.999, eps=1e-6, weight_decay=0.01, lr=1e-3, clip=0.002,
                loss_scale=4.0)),
    # fp16 grads stored times 1024, t = 7, no clipping
    "fp16_scale1024_t7": dict(
        seed=12, sizes=[6, 7], wd_flags=[1, 0], grad_dtype=oracle.GRAD_FP16, t=7,
        m_scale=1e-3, g_scale=1.0,
        hp=dict(beta1=0.9, beta2=0.999, eps=1e-6, weight_decay=0.01, lr=2e-3, clip=0.0,
                loss_scale=1024.0)),
    # late step: bias corrections near 1, eps comparable to sqrt(v); a clip
    # threshold above the norm (inactive)
    "late_step_t1000_small_eps": dict(
        seed=13, sizes=[8, 8, 2], wd_flags=[1, 1, 0], grad_dtype=oracle.GRAD_BF16, t=1000,
        m_scale=1e-5, v_scale=1e-4, g_scale=1e-4,
        hp=dict(beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1, lr=1e-2, clip=10.0,
                loss_scale=1.0)),
    # first step from zero moments, other betas, strong decay, one element
    "first_step_betas_095_098": dict(
        seed=14, sizes=[1, 4, 8], wd_flags=[1, 1, 1], grad_dtype=oracle.GRAD_BF16, t=1,
        m_scale=0.0, g_scale=1e-2,
        hp=dict(beta1=0.95, beta2=0.98, eps=1e-6, weight_decay=0.5, lr=5e-2, clip=0.0,
                loss_scale=1.0)),
}


@pytest.mark.parametrize("name", list(CASES))
def test_oracle_matches_fifty_digit_evaluation(name):
    c = CASES[name]
    gd = c["grad_dtype"]
    w, m, v, g = make_case(c["seed"], c["sizes"], grad_dtype=gd, t=c["t"],
                           m_scale=c["m_scale"], g_scale=c["g_scale"],
                           zero_w=c.get("zero_w", ()), v_scale=c.get("v_scale"))
    # hyperparameters cross the library's interface as fp32: use those values
    hp = {k: float(F32(x)) for k, x in c["hp"].items()}
    gvals = [values_of(b, gd) for b in g]
    G, trust, m_ex, v_ex, w_ex = decimal_step(w, m, v, gvals, c["wd_flags"], t=c["t"], **hp)

    wo, mo, vo = [a.copy() for a in w], [a.copy() for a in m], [a.copy() for a in v]
    w16 = [np.zeros(n, np.uint16) for n in c["sizes"]]
    skipped, gn, tr = oracle.lamb_step(wo, mo, vo, w16, g, c["wd_flags"], grad_dtype=gd,
                                       t=c["t"], want_trust=True, **hp)
    assert skipped == 0
    assert abs(gn - float(G)) <= 1e-14 * float(G)
    clip_active = hp["clip"] > 0 and float(G) > hp["clip"]
    assert clip_active == (name == "mixed_clip_scale4_t3")
    for i in range(len(g)):
        assert abs(tr[i] - float(trust[i])) <= 1e-13 * float(trust[i]), (i, tr[i], trust[i])
        for got, ex, what in ((mo[i], m_ex[i], "m"), (vo[i], v_ex[i], "v"),
                              (wo[i], w_ex[i], "w")):
            ok, ulps = half_ulp_ok(got, ex)
            assert ok, (name, i, what, ulps)
        # w16 is bf16 round-to-nearest-even of the stored fp32 w (torch's conversion)
        ref16 = torch.from_numpy(wo[i]).to(torch.bfloat16).view(torch.int16).numpy()
        assert np.array_equal(w16[i], ref16.view(np.uint16))
    # the zero-weight tensor takes trust 1
    for i in c.get("zero_w", ()):
        assert tr[i] == 1.0


def test_fifty_digit_evaluation_sees_a_dropped_momentum_term():
    """The check has teeth: an oracle that dropped b1*m (planted here, on the
    CPU, by zeroing the old m before the call) disagrees with the decimal
    evaluation of the true inputs."""
    c = CASES["mixed_clip_scale4_t3"]
    gd = c["grad_dtype"]
    w, m, v, g = make_case(c["seed"], c["sizes"], grad_dtype=gd, t=c["t"],
                           m_scale=c["m_scale"], g_scale=c["g_scale"], zero_w=c["zero_w"])
    hp = {k: float(F32(x)) for k, x in c["hp"].items()}
    _, _, m_ex, _, _ = decimal_step(w, m, v, [values_of(b, gd) for b in g], c["wd_flags"],
                                    t=c["t"], **hp)
    wo, vo = [a.copy() for a in w], [a.copy() for a in v]
    mo = [np.zeros_like(a) for a in m]
    w16 = [np.zeros(n, np.uint16) for n in c["sizes"]]
    oracle.lamb_step(wo, mo, vo, w16, g, c["wd_flags"], grad_dtype=gd, t=c["t"], **hp)
    assert not half_ulp_ok(mo[0], m_ex[0])[0]


def test_oracle_matches_fifty_digit_evaluation_on_random_cases():
    """The same 50-digit comparison on random hand-sized cases: 1 to 4
    tensors of 1 to 8 elements, random weight-decay flags, step numbers,
    betas, eps, learning rates, loss scales and clip thresholds (active or
    not), bf16 and fp16 grads, and now and then a zero-weight tensor."""
    hyp = pytest.importorskip("hypothesis")
    st = hyp.strategies

    case = st.fixed_dictionaries({
        "seed": st.integers(0, 2 ** 31 - 1),
        "sizes": st.lists(st.integers(1, 8), min_size=1, max_size=4),
        "fp16": st.booleans(),
        "t": st.integers(1, 2000),
        "beta1": st.sampled_from([0.0, 0.5, 0.9, 0.95]),
        "beta2": st.sampled_from([0.9, 0.98, 0.999, 0.9999]),
        "eps": st.sampled_from([1e-8, 1e-6, 1e-3]),
        "wd": st.sampled_from([0.0, 0.01, 0.1]),
        "lr": st.sampled_from([1e-4, 1e-3, 5e-2]),
        "S": st.sampled_from([1.0, 4.0, 1000.0, 65536.0]),
        "clip_frac": st.sampled_from([0.0, 0.3, 0.9, 2.0]),
        "zero_w": st.booleans(),
    })

    @hyp.settings(max_examples=60, deadline=None, derandomize=True)
    @hyp.given(case)
    def prop(c):
        rng = np.random.default_rng(c["seed"])
        sizes = c["sizes"]
        gd = oracle.GRAD_FP16 if c["fp16"] else oracle.GRAD_BF16
        wd_flags = [int(x) for x in rng.integers(0, 2, len(sizes))]
        w = [rng.normal(0, 0.02, n).astype(F32) for n in sizes]
        if c["zero_w"]:
            w[0][:] = 0
        first = c["t"] == 1
        m = [(np.zeros(n) if first else rng.normal(0, 1e-4, n)).astype(F32) for n in sizes]
        v = [(np.zeros(n) if first else 1e-8 * rng.chisquare(1, n)).astype(F32) for n in sizes]
        S = c["S"] if c["fp16"] else (c["S"] if c["S"] <= 4.0 else 1.0)
        g = [bits_of(rng.normal(0, 1e-2, n) * S, gd) for n in sizes]
        gvals = [values_of(b, gd) for b in g]
        G = float(np.sqrt(sum(float(np.sum((x / S) ** 2)) for x in gvals)))
        hyp.assume(G > 0)
        clip = c["clip_frac"] * G
        hyp.assume(clip == 0.0 or abs(float(F32(clip)) / G - 1.0) > 1e-6)
        hp = {k: float(F32(x)) for k, x in dict(
            beta1=c["beta1"], beta2=c["beta2"], eps=c["eps"], weight_decay=c["wd"],
            lr=c["lr"], clip=clip, loss_scale=S).items()}
        Gd, trust, m_ex, v_ex, w_ex = decimal_step(w, m, v, gvals, wd_flags, t=c["t"], **hp)
        wo, mo, vo = [a.copy() for a in w], [a.copy() for a in m], [a.copy() for a in v]
        w16 = [np.zeros(n, np.uint16) for n in sizes]
        skipped, gn, tr = oracle.lamb_step(wo, mo, vo, w16, g, wd_flags, grad_dtype=gd,
                                           t=c["t"], want_trust=True, **hp)
        assert skipped == 0
        assert abs(gn - float(Gd)) <= 1e-14 * float(Gd)
        for i in range(len(sizes)):
            assert abs(tr[i] - float(trust[i])) <= 1e-13 * float(trust[i]), (i, tr[i], trust[i])
            for got, ex, what in ((mo[i], m_ex[i], "m"), (vo[i], v_ex[i], "v"),
                                  (wo[i], w_ex[i], "w")):
                ok, ulps = half_ulp_ok(got, ex)
                assert ok, (c, i, what, ulps)

    prop()
