"""The seeded input generator: sizes match the configurations' stated parameter
counts, draws are reproducible, and planted inf/NaN land where stated."""
import math

import numpy as np
import pytest
import torch

import workloads as W


def test_parameter_counts():
    assert W.tiny().n_params == 1_573_888
    assert W.shard175b().n_params == 1_811_963_904
    assert W.fp16_24().n_params == 1_208_057_856
    assert W.llama7b().n_params == 6_738_411_520
    r = W.ragged()
    assert len(r.sizes) == 4000 and min(r.sizes) >= 1 and max(r.sizes) <= 1 << 22
    assert 0.9e9 < r.n_params < 1.3e9
    assert len(r.zero_w) == 80
    assert all(f == (0 if n <= 4096 else 1) for n, f in zip(r.sizes, r.wd_flags))


def test_layout_alignment():
    offs, total = W.offsets([1, 7, 64, 65, 0, 3])
    assert all(o % W.ALIGN == 0 for o in offs)
    assert total >= offs[-1] + 3


def test_state_is_reproducible_and_zero_w_respected():
    wl = W.scaled(W.ragged(n_tensors=60, max_log2=14, seed=5), 5000)
    wl.zero_w = [3, 10]
    a = W.make_state(wl, "cpu")
    b = W.make_state(wl, "cpu")
    assert torch.equal(a.w_flat, b.w_flat) and torch.equal(a.v_flat, b.v_flat)
    assert float(a.w[3].abs().max()) == 0.0 and float(a.w[10].abs().max()) == 0.0
    assert float(a.v_flat.min()) >= 0.0
    s = float(a.w_flat.std())
    assert 0.015 < s < 0.025


def test_grads_reproducible_and_injected():
    wl = W.scaled(W.fp16_24(), 3000)
    f1, v1 = W.make_grads(wl, 7, "cpu")
    f2, _ = W.make_grads(wl, 7, "cpu")
    assert torch.equal(f1.view(torch.int16), f2.view(torch.int16))
    ti, idx, kind = W.injection_site(wl, 7)
    assert kind == "inf" and math.isinf(float(v1[ti][idx]))
    f3, _ = W.make_grads(wl, 8, "cpu")
    assert torch.isfinite(f3.float()).all()
    f4, v4 = W.make_grads(wl, 15, "cpu")
    ti, idx, kind = W.injection_site(wl, 15)
    assert kind == "nan" and math.isnan(float(v4[ti][idx]))


def test_student_t_has_heavy_tails():
    wl = W.scaled(W.llama7b(), 20000)
    flat, _ = W.make_grads(wl, 1, "cpu")
    x = flat.float().numpy() / wl.grad_sigma
    x = x[x != 0]
    kurt = np.mean(x ** 4) / np.mean(x ** 2) ** 2
    assert kurt > 6  # a normal has 3; t(3) has infinite kurtosis


def _check_zero2(sizes, n_ranks):
    pieces, slots = W.zero2_pieces(sizes, n_ranks)
    assert len(pieces) == len(slots) == n_ranks
    seen = [np.zeros(n, np.int32) for n in sizes]
    at = 0  # pieces are the flattened state, in order, rank after rank
    for mine, sl in zip(pieces, slots):
        assert len(mine) == len(sl)
        for (i, b, e), k in zip(mine, sl):
            assert 0 <= b < e <= sizes[i]
            assert b % 8 == 0
            flat = sum(sizes[:i]) + b
            assert flat == at
            at = flat + (e - b)
            seen[i][b:e] += 1
            assert (k == -1) == (b == 0 and e == sizes[i])
    assert at == sum(sizes)
    assert all((x == 1).all() for x in seen)
    slot_of = {}
    for mine, sl in zip(pieces, slots):
        for (i, _, _), k in zip(mine, sl):
            if k >= 0:
                assert slot_of.setdefault(i, k) == k
    assert sorted(slot_of.values()) == list(range(len(slot_of)))


def test_zero2_pieces_on_random_tensor_lists():
    """The same properties on random tensor lists (empty tensors included)
    and group sizes: the pieces tile the flattened state in order."""
    hyp = pytest.importorskip("hypothesis")
    st = hyp.strategies

    @hyp.settings(max_examples=200, deadline=None, derandomize=True)
    @hyp.given(st.lists(st.integers(0, 50000), min_size=1, max_size=25), st.integers(1, 9))
    def prop(sizes, n_ranks):
        _check_zero2(sizes, n_ranks)

    prop()


def test_zero2_pieces_cover_every_element_once_with_aligned_cuts():
    sizes = [5000, 70001, 300, 200003, 17, 4096, 40000]
    for n_ranks in (1, 2, 3, 5, 8):
        _check_zero2(sizes, n_ranks)
        pieces, slots = W.zero2_pieces(sizes, n_ranks)
        seen = [np.zeros(n, np.int32) for n in sizes]
        for mine, sl in zip(pieces, slots):
            assert len(mine) == len(sl)
            for (i, b, e), k in zip(mine, sl):
                assert 0 <= b < e <= sizes[i]
                assert b % 8 == 0  # every piece starts 16-byte aligned for 16-bit grads
                seen[i][b:e] += 1
                whole = b == 0 and e == sizes[i]
                assert (k == -1) == whole
        assert all((x == 1).all() for x in seen)
        # the same shared tensor has the same slot on every rank
        slot_of = {}
        for mine, sl in zip(pieces, slots):
            for (i, _, _), k in zip(mine, sl):
                if k >= 0:
                    assert slot_of.setdefault(i, k) == k
        assert sorted(slot_of.values()) == list(range(len(slot_of)))
