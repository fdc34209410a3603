"""Host-side tests of the C ABI: the library builds and loads without a GPU,
exports every symbol include/lamb.h declares, and builds a work table that
covers every element of every tensor exactly once with aligned chunk starts."""
import os
import re
import subprocess

import numpy as np
import pytest

import optimizer_step_gb300 as og
from optimizer_step_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lamb.h")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"LAMB_API\s+[\w\s\*]+?\b(lamb_\w+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert declared_symbols() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = og.load()
    for name in declared_symbols():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", og.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert set(declared_symbols()) <= exported
    # Nothing else of ours leaks out of the library.
    assert not [s for s in exported if s.startswith("lamb") and s not in declared_symbols()]


C_CLIENT = r'''
/* A plain C99 client of the library: every entry point of the header is
   referenced, so the link fails if one is missing.  Only lamb_plan and
   lamb_plan_limits, which need no GPU, are called. */
#include <stdio.h>
#include "lamb.h"

typedef void (*entry_point)(void);
static const entry_point entry_points[] = {
  (entry_point)lamb_create, (entry_point)lamb_create_sharded, (entry_point)lamb_step,
  (entry_point)lamb_step_async, (entry_point)lamb_step_result,
  (entry_point)lamb_split_norms, (entry_point)lamb_split_moments,
  (entry_point)lamb_split_apply, (entry_point)lamb_get_info,
  (entry_point)lamb_set_speculative, (entry_point)lamb_state_buffers,
  (entry_point)lamb_set_step, (entry_point)lamb_loss_scale_device,
  (entry_point)lamb_set_loss_scaler, (entry_point)lamb_snapshot_async,
  (entry_point)lamb_snapshot_wait, (entry_point)lamb_destroy, (entry_point)lamb_last_error,
  (entry_point)lamb_get_trust, (entry_point)lamb_set_timing,
  (entry_point)lamb_step_kernel_times, (entry_point)lamb_kernel_times,
  (entry_point)lamb_plan, (entry_point)lamb_plan_limits,
  (entry_point)lamb_grad_norm_noalloc,
};

int main(void) {
  int64_t sizes[3] = {10, 70000, 0}, n_items = 0, n_packs = 0, chunk = 0;
  lamb_work_item items[8];
  int32_t packs[4];
  lamb_plan_limits(&chunk, NULL, NULL, NULL);
  if (lamb_plan(3, sizes, 0, items, 8, packs, 4, &n_items, &n_packs) != LAMB_OK) {
    fprintf(stderr, "%s\n", lamb_last_error());
    return 1;
  }
  printf("%d %lld %lld %lld\n", (int)(sizeof entry_points / sizeof entry_points[0]),
         (long long)chunk, (long long)n_items, (long long)n_packs);
  return 0;
}
'''


def test_header_is_plain_c_and_a_c_program_links_and_runs(tmp_path):
    """The boundary is a C ABI: a C99 program that includes lamb.h and
    references every entry point compiles with gcc -std=c99 -Wall -Werror,
    links against the library and runs the host-only calls."""
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    lib = og.library_path()
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.dirname(HEADER), str(src), "-o", str(exe), lib,
                    "-Wl,-rpath," + os.path.dirname(lib)], check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    assert int(out[0]) == len(declared_symbols())
    assert int(out[1]) == og.plan_limits()["chunk_elems"]
    items, packs = og.plan([10, 70000, 0])
    assert (int(out[2]), int(out[3])) == (len(items), len(packs))


def check_plan(sizes, chunk=0):
    lim = og.plan_limits()
    chunk_elems = chunk or lim["chunk_elems"]
    pack_budget = max(chunk_elems, lim["small_max"])
    items, packs = og.plan(sizes, chunk)
    covered = [np.zeros(n, np.int32) if n <= 1 << 24 else None for n in sizes]
    counts = {}
    seen_packed = []
    seen_chunk = False
    for it in items:
        b, c, t = int(it["begin"]), int(it["count"]), int(it["tensor"])
        assert c > 0
        if t >= 0:
            seen_chunk = True
            n = sizes[t]
            assert n > lim["small_max"]
            assert c <= chunk_elems and b % 8 == 0 and b + c <= n
            counts.setdefault(t, []).append((b, c))
            if covered[t] is not None:
                covered[t][b:b + c] += 1
        else:
            assert not seen_chunk, "pack items must precede chunk items"
            ids = packs[b:b + c]
            assert c <= lim["pack_max"]
            assert sum(sizes[i] for i in ids) <= pack_budget
            for i in ids:
                assert 0 < sizes[i] <= lim["small_max"]
                seen_packed.append(int(i))
                if covered[i] is not None:
                    covered[i][:] += 1
    for t, segs in counts.items():
        segs.sort()
        at = 0
        for b, c in segs:
            assert b == at
            at += c
        assert at == sizes[t]
    # chunk items of one tensor are contiguous in the table; tensors of one
    # chunk first, then the rest, each group in tensor order
    tens = [int(t) for t in items["tensor"] if t >= 0]
    single = [t for t in tens if len(counts[t]) == 1]
    multi = [t for t in tens if len(counts[t]) > 1]
    assert tens == single + multi
    assert single == sorted(single) and multi == sorted(multi)
    first = {}
    for k, t in enumerate(tens):
        first.setdefault(t, k)
        assert k - first[t] < len(counts[t])
    assert sorted(seen_packed) == seen_packed
    assert len(set(seen_packed)) == len(seen_packed)
    for i, n in enumerate(sizes):
        if covered[i] is not None and n:
            assert np.all(covered[i] == 1), i
        if n == 0:
            assert i not in counts and i not in seen_packed
    return items, packs


@pytest.mark.parametrize("chunk", [0, 2048, 4096, 12288])
@pytest.mark.parametrize("sizes", [
    [], [0], [1], [7, 8, 9], [4095, 4096, 4097], [32768, 32769, 65535, 65536, 65537],
    [0, 1, 0, 5000, 0], [3] * 1000, [4096] * 20, [2**31 + 5], [12288 * 36864, 12288, 12288],
])
def test_plan_covers_every_element_once(sizes, chunk):
    if chunk and sum(sizes) > 1 << 31:
        pytest.skip("too many items to enumerate quickly")
    check_plan(sizes, chunk)


def test_plan_properties_on_random_tensor_lists():
    """The work table's invariants (check_plan) on random tensor lists that
    mix empty, packed, one-chunk and many-chunk tensors and sizes next to the
    pack and chunk limits, for every kind of chunk size."""
    hyp = pytest.importorskip("hypothesis")
    st = hyp.strategies
    lim = og.plan_limits()
    edges = [0, 1, 7, 8, 9, lim["small_max"] - 1, lim["small_max"], lim["small_max"] + 1,
             2047, 2048, 2049, 32767, 32768, 32769, 65536 + 7]
    size = st.one_of(st.sampled_from(edges), st.integers(0, 20), st.integers(0, 300000))

    @hyp.settings(max_examples=150, deadline=None, derandomize=True)
    @hyp.given(st.lists(size, max_size=60), st.sampled_from([0, 2048, 4096, 12288, 32768]))
    def prop(sizes, chunk):
        check_plan(sizes, chunk)

    prop()


def test_plan_ragged_config():
    import workloads
    wl = workloads.ragged()
    items, packs = check_plan(wl.sizes)
    lim = og.plan_limits()
    big = [n for n in wl.sizes if n > lim["small_max"]]
    assert len(items) >= sum((n + lim["chunk_elems"] - 1) // lim["chunk_elems"] for n in big)
    small = [n for n in wl.sizes if n <= lim["small_max"]]
    assert len(packs) == len(small)


def test_plan_chunks_are_balanced():
    lim = og.plan_limits()
    n = 3 * lim["chunk_elems"] + 9
    items, _ = og.plan([n])
    counts = sorted(int(c) for c in items["count"])
    assert len(counts) == 4 and counts[-1] - counts[0] <= 8 * len(counts)


def test_plan_rejects_bad_chunk_sizes():
    for chunk in (1024, 2047, 4000, -256):
        with pytest.raises(og.LambError):
            og.plan([10000], chunk)


def test_plan_rejects_negative_sizes():
    with pytest.raises(og.LambError):
        og.plan([4, -1])


def test_create_rejects_bad_arguments_without_touching_the_gpu():
    """Argument checks run before any CUDA call."""
    import ctypes
    lib = og.load()
    h = ctypes.c_void_p()
    hp = _lib.LambHParams(0.9, 0.999, 1e-6, 0.01, 0)
    sizes = np.array([8], np.int64)
    flags = np.array([1], np.uint8)
    good = (ctypes.c_void_p * 1)(256)
    odd = (ctypes.c_void_p * 1)(258)
    null = (ctypes.c_void_p * 1)(None)
    assert lib.lamb_create(ctypes.byref(h), -1, None, None, None, None, None, None,
                           ctypes.byref(hp), None) == _lib.LAMB_ERR_INVALID
    assert b"n_tensors" in lib.lamb_last_error()
    assert lib.lamb_create(ctypes.byref(h), 1, sizes.ctypes.data, flags.ctypes.data, good, good,
                           odd, good, ctypes.byref(hp), None) == _lib.LAMB_ERR_ALIGN
    assert lib.lamb_create(ctypes.byref(h), 1, sizes.ctypes.data, flags.ctypes.data, good, null,
                           good, good, ctypes.byref(hp), None) == _lib.LAMB_ERR_INVALID
    for bad in (_lib.LambHParams(1.0, 0.999, 1e-6, 0.01, 0),
                _lib.LambHParams(0.9, -0.1, 1e-6, 0.01, 0),
                _lib.LambHParams(0.9, 0.999, -1.0, 0.01, 0),
                _lib.LambHParams(0.9, 0.999, 1e-6, float("nan"), 0),
                _lib.LambHParams(0.9, 0.999, 1e-6, 0.01, 5)):
        assert lib.lamb_create(ctypes.byref(h), 1, sizes.ctypes.data, flags.ctypes.data, good,
                               good, good, good, ctypes.byref(bad), None) == _lib.LAMB_ERR_INVALID
    neg = np.array([-3], np.int64)
    assert lib.lamb_create(ctypes.byref(h), 1, neg.ctypes.data, flags.ctypes.data, good, good,
                           good, good, ctypes.byref(hp), None) == _lib.LAMB_ERR_INVALID


def test_step_rejects_bad_arguments_without_touching_the_gpu():
    import ctypes
    lib = og.load()
    res = _lib.LambResult()
    assert lib.lamb_step(None, None, 1e-3, 1, 0.0, 1.0, ctypes.byref(res)) == _lib.LAMB_ERR_INVALID
    assert lib.lamb_destroy(None) == _lib.LAMB_OK
