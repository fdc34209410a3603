"""Seeded synthetic inputs for the LAMB step: tensor shapes, initial state and
per-step grads.  This module holds none of the optimizer's arithmetic; both
the CUDA path and the CPU oracle receive exactly the tensors it makes.

Shapes follow the parallel transformer block of MegaScale ("MegaScale: Scaling
Large Language Model Training to More Than 10,000 GPUs", guided-reading digest,
section 2: attention and MLP read the same input; section 8: the 175B model has
hidden size 12,288).  Values are drawn with torch generators seeded per
(config seed, purpose, step, chunk), so every tensor is reproducible and the
draws do not depend on the device's memory size.

Every tensor of a state lives at a 64-element-aligned offset inside one flat
buffer per array (w, m, v, w16), the layout of a ZeRO-2 shard; the tensors
handed to the optimizer are views into it.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np
import torch

ALIGN = 64            # elements between tensor starts (256 B of fp32)
GEN_CHUNK = 1 << 26   # elements drawn per generator seed

BETA1, BETA2, EPS, WEIGHT_DECAY = 0.9, 0.999, 1e-6, 0.01


@dataclasses.dataclass
class Workload:
    name: str
    description: str
    sizes: List[int]
    wd_flags: List[int]
    zero_w: List[int]                 # ids of tensors whose weights are all zero
    grad_dtype: torch.dtype
    t0: int                           # step number of the first step
    lr: float
    clip: float                       # <= 0: off
    loss_scale: float
    warm_state: bool                  # False: m = v = 0; True: m~N(0,1e-5), v=1e-8*chi2(1)
    grad_kind: str                    # "normal" or "student_t3"
    grad_sigma: float                 # std-dev (normal) or scale (student t)
    seed: int
    inject: Dict[int, str] = dataclasses.field(default_factory=dict)  # step -> "inf"/"nan"
    beta1: float = BETA1
    beta2: float = BETA2
    eps: float = EPS
    weight_decay: float = WEIGHT_DECAY

    @property
    def n_params(self) -> int:
        return int(sum(self.sizes))


# ------------------------------------------------------------------ configs
def _block(d: int, qkv: int, up: int, down_in: int) -> Tuple[List[int], List[int]]:
    """One parallel block: QKV, attention-out, MLP up, MLP down, LN gain, LN bias."""
    sizes = [d * qkv, d * d, d * up, down_in * d, d, d]
    return sizes, [1, 1, 1, 1, 0, 0]


def tiny() -> Workload:
    sizes, flags = [], []
    for _ in range(2):
        s, f = _block(256, 768, 1024, 1024)
        sizes += s
        flags += f
    return Workload("tiny-2L-d256", "2 parallel blocks, d=256, ffn=1024 (1,573,888 params)",
                    sizes, flags, [], torch.bfloat16, t0=1, lr=1e-3, clip=0.0, loss_scale=1.0,
                    warm_state=False, grad_kind="normal", grad_sigma=1e-3, seed=1001)


def shard175b() -> Workload:
    sizes, flags = _block(12288, 36864, 49152, 49152)
    return Workload("175B-block-shard", "one GPT-175B-shaped parallel block as a ZeRO-2 shard: "
                    "d=12288, ffn=49152 (1,811,963,904 params)", sizes, flags, [],
                    torch.bfloat16, t0=1000, lr=1e-3, clip=1.0, loss_scale=1.0, warm_state=True,
                    grad_kind="normal", grad_sigma=1e-4, seed=1002)


def ragged(n_tensors: int = 4000, max_log2: int = 22, seed: int = 1003) -> Workload:
    rng = np.random.default_rng(seed)
    u = rng.random(n_tensors)
    sizes = [max(1, int(math.floor(math.exp(x * max_log2 * math.log(2.0))))) for x in u]
    flags = [0 if n <= 4096 else 1 for n in sizes]
    n_zero = max(1, round(0.02 * n_tensors))
    zero = sorted(int(i) for i in rng.choice(n_tensors, n_zero, replace=False))
    return Workload(f"ragged-{n_tensors}", f"{n_tensors} tensors, sizes log-uniform in "
                    f"[1, 2^{max_log2}], 2% all-zero weights", sizes, flags, zero,
                    torch.bfloat16, t0=10, lr=1e-3, clip=0.0, loss_scale=1.0, warm_state=True,
                    grad_kind="normal", grad_sigma=1e-3, seed=seed)


def llama7b() -> Workload:
    sizes, flags = [32000 * 4096], [1]
    for _ in range(32):
        s, f = _block(4096, 12288, 22016, 11008)
        sizes += s
        flags += f
    sizes.append(32000 * 4096)
    flags.append(1)
    return Workload("7B-32L-d4096", "32 parallel blocks, d=4096, gated ffn=11008, "
                    "embed/unembed 32000x4096 (6,738,411,520 params)", sizes, flags, [],
                    torch.bfloat16, t0=500, lr=1e-3, clip=1.0, loss_scale=1.0, warm_state=True,
                    grad_kind="student_t3", grad_sigma=1e-4, seed=1004)


def fp16_24() -> Workload:
    sizes, flags = [], []
    for _ in range(24):
        s, f = _block(2048, 6144, 8192, 8192)
        sizes += s
        flags += f
    return Workload("fp16-24L-d2048", "24 parallel blocks, d=2048, ffn=8192, fp16 grads "
                    "x65536 (1,208,057,856 params)", sizes, flags, [], torch.float16, t0=1,
                    lr=1e-3, clip=0.0, loss_scale=65536.0, warm_state=False, grad_kind="normal",
                    grad_sigma=1e-3, seed=1005, inject={7: "inf", 15: "nan"})


WORKLOADS = {"tiny": tiny, "shard175b": shard175b, "ragged": ragged, "7b": llama7b,
           "fp16": fp16_24}


def scaled(wl: Workload, max_elems: int) -> Workload:
    """The same tensor mix with every tensor cut to at most max_elems elements
    (keeps the count of tensors, their wd flags and value recipes)."""
    return dataclasses.replace(wl, name=wl.name + f"-cut{max_elems}",
                               sizes=[min(n, max_elems) for n in wl.sizes])


# ------------------------------------------------------------------- layout
def offsets(sizes: Sequence[int], align: int = ALIGN) -> Tuple[List[int], int]:
    offs, at = [], 0
    for n in sizes:
        offs.append(at)
        at += (n + align - 1) // align * align
    return offs, max(at, align)


def _seed(*parts: int) -> int:
    h = 1469598103934665603
    for p in parts:
        h = ((h ^ (int(p) & 0xFFFFFFFFFFFFFFFF)) * 1099511628211) & 0xFFFFFFFFFFFFFFFF
    return h & 0x7FFFFFFFFFFFFFFF


def _fill_normal(buf: torch.Tensor, std: float, *key: int) -> None:
    """buf (flat fp32) <- N(0, std^2), chunk by chunk with one seed per chunk."""
    gen = torch.Generator(device=buf.device)
    for c, lo in enumerate(range(0, buf.numel(), GEN_CHUNK)):
        hi = min(buf.numel(), lo + GEN_CHUNK)
        gen.manual_seed(_seed(*key, c))
        torch.randn(hi - lo, generator=gen, device=buf.device, dtype=torch.float32,
                    out=buf[lo:hi])
        if std != 1.0:
            buf[lo:hi].mul_(std)


def _fill_chi2_1(buf: torch.Tensor, scale: float, *key: int) -> None:
    _fill_normal(buf, 1.0, *key)
    buf.square_().mul_(scale)


def _fill_grads(out16: torch.Tensor, kind: str, sigma: float, mult: float, *key: int) -> None:
    """out16 (flat bf16/fp16) <- (sigma * X) * mult rounded to its dtype, where X is
    N(0,1) ("normal") or Student-t with 3 degrees of freedom ("student_t3")."""
    gen = torch.Generator(device=out16.device)
    for c, lo in enumerate(range(0, out16.numel(), GEN_CHUNK)):
        hi = min(out16.numel(), lo + GEN_CHUNK)
        gen.manual_seed(_seed(*key, c))
        z = torch.randn(hi - lo, generator=gen, device=out16.device, dtype=torch.float32)
        if kind == "student_t3":
            chi = torch.zeros_like(z)
            for _ in range(3):
                chi.add_(torch.randn(hi - lo, generator=gen, device=out16.device,
                                     dtype=torch.float32).square_())
            z.div_(chi.div_(3.0).sqrt_())
        elif kind != "normal":
            raise ValueError(kind)
        z.mul_(sigma * mult)
        out16[lo:hi].copy_(z)
        del z


@dataclasses.dataclass
class State:
    wl: Workload
    offsets: List[int]
    total: int
    w_flat: torch.Tensor
    m_flat: torch.Tensor
    v_flat: torch.Tensor
    w16_flat: torch.Tensor

    def views(self, flat: torch.Tensor) -> List[torch.Tensor]:
        return [flat[o:o + n] for o, n in zip(self.offsets, self.wl.sizes)]

    def _cached(self, name: str, flat: torch.Tensor) -> List[torch.Tensor]:
        cache = self.__dict__.setdefault("_views", {})
        if name not in cache:
            cache[name] = self.views(flat)
        return cache[name]

    @property
    def w(self):
        return self._cached("w", self.w_flat)

    @property
    def m(self):
        return self._cached("m", self.m_flat)

    @property
    def v(self):
        return self._cached("v", self.v_flat)

    @property
    def w16(self):
        return self._cached("w16", self.w16_flat)

    def clone(self, device=None) -> "State":
        dev = device or self.w_flat.device
        return State(self.wl, self.offsets, self.total,
                     *(x.to(dev, copy=True) for x in
                       (self.w_flat, self.m_flat, self.v_flat, self.w16_flat)))


def make_state(wl: Workload, device) -> State:
    """Initial w, m, v and a zeroed bf16 copy (torch tensors on ``device``)."""
    offs, total = offsets(wl.sizes)
    dev = torch.device(device)
    w = torch.empty(total, dtype=torch.float32, device=dev)
    m = torch.empty(total, dtype=torch.float32, device=dev)
    v = torch.empty(total, dtype=torch.float32, device=dev)
    w16 = torch.zeros(total, dtype=torch.bfloat16, device=dev)
    _fill_normal(w, 0.02, wl.seed, 1)
    if wl.warm_state:
        _fill_normal(m, 1e-5, wl.seed, 2)
        _fill_chi2_1(v, 1e-8, wl.seed, 3)
    else:
        m.zero_()
        v.zero_()
    for i in wl.zero_w:
        w[offs[i]:offs[i] + wl.sizes[i]].zero_()
    return State(wl, offs, total, w, m, v, w16)


def grad_buffer(wl: Workload, device) -> Tuple[torch.Tensor, List[torch.Tensor]]:
    offs, total = offsets(wl.sizes)
    flat = torch.zeros(total, dtype=wl.grad_dtype, device=torch.device(device))
    return flat, [flat[o:o + n] for o, n in zip(offs, wl.sizes)]


def injection_site(wl: Workload, step: int) -> Optional[Tuple[int, int, str]]:
    """(tensor, index, kind) of the inf/NaN planted into this step's grads."""
    if step not in wl.inject:
        return None
    rng = np.random.default_rng(_seed(wl.seed, 99, step))
    nonempty = [i for i, n in enumerate(wl.sizes) if n > 0]
    ti = int(nonempty[int(rng.integers(len(nonempty)))])
    return ti, int(rng.integers(wl.sizes[ti])), wl.inject[step]


def fill_grads(wl: Workload, step: int, flat: torch.Tensor, loss_scale: float = None) -> None:
    """Grads of step ``step`` (1-based index in a run) into ``flat``; fp16
    grads carry the loss scale (``loss_scale`` if given, else the config's)."""
    if wl.grad_dtype == torch.float16:
        mult = wl.loss_scale if loss_scale is None else float(loss_scale)
    else:
        mult = 1.0
    _fill_grads(flat, wl.grad_kind, wl.grad_sigma, mult, wl.seed, 10, step)
    site = injection_site(wl, step)
    if site is not None:
        ti, idx, kind = site
        off = offsets(wl.sizes)[0][ti]
        flat[off + idx] = float("inf") if kind == "inf" else float("nan")


def make_grads(wl: Workload, step: int, device) -> Tuple[torch.Tensor, List[torch.Tensor]]:
    flat, views = grad_buffer(wl, device)
    fill_grads(wl, step, flat)
    return flat, views


# ------------------------------------------------------- numpy host copies
def as_bits(t: torch.Tensor) -> np.ndarray:
    """A 16-bit tensor as a host numpy uint16 array of its bit patterns."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def as_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy().astype(np.float32, copy=False)


# ------------------------------------------------------- ZeRO-2 rank pieces
def zero2_pieces(sizes: Sequence[int], n_ranks: int, align: int = 8):
    """Cut the concatenation of the tensors into ``n_ranks`` contiguous,
    nearly equal shards, as ZeRO-2 shards a flattened model over its
    data-parallel ranks; every cut is moved down to a multiple of ``align``
    elements within the tensor it falls in (so each piece keeps 16-byte
    alignment of 16-bit grads).

    Returns ``(pieces, slots)``: ``pieces[r]`` lists rank r's ``(tensor,
    begin, end)`` in order, and ``slots[r]`` gives each piece its exchange
    slot: -1 if the rank holds the whole tensor, else the tensor's index among
    the tensors that two or more ranks share (the same on every rank)."""
    total = int(sum(sizes))
    starts = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    cuts = [0]
    for r in range(1, n_ranks):
        c = (total * r) // n_ranks
        ti = int(np.searchsorted(starts, c, side="right") - 1)
        ti = min(ti, len(sizes) - 1)
        local = c - int(starts[ti])
        c = int(starts[ti]) + (local // align) * align
        cuts.append(max(c, cuts[-1]))
    cuts.append(total)
    pieces = []
    for r in range(n_ranks):
        lo, hi = cuts[r], cuts[r + 1]
        mine = []
        for i, n in enumerate(sizes):
            b, e = max(lo, int(starts[i])), min(hi, int(starts[i]) + int(n))
            if b < e:
                mine.append((i, b - int(starts[i]), e - int(starts[i])))
        pieces.append(mine)
    holders = {}
    for r, mine in enumerate(pieces):
        for i, b, e in mine:
            holders.setdefault(i, set()).add(r)
    shared = sorted(i for i, rs in holders.items() if len(rs) > 1)
    slot_of = {i: k for k, i in enumerate(shared)}
    slots = [[slot_of.get(i, -1) for i, _, _ in mine] for mine in pieces]
    return pieces, slots
