"""Python binding of the LAMB step library: marshalling of torch tensors to
the C ABI of ``include/lamb.h``.  Every step of the optimizer runs in the
library's CUDA kernels; PyTorch only owns the memory and the stream.

LAMB (You et al., ICLR 2020) as adopted by MegaScale ("MegaScale: Scaling
Large Language Model Training to More Than 10,000 GPUs", guided-reading
digest, section 2), applied to one data-parallel rank's ZeRO-2 shard (digest
section 3).
"""
from __future__ import annotations

import ctypes
from typing import Sequence

import numpy as np
import torch

from . import _lib
from ._lib import LambError, LambHParams, LambLossScaler, LambResult, LambWorkItem, check

_GRAD_CODES = {torch.bfloat16: _lib.LAMB_GRAD_BF16, torch.float16: _lib.LAMB_GRAD_FP16}


def _ptrs(tensors) -> ctypes.Array:
    arr = (ctypes.c_void_p * max(1, len(tensors)))()
    for i, t in enumerate(tensors):
        arr[i] = t.data_ptr() if t.numel() else None
    return arr


def _check_tensors(name, tensors, dtype, sizes, device):
    if len(tensors) != len(sizes):
        raise ValueError(f"{name}: expected {len(sizes)} tensors, got {len(tensors)}")
    for i, (t, n) in enumerate(zip(tensors, sizes)):
        if not isinstance(t, torch.Tensor) or t.dtype != dtype:
            raise TypeError(f"{name}[{i}]: expected a {dtype} tensor")
        if t.device != device:
            raise ValueError(f"{name}[{i}]: on {t.device}, expected {device}")
        if not t.is_contiguous() or t.numel() != n:
            raise ValueError(f"{name}[{i}]: must be contiguous with {n} elements")


class GradSet:
    """Grad tensors already checked against a handle, with their pointer array."""

    __slots__ = ("tensors", "ptrs")

    def __init__(self, tensors, ptrs):
        self.tensors = tensors
        self.ptrs = ptrs


class Lamb:
    """LAMB optimizer state bound to caller-owned CUDA tensors.

    ``weights``, ``exp_avg``, ``exp_avg_sq``: fp32 tensors updated in place;
    ``weights_bf16``: bf16 tensors receiving the rounded weights; ``wd_flags``:
    per-tensor 0/1 (1 = apply weight decay).  All tensors must be contiguous,
    16-byte aligned and on one CUDA device.  ``stream`` defaults to the
    current torch stream at construction; every step runs on it.

    For one rank of a data-parallel group whose shard boundaries cut tensors
    (the split step, ``split_norms`` / ``split_moments`` / ``split_apply``):
    ``norm_exchange`` is a float64 CUDA tensor of 2 elements and
    ``tensor_exchange`` one of 2 * n_slots elements, both caller-owned, and
    ``exchange_slots`` gives each tensor -1 (held whole) or its slot.
    """

    def __init__(self, weights: Sequence[torch.Tensor], exp_avg: Sequence[torch.Tensor],
                 exp_avg_sq: Sequence[torch.Tensor], weights_bf16: Sequence[torch.Tensor],
                 wd_flags: Sequence[int], *, beta1: float = 0.9, beta2: float = 0.999,
                 eps: float = 1e-6, weight_decay: float = 0.01,
                 grad_dtype: torch.dtype = torch.bfloat16, stream=None,
                 exchange_slots: Sequence[int] | None = None,
                 norm_exchange: torch.Tensor | None = None,
                 tensor_exchange: torch.Tensor | None = None):
        self._lib = _lib.load()
        self._h = None
        if grad_dtype not in _GRAD_CODES:
            raise TypeError("grad_dtype must be torch.bfloat16 or torch.float16")
        n = len(weights)
        if len(wd_flags) != n:
            raise ValueError("wd_flags must have one entry per tensor")
        self.sizes = [int(t.numel()) for t in weights]
        self.device = weights[0].device if n else torch.device("cuda", torch.cuda.current_device())
        if self.device.type != "cuda":
            raise ValueError("LAMB state must live on a CUDA device")
        _check_tensors("weights", weights, torch.float32, self.sizes, self.device)
        _check_tensors("exp_avg", exp_avg, torch.float32, self.sizes, self.device)
        _check_tensors("exp_avg_sq", exp_avg_sq, torch.float32, self.sizes, self.device)
        _check_tensors("weights_bf16", weights_bf16, torch.bfloat16, self.sizes, self.device)
        self.grad_dtype = grad_dtype
        self._keep = (list(weights), list(exp_avg), list(exp_avg_sq), list(weights_bf16))
        with torch.cuda.device(self.device):
            self.stream = stream if stream is not None else torch.cuda.current_stream()
            hp = LambHParams(beta1, beta2, eps, weight_decay, _GRAD_CODES[grad_dtype])
            sizes = np.asarray(self.sizes, dtype=np.int64)
            flags = np.asarray([1 if f else 0 for f in wd_flags], dtype=np.uint8)
            h = ctypes.c_void_p()
            if norm_exchange is None and tensor_exchange is None and exchange_slots is None:
                check(self._lib.lamb_create(
                    ctypes.byref(h), n, sizes.ctypes.data, flags.ctypes.data, _ptrs(weights),
                    _ptrs(exp_avg), _ptrs(exp_avg_sq), _ptrs(weights_bf16), ctypes.byref(hp),
                    ctypes.c_void_p(self.stream.cuda_stream)))
            else:
                slots = np.full(max(1, n), -1, dtype=np.int32)
                if exchange_slots is not None:
                    if len(exchange_slots) != n:
                        raise ValueError("exchange_slots must have one entry per tensor")
                    slots[:n] = np.asarray(exchange_slots, dtype=np.int32)
                n_slots = 0
                for name, x in (("norm_exchange", norm_exchange),
                                ("tensor_exchange", tensor_exchange)):
                    if x is not None and (x.dtype != torch.float64 or x.device != self.device
                                          or not x.is_contiguous()):
                        raise ValueError(f"{name}: need a contiguous float64 tensor on "
                                         f"{self.device}")
                if tensor_exchange is not None:
                    if tensor_exchange.numel() % 2:
                        raise ValueError("tensor_exchange: need 2 * n_slots elements")
                    n_slots = tensor_exchange.numel() // 2
                if norm_exchange is not None and norm_exchange.numel() != 2:
                    raise ValueError("norm_exchange: need 2 elements")
                self._exchange_keep = (norm_exchange, tensor_exchange)
                ptr = lambda x: None if x is None else x.data_ptr()
                check(self._lib.lamb_create_sharded(
                    ctypes.byref(h), n, sizes.ctypes.data, flags.ctypes.data, _ptrs(weights),
                    _ptrs(exp_avg), _ptrs(exp_avg_sq), _ptrs(weights_bf16), slots.ctypes.data,
                    n_slots, ptr(norm_exchange), ptr(tensor_exchange), ctypes.byref(hp),
                    ctypes.c_void_p(self.stream.cuda_stream)))
        self._h = h
        self._n = n
        self._grad_ptrs = None
        self._grads_keep = None
        self._result = LambResult()
        self.loss_scale = None       # S the last step used
        self.next_loss_scale = None  # S the next step uses (dynamic scaling: for the backward)

    # ------------------------------------------------------------------ steps
    def prepare_grads(self, grads: Sequence[torch.Tensor]) -> "GradSet":
        """Validate a list of grad tensors once and return it in a form that
        ``set_grads`` / ``step`` / ``step_async`` take without checking again."""
        _check_tensors("grads", grads, self.grad_dtype, self.sizes, self.device)
        return GradSet(list(grads), _ptrs(grads))

    def set_grads(self, grads) -> None:
        """Remember the grad tensors used by ``step()`` (a list of tensors, or
        a ``GradSet`` from ``prepare_grads``)."""
        if not isinstance(grads, GradSet):
            grads = self.prepare_grads(grads)
        self._grads_keep = grads.tensors
        self._grad_ptrs = grads.ptrs

    def step(self, lr: float, t: int, clip: float = 0.0, loss_scale: float = 1.0,
             grads: Sequence[torch.Tensor] | None = None):
        """One LAMB step; returns ``(skipped, grad_norm)``.

        ``grads`` (optional) replaces the tensors given to ``set_grads``.  The
        call returns after the step has finished on the GPU.
        """
        if self._h is None:
            raise RuntimeError("handle is closed")
        if grads is not None:
            self.set_grads(grads)
        if self._grad_ptrs is None:
            raise ValueError("no grads: pass grads= or call set_grads first")
        check(self._lib.lamb_step(self._h, self._grad_ptrs, float(lr), int(t), float(clip),
                                  float(loss_scale), ctypes.byref(self._result)))
        self.loss_scale = float(self._result.loss_scale)
        self.next_loss_scale = float(self._result.next_loss_scale)
        return bool(self._result.skipped), float(self._result.grad_norm)

    def step_async(self, lr: float, clip: float = 0.0, loss_scale: float = 1.0,
                   grads: Sequence[torch.Tensor] | None = None) -> int:
        """Enqueue one LAMB step whose step number is the GPU's counter (see
        ``set_step``); returns its sequence number at once, without waiting
        for the GPU.  ``result(seq)`` gives its outcome."""
        if self._h is None:
            raise RuntimeError("handle is closed")
        if grads is not None:
            self.set_grads(grads)
        if self._grad_ptrs is None:
            raise ValueError("no grads: pass grads= or call set_grads first")
        seq = ctypes.c_int64()
        check(self._lib.lamb_step_async(self._h, self._grad_ptrs, float(lr), float(clip),
                                        float(loss_scale), ctypes.byref(seq)))
        return int(seq.value)

    def result(self, seq: int, wait: bool = True):
        """Outcome of step ``seq`` as ``(skipped, grad_norm, t)``, or ``None``
        if ``wait`` is false and the step has not finished."""
        res = LambResult()
        rc = self._lib.lamb_step_result(self._h, int(seq), 1 if wait else 0, ctypes.byref(res))
        if rc == _lib.LAMB_NOT_READY:
            return None
        check(rc)
        self.loss_scale = float(res.loss_scale)
        self.next_loss_scale = float(res.next_loss_scale)
        return bool(res.skipped), float(res.grad_norm), int(res.t)

    # ------------------------------------------------------------ split step
    def split_norms(self, grads=None, loss_scale: float = 1.0) -> None:
        """Phase 1 of a split step: this shard's grad-norm partials into
        ``norm_exchange`` (sum them over the group before phase 2)."""
        if grads is not None:
            self.set_grads(grads)
        if self._grad_ptrs is None:
            raise ValueError("no grads: pass grads= or call set_grads first")
        check(self._lib.lamb_split_norms(self._h, self._grad_ptrs, float(loss_scale)))

    def split_moments(self, lr: float, clip: float = 0.0, t: int = 0) -> None:
        """Phase 2: moments from the summed ``norm_exchange``; the shared
        tensors' {sum w^2, sum r^2} into ``tensor_exchange`` (sum them over the
        group before phase 3).  ``t`` 0: the GPU's step counter."""
        check(self._lib.lamb_split_moments(self._h, float(lr), int(t), float(clip)))

    def split_apply(self) -> int:
        """Phase 3: the update from the summed ``tensor_exchange``; returns
        the step's sequence number for ``result``."""
        seq = ctypes.c_int64()
        check(self._lib.lamb_split_apply(self._h, ctypes.byref(seq)))
        return int(seq.value)

    def split_step(self, lr: float, clip: float = 0.0, t: int = 0, grads=None,
                   loss_scale: float = 1.0, all_reduce=None) -> int:
        """One whole split step: the three phases with the group's two sums
        between them; returns the step's sequence number for ``result``.

        ``all_reduce(buf)`` must sum the float64 CUDA tensor ``buf`` over the
        data-parallel group in place, in order with this handle's stream (it
        is called with that stream current; ``torch.distributed.all_reduce``
        on an NCCL group does that).  ``None`` stands for a group of one.
        Slots of ``tensor_exchange`` that this rank does not hold are zeroed
        before phase 2, so that they add nothing to the sum."""
        keep = getattr(self, "_exchange_keep", None)
        if keep is None:
            raise ValueError("split steps need a handle made with the exchange buffers")
        norm_exchange, tensor_exchange = keep
        self.split_norms(grads, loss_scale)
        with torch.cuda.device(self.device), torch.cuda.stream(self.stream):
            if all_reduce is not None:
                all_reduce(norm_exchange)
            if tensor_exchange is not None:
                tensor_exchange.zero_()
        self.split_moments(lr, clip, t)
        if all_reduce is not None and tensor_exchange is not None:
            with torch.cuda.device(self.device), torch.cuda.stream(self.stream):
                all_reduce(tensor_exchange)
        return self.split_apply()

    def info(self) -> dict:
        """What the handle was built with: n_params, one_pass_params (elements
        whose whole step the moments kernel finishes, at 30 B/param),
        chunk_elems, n_items, and fused (moments and apply in one kernel)."""
        out = _lib.LambInfo()
        check(self._lib.lamb_get_info(self._h, ctypes.byref(out)))
        return {k: int(getattr(out, k)) for k, _ in out._fields_}

    def set_speculative(self, exp_avg2: Sequence[torch.Tensor] | None,
                        exp_avg_sq2: Sequence[torch.Tensor] | None) -> None:
        """Turn speculative mode on with a second set of m and v tensors (fp32,
        the state's sizes, caller-owned), or off with ``None, None``."""
        if exp_avg2 is None and exp_avg_sq2 is None:
            check(self._lib.lamb_set_speculative(self._h, None, None))
            self._second = None
            return
        _check_tensors("exp_avg2", exp_avg2, torch.float32, self.sizes, self.device)
        _check_tensors("exp_avg_sq2", exp_avg_sq2, torch.float32, self.sizes, self.device)
        second = (list(exp_avg2), list(exp_avg_sq2))
        check(self._lib.lamb_set_speculative(self._h, _ptrs(second[0]), _ptrs(second[1])))
        self._second = second

    def state_buffers(self):
        """The (m, v) tensor lists that hold the state now (speculative mode
        alternates between the two sets; waits for the stream)."""
        which = ctypes.c_int32()
        check(self._lib.lamb_state_buffers(self._h, ctypes.byref(which)))
        if which.value and getattr(self, "_second", None) is not None:
            return self._second
        return self._keep[1], self._keep[2]

    def set_step(self, t: int) -> None:
        """Set the GPU's step counter: the t of the next ``step_async``."""
        check(self._lib.lamb_set_step(self._h, int(t)))

    def loss_scale_device_ptr(self) -> int:
        """Device address of the dynamic loss scale (one fp32)."""
        p = ctypes.c_void_p()
        check(self._lib.lamb_loss_scale_device(self._h, ctypes.byref(p)))
        return int(p.value)

    def set_loss_scaler(self, init_scale: float = 65536.0, growth_factor: float = 2.0,
                        backoff_factor: float = 0.5, growth_interval: int = 2000,
                        min_scale: float = 1.0, max_scale: float = float("inf")) -> None:
        """Keep the loss scale on the GPU and adapt it after every step (back off
        after an overflow, grow after ``growth_interval`` clean steps); while on,
        ``step``'s ``loss_scale`` argument is ignored and ``next_loss_scale``
        tells the next backward pass which scale to use."""
        cfg = LambLossScaler(init_scale, growth_factor, backoff_factor, int(growth_interval),
                             min_scale, max_scale)
        check(self._lib.lamb_set_loss_scaler(self._h, ctypes.byref(cfg)))
        self.next_loss_scale = float(init_scale)

    def clear_loss_scaler(self) -> None:
        """Back to the fixed loss scale passed to each ``step``."""
        check(self._lib.lamb_set_loss_scaler(self._h, None))

    def trust(self) -> np.ndarray:
        """Per-tensor trust ratios of the last step that was not skipped."""
        out = np.empty(max(1, self._n), dtype=np.float32)
        check(self._lib.lamb_get_trust(self._h, out.ctypes.data, self._n))
        return out[: self._n]

    def snapshot_async(self, host_w, host_m, host_v, stream=None) -> None:
        """Copy every tensor's w, m, v into host tensors (page-locked for an
        asynchronous copy) on ``stream`` (default: a stream of this object's
        own).  The next ``step`` waits on the GPU for the copies before it
        writes the state; ``snapshot_wait`` blocks until they are done."""
        for name, lst in (("host_w", host_w), ("host_m", host_m), ("host_v", host_v)):
            if len(lst) != self._n:
                raise ValueError(f"{name}: expected {self._n} tensors")
            for t, n in zip(lst, self.sizes):
                if (not isinstance(t, torch.Tensor) or t.device.type != "cpu"
                        or t.dtype != torch.float32 or not t.is_contiguous() or t.numel() != n):
                    raise ValueError(f"{name}: need contiguous fp32 CPU tensors of the "
                                     f"state's sizes")
        if stream is None:
            if getattr(self, "_snap_stream", None) is None:
                self._snap_stream = torch.cuda.Stream(device=self.device)
            stream = self._snap_stream
        # The host tensors must outlive their copies: keep every outstanding set
        # (not one the library refused before enqueueing anything).
        if getattr(self, "_snap_keep", None) is None:
            self._snap_keep = []
        self._snap_keep.append((list(host_w), list(host_m), list(host_v)))
        try:
            check(self._lib.lamb_snapshot_async(self._h, _ptrs(host_w), _ptrs(host_m),
                                                _ptrs(host_v),
                                                ctypes.c_void_p(stream.cuda_stream)))
        except LambError as e:
            if e.code in (_lib.LAMB_ERR_INVALID, _lib.LAMB_ERR_ALIGN):
                self._snap_keep.pop()
            raise

    def snapshot_wait(self) -> None:
        """Block until every outstanding snapshot is in host memory."""
        check(self._lib.lamb_snapshot_wait(self._h))
        self._snap_keep = []

    def set_timing(self, enable: bool = True) -> None:
        """Turn the library's CUDA event monitor on or off."""
        check(self._lib.lamb_set_timing(self._h, 1 if enable else 0))

    def kernel_times(self, seq: int | None = None):
        """Device milliseconds of the (grad-norm, moments, apply) kernels of
        step ``seq`` (default: the last step enqueued)."""
        ms = (ctypes.c_float * 3)()
        if seq is None:
            check(self._lib.lamb_kernel_times(self._h, ms))
        else:
            check(self._lib.lamb_step_kernel_times(self._h, int(seq), ms))
        return float(ms[0]), float(ms[1]), float(ms[2])

    def close(self) -> None:
        if self._h is not None:
            h, self._h = self._h, None
            check(self._lib.lamb_destroy(h))

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


# --------------------------------------------------------------- work table
def plan(sizes: Sequence[int], chunk_elems: int = 0):
    """A work table like the one ``lamb_create`` builds (host only).

    ``chunk_elems`` 0 means the largest chunk size.  Returns ``(items,
    pack_ids)``: a structured array with fields ``begin, count, tensor`` and
    an int32 array of packed tensor ids.
    """
    lib = _lib.load()
    s = np.ascontiguousarray(np.asarray(sizes, dtype=np.int64))
    ni, npk = ctypes.c_int64(), ctypes.c_int64()
    check(lib.lamb_plan(len(s), s.ctypes.data, int(chunk_elems), None, 0, None, 0,
                        ctypes.byref(ni), ctypes.byref(npk)))
    items = (LambWorkItem * max(1, ni.value))()
    packs = np.zeros(max(1, npk.value), dtype=np.int32)
    check(lib.lamb_plan(len(s), s.ctypes.data, int(chunk_elems), items, ni.value,
                        packs.ctypes.data, npk.value, ctypes.byref(ni), ctypes.byref(npk)))
    dt = np.dtype([("begin", np.int64), ("count", np.int32), ("tensor", np.int32)])
    arr = np.frombuffer(bytes(items), dtype=dt)[: ni.value].copy()
    return arr, packs[: npk.value].copy()


def plan_limits() -> dict:
    lib = _lib.load()
    vals = [ctypes.c_int64() for _ in range(4)]
    lib.lamb_plan_limits(*[ctypes.byref(v) for v in vals])
    return dict(zip(("chunk_elems", "min_chunk_elems", "small_max", "pack_max"),
                    (v.value for v in vals)))


__all__ = ["Lamb", "GradSet", "LambError", "plan", "plan_limits"]
