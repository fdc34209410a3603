"""Guard bands around every array the kernels touch (GPU).

Without a memory checker, out-of-range accesses are looked for the way a
red-zone allocator finds them.  Every w, m, v, w16 and grad array is carved
out of a larger device buffer, with 4 KB guard bands on both sides filled with
NaN bit patterns:
- a kernel that reads a guard element of w, m or v poisons that tensor's norms,
  trust ratio and update, which the comparison with the oracle catches;
- a read of a grad guard element makes the step non-finite, so the step is
  skipped where the oracle's is not;
- a write into any guard band changes its bits.

The sizes cover every path: packed tensors (warp per tensor), a chunk per
tensor, several chunks, the TMA-staged pieces of the apply kernel with ragged
last pieces, and tails of fewer than 8 elements.
"""
import numpy as np
import pytest
import torch

import oracle
from optimizer_step_gb300 import Lamb

from parity import assert_close, check_bf16_copy, f32, rtol_for

pytestmark = pytest.mark.gpu

GUARD_BYTES = 4096
SIZES = [1, 7, 8, 9, 15, 100, 2047, 2048, 2049, 4095, 4096, 4097, 6143, 32767, 32768,
         32769, 65539, 5 * 32768 + 1234, 300001]
NAN32 = 0x7FC00000
NAN16 = {torch.bfloat16: 0x7FC0, torch.float16: 0x7E00}
INT_OF = {4: torch.int32, 2: torch.int16}


class Guarded:
    """A device buffer of ``n`` elements between two NaN guard bands."""

    def __init__(self, n, dtype, nan_bits, device):
        es = torch.tensor([], dtype=dtype).element_size()
        self.pad = GUARD_BYTES // es
        self.buf = torch.empty(self.pad + n + self.pad, dtype=dtype, device=device)
        ints = self.buf.view(INT_OF[es])
        bits = nan_bits if nan_bits < 1 << (8 * es - 1) else nan_bits - (1 << (8 * es))
        ints.fill_(bits)
        self.view = self.buf[self.pad:self.pad + n]
        self.guard_bits = self._guards().clone()

    def _guards(self):
        ints = self.buf.view(INT_OF[self.buf.element_size()])
        return torch.cat([ints[:self.pad], ints[self.buf.numel() - self.pad:]])

    def guards_intact(self):
        return torch.equal(self._guards(), self.guard_bits)


def bits16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16).copy()


@pytest.mark.parametrize("speculative", [False, True])
@pytest.mark.parametrize("grad_dtype", [torch.bfloat16, torch.float16])
def test_no_kernel_touches_the_guard_bands(grad_dtype, speculative):
    dev = torch.device("cuda")
    rng = np.random.default_rng(29)
    n_t = len(SIZES)
    wd = [1 if n > 4096 else 0 for n in SIZES]
    gcode = oracle.GRAD_FP16 if grad_dtype == torch.float16 else oracle.GRAD_BF16
    S = 1024.0 if grad_dtype == torch.float16 else 1.0

    # host state (the oracle's copy) and the guarded device copies
    hw = [rng.normal(0, 0.02, n).astype(np.float32) for n in SIZES]
    hw[2][:] = 0.0  # a zero-weight tensor (trust 1)
    hm = [rng.normal(0, 1e-5, n).astype(np.float32) for n in SIZES]
    hv = [(1e-8 * rng.chisquare(1, n)).astype(np.float32) for n in SIZES]
    h16 = [np.zeros(n, np.uint16) for n in SIZES]
    gw = [Guarded(n, torch.float32, NAN32, dev) for n in SIZES]
    gm = [Guarded(n, torch.float32, NAN32, dev) for n in SIZES]
    gv = [Guarded(n, torch.float32, NAN32, dev) for n in SIZES]
    g16 = [Guarded(n, torch.bfloat16, NAN16[torch.bfloat16], dev) for n in SIZES]
    gg = [Guarded(n, grad_dtype, NAN16[grad_dtype], dev) for n in SIZES]
    for i in range(n_t):
        gw[i].view.copy_(torch.from_numpy(hw[i]))
        gm[i].view.copy_(torch.from_numpy(hm[i]))
        gv[i].view.copy_(torch.from_numpy(hv[i]))
        g16[i].view.zero_()
    everything = gw + gm + gv + g16 + gg

    opt = Lamb([x.view for x in gw], [x.view for x in gm], [x.view for x in gv],
               [x.view for x in g16], wd, grad_dtype=grad_dtype)
    opt.set_grads([x.view for x in gg])
    if speculative:  # the second m and v set between guard bands too (its contents: any)
        gm2 = [Guarded(n, torch.float32, NAN32, dev) for n in SIZES]
        gv2 = [Guarded(n, torch.float32, NAN32, dev) for n in SIZES]
        for x in gm2 + gv2:
            x.view.zero_()
        everything += gm2 + gv2
        opt.set_speculative([x.view for x in gm2], [x.view for x in gv2])
    hp = dict(beta1=f32(0.9), beta2=f32(0.999), eps=f32(1e-6), weight_decay=f32(0.01),
              lr=f32(1e-3), clip=f32(0.05), loss_scale=S)
    try:
        for k, t in enumerate(range(5, 8), start=1):
            g_host = []
            for i, n in enumerate(SIZES):
                vals = torch.from_numpy(rng.normal(0, 1e-3, n) * S).to(grad_dtype)
                gg[i].view.copy_(vals)
                g_host.append(bits16(vals))
            torch.cuda.synchronize()
            sk, gn = opt.step(hp["lr"], t, hp["clip"], S)
            osk, ogn, otr = oracle.lamb_step(hw, hm, hv, h16, g_host, wd, grad_dtype=gcode,
                                             t=t, want_trust=True, **hp)
            assert not sk and not osk, "a step saw a non-finite grad: a guard band was read"
            assert_close(np.array([gn]), np.array([ogn]), rtol_for(k), f"step {k} grad_norm")
            rtol = rtol_for(k)
            cur_m, cur_v = opt.state_buffers()  # speculative mode: the set holding the state
            for i in range(n_t):
                w_gpu = gw[i].view.cpu().numpy()
                assert_close(w_gpu, hw[i], rtol, f"step {k} w[{i}] (n={SIZES[i]})")
                assert_close(cur_m[i].cpu().numpy(), hm[i], rtol, f"step {k} m[{i}]")
                assert_close(cur_v[i].cpu().numpy(), hv[i], rtol, f"step {k} v[{i}]")
                check_bf16_copy(bits16(g16[i].view), w_gpu, h16[i], hw[i], rtol,
                                f"step {k} w16[{i}]")
            assert_close(opt.trust(), otr, 1e-5, f"step {k} trust")
            bad = [j for j, x in enumerate(everything) if not x.guards_intact()]
            assert not bad, f"step {k}: guard bands written: {bad}"
    finally:
        opt.close()
