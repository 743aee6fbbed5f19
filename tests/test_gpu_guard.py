"""Guard bytes around every output of every call.

Each output lives inside a larger buffer filled with a canary byte (0xA5),
with a gap of canaries before it, after it and, for row-strided outputs,
between its rows (leading dimension > width).  After the call every canary
byte must be unchanged and the output itself must match the oracle (or the
library's own direct call).  This covers the argmax, log-probability, logits,
BF16 GEMV output, quantised codes, block scales, global scale and absmax,
the FP8 codes and row scales, and the GEMM output at a ragged m.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

CANARY = 0xA5
PAD = 64  # bytes of canaries before and after each output (keeps 16-byte alignment)


def nd():
    import nvfp4_speculative_draft_gb300 as m
    return m


class Guarded:
    """A device tensor of `shape` (row stride `ld` elements) inside a canary buffer."""

    def __init__(self, shape, dtype, dev, ld=None):
        esize = torch.tensor([], dtype=dtype).element_size()
        rows, cols = (shape[0], shape[1]) if len(shape) == 2 else (1, shape[0])
        self.ld = ld if ld is not None else cols
        self.nbytes = (rows - 1) * self.ld * esize + cols * esize
        self.buf = torch.full((PAD + self.nbytes + PAD,), CANARY, dtype=torch.uint8, device=dev)
        flat = self.buf[PAD:PAD + self.nbytes + (self.ld - cols) * esize].view(dtype)
        if len(shape) == 2:
            self.t = flat.as_strided((rows, cols), (self.ld, 1))
        else:
            self.t = flat[:cols]
        self.rows, self.cols, self.esize = rows, cols, esize

    def check(self):
        b = self.buf.cpu().numpy()
        mask = np.ones(b.size, dtype=bool)  # True where a canary must survive
        for r in range(self.rows):
            s = PAD + r * self.ld * self.esize
            mask[s:s + self.cols * self.esize] = False
        bad = np.flatnonzero(mask & (b != CANARY))
        assert bad.size == 0, f"{bad.size} guard bytes overwritten, first at offset {bad[0] - PAD}"


def test_guard_bytes_quantisers(dev):
    m = nd()
    n, k = 37, 160
    case = workloads.propose_m8(n=n, k=k, m=1)
    w = case.w.to(dev)
    pk, sc, gs, am = (Guarded((n, k // 2), torch.uint8, dev), Guarded((n, k // 16), torch.uint8, dev),
                      Guarded((1,), torch.float32, dev), Guarded((1,), torch.float32, dev))
    out = m.Nvfp4Weight(pk.t, sc.t, gs.t, n, k)
    m.nvfp4_quantize(w, out=out, absmax=am.t)
    c8, rs = Guarded((n, k), torch.uint8, dev), Guarded((n,), torch.float32, dev)
    m.fp8w_quantize(w, out=m.Fp8Weight(c8.t, rs.t, n, k))
    torch.cuda.synchronize()
    for gd in (pk, sc, gs, am, c8, rs):
        gd.check()
    p, s, g, a = oracle.quantize(workloads.bits(case.w))
    assert np.array_equal(pk.t.cpu().numpy(), p) and np.array_equal(sc.t.cpu().numpy(), s)
    assert gs.t.item() == float(g) and am.t.item() == float(a)
    cc, ss = oracle.fp8_quantize(workloads.bits(case.w))
    assert np.array_equal(c8.t.cpu().numpy(), cc) and np.array_equal(rs.t.cpu().numpy(), ss)


@pytest.mark.parametrize("m_rows", [1, 3, 12, 20])
def test_guard_bytes_gemv_outputs(dev, m_rows):
    """logits (row gaps), argmax, log-probability, BF16 output; ragged n."""
    m = nd()
    n, k = 301, 512
    case = workloads.propose_m8(n=n, k=k, m=32)
    wq, _ = m.nvfp4_quantize(case.w.to(dev))
    x = case.segments[0][0][:m_rows].contiguous().to(dev)
    lg, ix, lp = (Guarded((m_rows, n), torch.float32, dev, ld=n + 13), Guarded((m_rows,), torch.int32, dev),
                  Guarded((m_rows,), torch.float32, dev))
    mask = torch.from_numpy(np.full((m_rows, (n + 31) // 32), -1, dtype=np.int32)).to(dev)
    m.w4a16_gemv_argmax_ex([(x, None)], wq, mask=mask, out_logits=lg.t, out_argmax=ix.t, out_logprob=lp.t)
    yb = Guarded((m_rows, n), torch.bfloat16, dev, ld=n + 5)
    m.w4a16_gemv([(x, None)], wq, out=yb.t)
    ix2 = Guarded((m_rows,), torch.int32, dev)
    m.w4a16_gemv_argmax([(x, None)], wq, logits=False, out_argmax=ix2.t)
    torch.cuda.synchronize()
    for gd in (lg, ix, lp, yb, ix2):
        gd.check()
    ref_l, ref_i = m.w4a16_gemv_argmax([(x, None)], wq)
    torch.cuda.synchronize()
    assert torch.equal(lg.t.cpu(), ref_l.cpu())
    assert torch.equal(ix.t.cpu(), ref_i.cpu()) and torch.equal(ix2.t.cpu(), ref_i.cpu())
    assert torch.equal(yb.t.cpu(), ref_l.to(torch.bfloat16).cpu())
    assert torch.isfinite(lp.t).all().item()


def test_guard_bytes_gemm_ragged_m(dev):
    m = nd()
    mm, n, k = 130, 256, 128
    case = workloads.prefill_gemm(m=mm, n=n, k=k)
    wq, _ = m.nvfp4_quantize(case.w.to(dev))
    c = Guarded((mm, n), torch.bfloat16, dev, ld=n + 24)
    m.w4a16_gemm(case.a.to(dev), wq, out=c.t)
    torch.cuda.synchronize()
    c.check()
    ref = m.w4a16_gemm(case.a.to(dev), wq)
    torch.cuda.synchronize()
    assert torch.equal(c.t.cpu(), ref.cpu())
