"""Run-to-run bit identity of every kernel at realistic sizes.

Each kernel computes in a fixed order (fixed-order reductions, one writer per
output, the argmax by 64-bit keys whose maximum does not depend on arrival
order), so repeated calls on the same inputs must give the same bits.  A
shared-memory stage read before its copy lands, a buffer refilled while still
being read, or a missing wait between programmatically overlapped launches
shows up here as differing outputs between runs, even when each run alone is
within the parity tolerance.  The calls run back to back on one stream, so
consecutive launches overlap the way the benchmark's do.
"""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


def nd():
    import nvfp4_speculative_draft_gb300 as m
    return m


def test_lm_head_gemv_argmax_repeatable(dev):
    """32768 x 4096, RMSNorm + GEMV + argmax, M = 1, 30 calls back to back."""
    m = nd()
    case = workloads.lm_head_m1(rows=4, device=dev)
    wq, _ = m.nvfp4_quantize(case.w)
    h, gamma = case.segments[0]
    outs = [m.w4a16_gemv_argmax([(h[i % 4:i % 4 + 1], gamma, 1e-6)], wq) for i in range(30)]
    torch.cuda.synchronize()
    for i, (lg, ix) in enumerate(outs[4:], start=4):
        ref_l, ref_i = outs[i % 4]
        assert torch.equal(lg.view(torch.int32), ref_l.view(torch.int32)), f"call {i}: logits differ"
        assert torch.equal(ix, ref_i), f"call {i}: argmax differs"


@pytest.mark.parametrize("m_rows", [8, 16])
def test_propose_gemv_argmax_repeatable(dev, m_rows):
    """151936 x 5120, M = 8 (prepared activations) and 16, 6 calls each."""
    m = nd()
    case = workloads.propose_m8(m=16, device=dev)
    wq, _ = m.nvfp4_quantize(case.w)
    x = case.segments[0][0][:m_rows].contiguous()
    del case
    outs = [m.w4a16_gemv_argmax([(x, None)], wq) for _ in range(6)]
    torch.cuda.synchronize()
    for lg, ix in outs[1:]:
        assert torch.equal(lg.view(torch.int32), outs[0][0].view(torch.int32))
        assert torch.equal(ix, outs[0][1])


def test_gemm_repeatable(dev):
    """1024 x 4864 x 2048 (the 240-wide tiles), BF16 and FP16-staged paths."""
    m = nd()
    case = workloads.prefill_gemm(m=1024, n=4864, k=2048, device=dev)
    wq, _ = m.nvfp4_quantize(case.w)
    ws = torch.empty(m.gemm_workspace_bytes(1024, 2048), dtype=torch.uint8, device=dev)
    for work in (None, ws):
        outs = [m.w4a16_gemm(case.a, wq, workspace=work) for _ in range(5)]
        torch.cuda.synchronize()
        for c in outs[1:]:
            assert torch.equal(c.view(torch.int16), outs[0].view(torch.int16))


def test_fp8_quantize_repeatable(dev):
    """The 151936 x 5120 FP8 quantisation, 4 calls."""
    m = nd()
    case = workloads.propose_m8(m=1, device=dev)
    outs = [m.fp8w_quantize(case.w) for _ in range(4)]
    torch.cuda.synchronize()
    for w8 in outs[1:]:
        assert torch.equal(w8.codes, outs[0].codes)
        assert torch.equal(w8.row_scale.view(torch.int32), outs[0].row_scale.view(torch.int32))
