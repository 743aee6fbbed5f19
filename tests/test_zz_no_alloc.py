"""The workspace-free GEMV + argmax entry point (for callers that cannot
allocate device memory), called through the C ABI and checked against the
workspace-taking entry point on the same inputs, on two calls in a row.

Kept in its own file, collected last, so that a run stopping at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

TOL_REL, TOL_ABS = 1e-3, 1e-6


def test_noalloc_matches_workspace_entry_point_twice(dev):
    import nvfp4_speculative_draft_gb300 as nd
    L = nd.load()
    case = workloads.lm_head_m1(n=3000, k=1024, rows=3)
    p, s, g, _ = oracle.quantize(workloads.bits(case.w))
    wq = nd.Nvfp4Weight(torch.from_numpy(p).to(dev), torch.from_numpy(s).to(dev),
                        torch.tensor([g], dtype=torch.float32, device=dev), p.shape[0], p.shape[1] * 2)
    h, gamma = case.segments[0]
    h, gamma = h.to(dev), gamma.to(dev)
    ref_logits, ref_idx = nd.w4a16_gemv_argmax([(h, gamma, case.eps)], wq)
    torch.cuda.synchronize()
    ref_l, ref_i = ref_logits.cpu().numpy(), ref_idx.cpu().numpy()
    # tolerance scale from the oracle: S = sum |a_i w_i|
    a = oracle.rmsnorm_concat([(workloads.bits(case.segments[0][0]), workloads.bits(case.segments[0][1]),
                                case.eps)], 3)
    _, sabs = oracle.gemv(a, p, s, g)
    segs, m = nd._segments([(h, gamma, case.eps)])
    w = wq.c()
    stream = torch.cuda.current_stream().cuda_stream
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(2):
        logits = torch.full((3, 3000), float("nan"), dtype=torch.float32, device=dev)
        idx = torch.full((3,), -1, dtype=torch.int32, device=dev)
        rc = L.w4a16_gemv_argmax_noalloc(segs, 1, m, ctypes.byref(w), logits.data_ptr(),
                                         logits.stride(0), idx.data_ptr(), stream,
                                         status.data_ptr())
        assert rc == 0
        torch.cuda.synchronize()
        got_l, got_i = logits.cpu().numpy(), idx.cpu().numpy()
        assert np.all(np.abs(got_l.astype(np.float64) - ref_l) <= TOL_REL * sabs + TOL_ABS)
        assert np.array_equal(got_i, ref_i)
        assert status.item() == 0


def test_noalloc_rejects_batch_beyond_its_scratch(dev):
    import nvfp4_speculative_draft_gb300 as nd
    L = nd.load()
    w = nd._Weight(0x1000, 0x2000, 0x3000, 256, 512)
    seg = (nd._Segment * 1)(nd._Segment(0x4000, 512, 512, None, 1e-6))
    assert L.w4a16_gemv_argmax_noalloc(seg, 1, 17, ctypes.byref(w), None, 0, 0x7000, None,
                                       None) == 2
