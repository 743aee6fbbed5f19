"""The workspace-free GEMV + argmax entry point, for callers that cannot
allocate device memory (a fixed up-front device-memory budget, an allocator
that forbids side allocations, a decode loop that must not meet cudaMalloc's
implicit synchronisation), called through the C ABI.

Each batch width is checked against the CPU oracle (every logit within the
GEMV tolerance, the argmax by the top-2-gap rule) on two calls in a row, and
against the workspace-taking entry point (bit-equal argmax).  The widths cover
one and both MMA column groups, so every key slot of the library's fixed
scratch is used.

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
N, K = 3000, 1024


def check_against_oracle(lg, idx, y, sabs):
    tol = TOL_REL * sabs + TOL_ABS
    err = np.abs(lg.astype(np.float64) - y)
    assert np.all(err <= tol), f"{int((err > tol).sum())} logits out of tolerance"
    for r in range(y.shape[0]):
        i = int(idx[r])
        assert i == oracle.argmax(lg[r].astype(np.float64)), "not the first max of the GPU logits"
        j = oracle.argmax(y[r])
        order = np.argsort(-y[r], kind="stable")
        second = order[1] if order[0] == j else order[0]
        if y[r, j] - y[r, second] > tol[r, j] + tol[r, second]:
            assert i == j, f"row {r}: gpu argmax {i}, oracle {j}"
        else:
            assert y[r, i] >= y[r, j] - tol[r, j] - tol[r, i]


@pytest.mark.parametrize("m_rows", [1, 8, 16])
def test_noalloc_matches_oracle_twice(dev, m_rows):
    import nvfp4_speculative_draft_gb300 as nd
    L = nd.load()
    case = workloads.lm_head_m1(n=N, k=K, rows=m_rows)
    p, s, g, _ = oracle.quantize(workloads.bits(case.w))
    wq = nd.Nvfp4Weight(torch.from_numpy(p).to(dev), torch.from_numpy(s).to(dev),
                        torch.tensor([g], dtype=torch.float32, device=dev), N, K)
    h, gamma = case.segments[0]
    a = oracle.rmsnorm_concat([(workloads.bits(h), workloads.bits(gamma), case.eps)], m_rows)
    y, sabs = oracle.gemv(a, p, s, g)
    h, gamma = h.to(dev), gamma.to(dev)
    _, ws_idx = nd.w4a16_gemv_argmax([(h, gamma, case.eps)], wq, logits=False)
    segs, m = nd._segments([(h, gamma, case.eps)])
    w = wq.c()
    stream = torch.cuda.current_stream(dev).cuda_stream
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(2):
        logits = torch.full((m_rows, N), float("nan"), dtype=torch.float32, device=dev)
        idx = torch.full((m_rows,), -1, dtype=torch.int32, device=dev)
        rc = L.w4a16_gemv_argmax_noalloc(segs, 1, m, ctypes.byref(w), logits.data_ptr(),
                                         logits.stride(0), idx.data_ptr(), stream,
                                         status.data_ptr())
        assert rc == 0
        torch.cuda.synchronize()
        assert status.item() == 0
        got_i = idx.cpu().numpy()
        check_against_oracle(logits.cpu().numpy(), got_i, y, sabs)
        assert np.array_equal(got_i, ws_idx.cpu().numpy())


def test_noalloc_rejects_batch_beyond_its_scratch(dev):
    import nvfp4_speculative_draft_gb300 as nd
    L = nd.load()
    w = nd._Weight(0x1000, 0x2000, 0x3000, 256, 512)
    seg = (nd._Segment * 1)(nd._Segment(0x4000, 512, 512, None, 1e-6))
    assert L.w4a16_gemv_argmax_noalloc(seg, 1, 33, ctypes.byref(w), None, 0, 0x7000, None,
                                       None) == 2
