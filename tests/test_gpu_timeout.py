"""Bounded waits that run out, on the GPU, without faulting or hanging it.

The test build of the library (libnvfp4draft_withhold.so, built beside the
library; see NVFP4_TEST_WITHHOLD) never issues one TMA copy in CTA 0 -- the
GEMV's first weight stage of warp 0, the GEMM's first A tile -- and shortens
the wait limit to 20 ms.  Nothing of the withheld copy is ever in flight, so
the wait on it simply runs out.  Each call must return, report
NVFP4_ERR_TIMEOUT in the status word and leave the argmax workspace zeroed;
the context must stay usable: a normal call on the same stream afterwards
matches the oracle.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

TOL_REL, TOL_ABS = 1e-3, 1e-6
NVFP4_ERR_TIMEOUT = 6


def nd():
    import nvfp4_speculative_draft_gb300 as m
    return m


@pytest.fixture(scope="module")
def wl():
    """The withholding test build, through the same C ABI as the library."""
    from nvfp4_speculative_draft_gb300 import build
    if not os.path.exists(build.WITHHOLD_LIB):
        build.build(withhold=True)
    m = nd()
    L = ctypes.CDLL(build.WITHHOLD_LIB)
    vp, i64, i32, P = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.POINTER
    L.w4a16_gemv_argmax.argtypes = [P(m._Segment), i32, i32, P(m._Weight), vp, i64, vp, P(m._Exec)]
    L.w4a16_gemm.argtypes = [vp, i64, i64, P(m._Weight), vp, i64, P(m._Exec)]
    L.w4a16_gemv_argmax.restype = L.w4a16_gemm.restype = ctypes.c_int
    return L


@pytest.mark.parametrize("m_rows", [1, 8])
def test_gemv_wait_runs_out_and_the_call_returns(dev, wl, m_rows):
    m = nd()
    case = workloads.propose_m8(n=3000, k=1024, m=8)
    p, s, g, _ = oracle.quantize(workloads.bits(case.w))
    wq = m.Nvfp4Weight(torch.from_numpy(p).to(dev), torch.from_numpy(s).to(dev),
                       torch.tensor([g], dtype=torch.float32, device=dev), 3000, 1024)
    x = case.segments[0][0][:m_rows].contiguous().to(dev)
    ws = torch.zeros(m.gemv_workspace_bytes(m_rows, 1024), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    logits = torch.empty((m_rows, 3000), dtype=torch.float32, device=dev)
    idx = torch.empty((m_rows,), dtype=torch.int32, device=dev)
    segs, mm = m._segments([(x, None)])
    w = wq.c()
    stream = torch.cuda.current_stream(dev)
    ex = m._Exec(stream.cuda_stream, ws.data_ptr(), ws.numel(), status.data_ptr())
    rc = wl.w4a16_gemv_argmax(segs, 1, mm, ctypes.byref(w), logits.data_ptr(), logits.stride(0),
                              idx.data_ptr(), ctypes.byref(ex))
    assert rc == 0
    torch.cuda.synchronize()  # the kernel returned
    assert status.item() == NVFP4_ERR_TIMEOUT
    assert not ws[:m.ARGMAX_WS_BYTES].any().item(), "argmax workspace not returned to zero"
    # the same stream, the library proper: a normal call matches the oracle
    lg, ix = m.w4a16_gemv_argmax([(x, None)], wq, workspace=ws, stream=stream)
    torch.cuda.synchronize()
    y, sabs = oracle.gemv(workloads.bits(case.segments[0][0][:m_rows]), p, s, g)
    assert np.all(np.abs(lg.cpu().numpy().astype(np.float64) - y) <= TOL_REL * sabs + TOL_ABS)
    lgn = lg.cpu().numpy().astype(np.float64)
    for r in range(m_rows):
        assert int(ix[r]) == oracle.argmax(lgn[r])


def test_gemm_wait_runs_out_and_the_call_returns(dev, wl):
    m = nd()
    case = workloads.prefill_gemm(m=300, n=512, k=256)
    p, s, g, _ = oracle.quantize(workloads.bits(case.w))
    wq = m.Nvfp4Weight(torch.from_numpy(p).to(dev), torch.from_numpy(s).to(dev),
                       torch.tensor([g], dtype=torch.float32, device=dev), 512, 256)
    a = case.a.to(dev)
    c = torch.empty((300, 512), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    ex = m._Exec(stream.cuda_stream, None, 0, status.data_ptr())
    w = wq.c()
    rc = wl.w4a16_gemm(a.data_ptr(), 300, a.stride(0), ctypes.byref(w), c.data_ptr(), c.stride(0),
                       ctypes.byref(ex))
    assert rc == 0
    torch.cuda.synchronize()  # every role unwound, TMEM freed, the kernel returned
    assert status.item() == NVFP4_ERR_TIMEOUT
    c2 = m.w4a16_gemm(a, wq, stream=stream)
    torch.cuda.synchronize()
    rows = np.repeat(np.arange(0, 300, 37), 8)
    cols = np.tile(np.arange(0, 512, 67), 9)[:rows.size]
    exact, sabs = oracle.gemm_pairs(workloads.bits(case.a), p, s, g, rows, cols)
    got = c2.float().cpu().numpy()[rows, cols].astype(np.float64)
    assert np.all(np.abs(got - exact) <= TOL_REL * sabs + TOL_ABS + np.abs(exact) * 2.0 ** -8)
