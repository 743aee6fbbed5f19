"""GPU parity of the FP8 weight variant (per-row E4M3 codes, fp8w_*) against
the oracle.

Bars: codes and row scales bit-exact; FP32 outputs within 1e-3 * S + 1e-6
(BF16 outputs plus one BF16 ulp); argmax equal to the first maximum of the
GPU's own logits and to the oracle's index when its top-2 gap exceeds both
tolerances.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

TOL_REL, TOL_ABS = 1e-3, 1e-6


def nd():
    import nvfp4_speculative_draft_gb300 as m
    return m


def quantize_both(w, dev):
    m = nd()
    wq = m.fp8w_quantize(w.to(dev).contiguous())
    codes, scales = oracle.fp8_quantize(workloads.bits(w))
    torch.cuda.synchronize()
    assert np.array_equal(wq.row_scale.cpu().numpy(), scales), "row scales differ"
    gc = wq.codes.cpu().numpy()
    if not np.array_equal(gc, codes):
        bad = np.argwhere(gc != codes)[:5]
        raise AssertionError(f"codes differ at {bad.tolist()}")
    return wq, codes, scales


@pytest.mark.parametrize("n,k", [(1, 32), (37, 160), (256, 512), (129, 4096)])
def test_fp8_quantize_bit_exact(dev, n, k):
    g = torch.Generator().manual_seed(n * 7 + k)
    w = (torch.randn((n, k), generator=g) * 0.02 *
         torch.exp2(torch.randint(-10, 6, (n, 1), generator=g).float())).to(torch.bfloat16)
    quantize_both(w, dev)


def test_fp8_quantize_zero_rows_signs_and_saturation(dev):
    w = torch.zeros((4, 64), dtype=torch.bfloat16)
    w[1, 3] = -0.5
    w[1, 4] = -0.0
    w[2] = torch.linspace(-3, 3, 64).to(torch.bfloat16)
    w[3, 0] = 1e30
    w[3, 1:] = torch.linspace(-1e30, 1e30, 63).to(torch.bfloat16)
    quantize_both(w, dev)


def test_fp8_quantize_reports_nonfinite(dev):
    m = nd()
    w = torch.ones((2, 64), dtype=torch.bfloat16, device=dev)
    w[1, 5] = float("inf")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    m.fp8w_quantize(w, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 7


@pytest.mark.parametrize("m_rows", [1, 2, 3, 8, 16])
def test_fp8_gemv_argmax_parity(dev, m_rows):
    m = nd()
    case = workloads.propose_m8(n=3001, k=640, m=m_rows)
    wq, codes, scales = quantize_both(case.w, dev)
    x = case.segments[0][0]
    y, sabs = oracle.fp8_gemv(workloads.bits(x), codes, scales)
    logits, idx = m.fp8w_gemv_argmax([(x.to(dev), None)], wq)
    y32 = m.fp8w_gemv([(x.to(dev), None)], wq)
    torch.cuda.synchronize()
    lg = logits.cpu().numpy()
    tol = TOL_REL * sabs + TOL_ABS
    assert np.all(np.abs(lg.astype(np.float64) - y) <= tol)
    assert np.array_equal(y32.cpu().numpy(), lg)
    for r in range(m_rows):
        i = int(idx[r])
        assert i == oracle.argmax(lg[r].astype(np.float64))
        j = oracle.argmax(y[r])
        order = np.argsort(-y[r], kind="stable")
        second = order[1] if order[0] == j else order[0]
        if y[r, j] - y[r, second] > tol[r, j] + tol[r, second]:
            assert i == j
        else:
            assert y[r, i] >= y[r, j] - tol[r, i] - tol[r, j]


@pytest.mark.parametrize("m_rows", [1, 4])
def test_fp8_gemv_two_rmsnorm_segments_bf16_out(dev, m_rows):
    m = nd()
    case = workloads.fc_combiner(n=300, k_seg=512, m=m_rows)
    wq, codes, scales = quantize_both(case.w, dev)
    (e, ge), (h, gh) = case.segments
    out = m.fp8w_gemv([(e.to(dev), ge.to(dev), 1e-6), (h.to(dev), gh.to(dev), 1e-6)], wq,
                      out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    a = oracle.rmsnorm_concat([(workloads.bits(e), workloads.bits(ge), 1e-6),
                               (workloads.bits(h), workloads.bits(gh), 1e-6)], m_rows)
    y, sabs = oracle.fp8_gemv(a, codes, scales)
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - y) <= TOL_REL * sabs + TOL_ABS + np.abs(y) * 2.0 ** -8)


def test_fp8_gathered_segment_and_prepared_activations(dev):
    """The FP8 path takes the same activation options: a gathered embedding
    row and, from m = 2, the once-per-call activation grid."""
    m = nd()
    g = torch.Generator().manual_seed(78)
    V, H, N = 200, 256, 400
    table = torch.randn((V, H), generator=g).to(torch.bfloat16).to(dev)
    w = (torch.randn((N, H), generator=g) * 0.02).to(torch.bfloat16)
    wq, codes, scales = quantize_both(w, dev)
    idx = torch.tensor([3, 199, 0], dtype=torch.int32, device=dev)
    gamma = (1 + 0.05 * torch.randn(H, generator=g)).to(torch.bfloat16).to(dev)
    for prepare in (True, False):  # the gather is exact on either activation path
        y_g = m.fp8w_gemv([(table, gamma, 1e-6, idx)], wq, prepare=prepare)
        y_k = m.fp8w_gemv([(table[idx.long()].contiguous(), gamma, 1e-6)], wq, prepare=prepare)
        torch.cuda.synchronize()
        assert torch.equal(y_g, y_k)
    a = oracle.rmsnorm_concat([(workloads.bits(table[idx.long()].cpu()), workloads.bits(gamma.cpu()),
                                1e-6)], 3)
    y, sabs = oracle.fp8_gemv(a, codes, scales)
    assert np.all(np.abs(y_g.cpu().numpy().astype(np.float64) - y) <= TOL_REL * sabs + TOL_ABS)


@pytest.mark.parametrize("m_rows,k", [(4, 16384), (8, 16384), (16, 10240), (32, 10240)])
def test_fp8_gemv_wide_batches_at_large_k(dev, m_rows, k):
    from test_gpu_parity import run_wide
    run_wide(dev, m_rows, k, fp8=True)


def test_fp8_quantize_exact_midpoint_ties(dev):
    """Rows whose scale is an exact power of two (row max 448 * 2^e) with
    elements on E4M3 rounding midpoints (normal and subnormal) and one BF16
    ulp either side."""
    grid = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    mids = ((grid[1:] + grid[:-1]) / 2)
    mids = mids[mids.to(torch.bfloat16).double().eq(mids)]   # the midpoints BF16 holds exactly
    assert len(mids) > 40
    rows = []
    for e in (-20, -4, 0, 3):
        for sign in (1.0, -1.0):
            r = torch.zeros(128, dtype=torch.float64)
            r[0] = 448.0
            r[1:1 + len(mids)] = sign * mids[:127]
            rows.append(r * 2.0 ** e)
    wb = torch.stack(rows).to(torch.bfloat16)
    assert wb.double().eq(torch.stack(rows)).all()
    bits = wb.view(torch.int16)
    nz = (bits & 0x7FFF) != 0                              # zeros stay zeros
    up = torch.where(nz, bits + 1, bits).view(torch.bfloat16)  # one BF16 ulp either side
    down = torch.where(nz, bits - 1, bits).view(torch.bfloat16)
    up[:, 0], down[:, 0] = wb[:, 0], wb[:, 0]              # keep each row's maximum
    quantize_both(torch.cat([wb, up, down]), dev)


def near_tie_rows(k=256):
    """One row per row maximum A in [1, 2) (every BF16 value there): elements x
    whose quotient fl32(x / s) falls within two binary32 ulps of an E4M3
    rounding midpoint while x / s is not the midpoint (s = fl32(A / 448)
    inexact), with their negations; the row's codes then hang on the
    correctly rounded quotient."""
    v = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    mids = (v[1:] + v[:-1]) / 2
    rows, hits = [], 0
    for a in torch.arange(0x3F80, 0x4000, dtype=torch.int16).view(torch.bfloat16).float().numpy():
        s = np.float32(a) / np.float32(448)
        near = torch.from_numpy(mids * float(s)).to(torch.bfloat16).view(torch.int16)
        row = [float(a)]
        for off in (-1, 0, 1):
            x = (near + off).view(torch.bfloat16).float().numpy()
            q = (x / s).astype(np.float32)
            ul = np.spacing(mids.astype(np.float32)).astype(np.float64)
            hit = ((np.abs(q.astype(np.float64) - mids) <= 2 * ul)
                   & (x.astype(np.float64) != mids * float(s)) & (x <= a))
            for i in np.nonzero(hit)[0]:
                row += [float(x[i]), -float(x[i])]
        hits += (len(row) - 1) // 2
        row = row[:k] + [0.0] * max(0, k - len(row))
        rows.append(row)
    return torch.tensor(rows, dtype=torch.float32).to(torch.bfloat16), hits


def test_fp8_quantize_near_tie_quotients(dev):
    """Codes where the quotient's binary32 rounding lands on or next to an
    E4M3 midpoint (double rounding): each must equal the oracle's."""
    w, hits = near_tie_rows()
    assert hits > 500, "the construction should find many near-tie quotients"
    quantize_both(w, dev)
