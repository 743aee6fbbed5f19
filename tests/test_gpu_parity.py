"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Bar (stated per test):
  * packed codes, scale bytes, absmax, g: bit-exact;
  * FP32 logits: |gpu - oracle| <= 1e-3 * S + 1e-6, S = sum |a_i w_i|;
  * BF16 outputs: the same plus one BF16 ulp of the oracle value;
  * argmax: equal to the first maximum of the GPU's own FP32 logits (same
    precision), and equal to the oracle's index whenever the oracle's top-2
    gap exceeds both tolerances, else inside the oracle's near-max set.
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


def upload_weight(packed, scales, g, dev):
    m = nd()
    n, kh = packed.shape
    return m.Nvfp4Weight(torch.from_numpy(packed).to(dev), torch.from_numpy(scales).to(dev),
                         torch.tensor([g], dtype=torch.float32, device=dev), n, kh * 2)


def quantize_both(w_bf16, dev):
    """GPU quantisation checked bit-exact against the oracle's."""
    m = nd()
    wq, amax = m.nvfp4_quantize(w_bf16.to(dev).contiguous())
    p, s, g, a = oracle.quantize(workloads.bits(w_bf16))
    torch.cuda.synchronize()
    assert amax.item() == float(a), "absmax differs"
    assert wq.global_scale.item() == float(g), "global scale differs"
    gp, gs = wq.packed.cpu().numpy(), wq.scales.cpu().numpy()
    if not np.array_equal(gs, s):
        bad = np.argwhere(gs != s)[:5]
        raise AssertionError(f"scale bytes differ at {bad.tolist()}: gpu {gs[tuple(bad[0])]} "
                             f"oracle {s[tuple(bad[0])]}")
    if not np.array_equal(gp, p):
        bad = np.argwhere(gp != p)[:5]
        raise AssertionError(f"packed codes differ at {bad.tolist()}")
    return wq, (p, s, g)


def oracle_input(segments, eps_default=1e-6):
    m = segments[0][0].shape[0]
    return oracle.rmsnorm_concat(
        [(workloads.bits(x), None if gm is None else workloads.bits(gm), eps_default)
         for x, gm in segments], m)


def check_logits(got, y, sabs):
    err = np.abs(got.astype(np.float64) - y)
    tol = TOL_REL * sabs + TOL_ABS
    bad = np.argwhere(err > tol)
    assert bad.size == 0, (f"{len(bad)} logits out of tolerance, first {bad[0].tolist()}: "
                           f"gpu {got[tuple(bad[0])]} oracle {y[tuple(bad[0])]} tol {tol[tuple(bad[0])]}")


def check_argmax(idx, logits_gpu, y, sabs):
    tol = TOL_REL * sabs + TOL_ABS
    for r in range(y.shape[0]):
        i = int(idx[r])
        assert i == oracle.argmax(logits_gpu[r].astype(np.float64)), "not the first max of GPU logits"
        j = oracle.argmax(y[r])
        order = np.argsort(-y[r], kind="stable")
        second = order[1] if order[0] == j else order[0]
        if y[r, j] - y[r, second] > tol[r, j] + tol[r, second]:
            assert i == j, f"row {r}: gpu argmax {i}, oracle {j}"
        else:
            assert y[r, i] >= y[r, j] - tol[r, j] - tol[r, i]


def run_gemv_case(case, dev, m_rows=None, with_bf16=False):
    m = nd()
    p, s, g, _ = oracle.quantize(workloads.bits(case.w))
    wq = upload_weight(p, s, g, dev)
    segs = [(x if m_rows is None else x[:m_rows], gm) for x, gm in case.segments]
    a = oracle_input(segs, case.eps)
    y, sabs = oracle.gemv(a, p, s, g)
    dsegs = [(x.to(dev), None if gm is None else gm.to(dev), case.eps) for x, gm in segs]
    logits, idx = m.w4a16_gemv_argmax(dsegs, wq)
    y32 = m.w4a16_gemv(dsegs, wq)
    torch.cuda.synchronize()
    lg = logits.cpu().numpy()
    check_logits(lg, y, sabs)
    assert np.array_equal(y32.cpu().numpy(), lg), "w4a16_gemv and w4a16_gemv_argmax logits differ"
    check_argmax(idx.cpu().numpy(), lg, y, sabs)
    if with_bf16:
        yb = m.w4a16_gemv(dsegs, wq, out_dtype=torch.bfloat16)
        got = yb.float().cpu().numpy().astype(np.float64)
        ulp = np.abs(y) * 2.0 ** -8
        err = np.abs(got - y)
        assert np.all(err <= TOL_REL * sabs + TOL_ABS + ulp)
    return lg, idx.cpu().numpy(), y


# ---------------------------------------------------------------- quantiser

@pytest.mark.parametrize("n,k", [(256, 512), (1, 32), (3, 96), (37, 160), (129, 4096)])
def test_quantize_bit_exact_shapes(dev, n, k):
    quantize_both(workloads.tiny(n=n, k=k).w, dev)


def test_quantize_bit_exact_wide_block_range(dev):
    quantize_both(workloads.propose_m8(n=512, k=1024).w, dev)


def test_quantize_outlier_rows(dev):
    quantize_both(workloads.lm_head_m1(n=1000, k=512, rows=1).w, dev)


def test_quantize_special_values(dev):
    rng = np.random.default_rng(7)
    x = rng.standard_normal((64, 128)).astype(np.float32) * 0.02
    x[0, :16] = 0.0                                        # zero block
    x[1, :] = -0.0                                         # negative zeros
    x[2, :16] = 1e-30                                      # subnormal-scale block
    x[3, 16:32] = 1.0                                      # constant block
    x[4, :] = np.linspace(-5, 5, 128)                      # ties after scaling
    x[5, 7] = 300.0                                        # dominant element: most scales tiny
    w = torch.from_numpy(x).to(torch.bfloat16)
    w.view(torch.int16)[1] = -32768                        # exact -0.0 bit pattern
    w.view(torch.int16)[6, 3] = -32768                     # -0.0 inside a non-zero block: code 0x8
    quantize_both(w, dev)
    quantize_both(torch.zeros((8, 64), dtype=torch.bfloat16), dev)
    big = torch.full((4, 32), 3.3e38).to(torch.bfloat16)
    big[1] = -big[1]
    quantize_both(big, dev)


def test_quantize_exactly_representable_round_trip(dev):
    rng = np.random.default_rng(8)
    n, k = 16, 64
    codes = rng.integers(0, 16, size=(n, k))
    codes.reshape(n, -1, 16)[:, :, 3] = 7
    sc = rng.integers(0x10, 0x7E, size=(n, k // 16))
    sc[0, 0] = 0x7E
    val = np.vectorize(oracle.e2m1_value)(codes) * np.repeat(np.vectorize(oracle.e4m3_value)(sc), 16, 1)
    w = torch.from_numpy(val * 2.0 ** -12).to(torch.bfloat16)
    wq, (p, s, g) = quantize_both(w, dev)
    assert np.array_equal(s, sc.astype(np.uint8))


def test_quantize_nonfinite_is_reported(dev):
    m = nd()
    w = torch.ones((4, 64), dtype=torch.bfloat16)
    w[2, 5] = float("inf")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    m.nvfp4_quantize(w.to(dev), dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 7  # NVFP4_ERR_NONFINITE


# --------------------------------------------------------------------- GEMV

@pytest.mark.parametrize("m_rows", [1, 2, 3, 4, 5, 8])
def test_gemv_small_all_batch_widths(dev, m_rows):
    run_gemv_case(workloads.propose_m8(n=1000, k=640, m=8), dev, m_rows=m_rows)


@pytest.mark.parametrize("m_rows", [9, 12, 16])
def test_gemv_two_column_groups(dev, m_rows):
    """9..16 batch rows: two MMA column groups share each dequantised weight
    fragment; logits, BF16 output and argmax against the oracle, for both
    activation paths (once per call, per CTA)."""
    run_gemv_case(workloads.propose_m8(n=1100, k=768, m=16), dev, m_rows=m_rows, with_bf16=True)
    m = nd()
    case = workloads.fc_combiner(n=300, k_seg=1024, m=16)
    p, s, g, _ = oracle.quantize(workloads.bits(case.w))
    wq = upload_weight(p, s, g, dev)
    (e, ge), (h, gh) = case.segments
    segs = [(e[:m_rows].contiguous().to(dev), ge.to(dev), 1e-6), (h[:m_rows].contiguous().to(dev), gh.to(dev), 1e-6)]
    a = oracle.rmsnorm_concat([(workloads.bits(e[:m_rows]), workloads.bits(ge), 1e-6),
                               (workloads.bits(h[:m_rows]), workloads.bits(gh), 1e-6)], m_rows)
    y, sabs = oracle.gemv(a, p, s, g)
    for prepare in (True, False):
        out = m.w4a16_gemv(segs, wq, prepare=prepare)
        torch.cuda.synchronize()
        check_logits(out.cpu().numpy(), y, sabs)


def run_wide(dev, m_rows, k, fp8):
    """RMSNorm + GEMV + argmax for wide batches at large k, on a ragged number
    of weight rows: batches whose activations do not fit one CTA's shared
    memory (and every batch over 16 rows) run as consecutive row blocks, each
    against the oracle.  Then the refusals: k past W4A16_GEMV_MAX_K and m past
    W4A16_GEMV_MAX_M."""
    m = nd()
    g = torch.Generator().manual_seed(m_rows * 100000 + k)
    n = 70
    w = (torch.randn((n, k), generator=g) * 0.02).to(torch.bfloat16)
    x = torch.randn((m_rows, k), generator=g).to(torch.bfloat16)
    gamma = (1 + 0.05 * torch.randn(k, generator=g)).to(torch.bfloat16)
    a = oracle.rmsnorm_concat([(workloads.bits(x), workloads.bits(gamma), 1e-6)], m_rows)
    if fp8:
        codes, scales = oracle.fp8_quantize(workloads.bits(w))
        wq = m.Fp8Weight(torch.from_numpy(codes).to(dev), torch.from_numpy(scales).to(dev), n, k)
        y, sabs = oracle.fp8_gemv(a, codes, scales)
        gemv, gemv_argmax, quantize = m.fp8w_gemv, m.fp8w_gemv_argmax, m.fp8w_quantize
    else:
        p, s, gs, _ = oracle.quantize(workloads.bits(w))
        wq = upload_weight(p, s, gs, dev)
        y, sabs = oracle.gemv(a, p, s, gs)
        gemv, gemv_argmax = m.w4a16_gemv, m.w4a16_gemv_argmax
        quantize = lambda t: m.nvfp4_quantize(t)[0]  # noqa: E731
    segs = [(x.to(dev), gamma.to(dev), 1e-6)]
    logits, idx = gemv_argmax(segs, wq)
    yb = gemv(segs, wq, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    lg = logits.cpu().numpy()
    check_logits(lg, y, sabs)
    check_argmax(idx.cpu().numpy(), lg, y, sabs)
    got = yb.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - y) <= TOL_REL * sabs + TOL_ABS + np.abs(y) * 2.0 ** -8)
    kk = m.GEMV_MAX_K + 32
    w2 = quantize(torch.zeros((32, kk), dtype=torch.bfloat16, device=dev))
    x2 = torch.zeros((m_rows, kk), dtype=torch.bfloat16, device=dev)
    with pytest.raises(m.Nvfp4Error) as e:
        gemv([(x2, None)], w2)
    assert e.value.status == 2  # NVFP4_ERR_SHAPE
    x3 = torch.zeros((m.GEMV_MAX_M + 1, k), dtype=torch.bfloat16, device=dev)
    with pytest.raises(m.Nvfp4Error) as e:
        gemv([(x3, None)], wq)
    assert e.value.status == 2


@pytest.mark.parametrize("m_rows,k", [(5, 16384), (8, 16384), (16, 10240), (16, 5120), (24, 5120),
                                        (32, 5120), (32, 10240)])
def test_gemv_wide_batches_at_large_k(dev, m_rows, k):
    run_wide(dev, m_rows, k, fp8=False)


@pytest.mark.parametrize("n,k", [(16, 32), (17, 64), (100, 96), (257, 224), (2003, 1056)])
def test_gemv_ragged_shapes(dev, n, k):
    run_gemv_case(workloads.propose_m8(n=n, k=k, m=3), dev, with_bf16=True)


def test_gemv_tiny_config(dev):
    run_gemv_case(workloads.tiny(), dev)


def test_gemv_rmsnorm_fused(dev):
    run_gemv_case(workloads.lm_head_m1(n=3000, k=1024, rows=4), dev)


@pytest.mark.parametrize("n,k", [(24437, 2048), (16 * 152 * 9 + 3, 1024)])
def test_gemv_m1_split_k_over_many_tiles(dev, n, k):
    """M = 1 with 10 and 11 tiles per CTA on 152 SMs: whole tiles as contiguous
    runs over 16 warps with the idle warps between busy ones; ragged last tile
    and a last CTA with fewer tiles."""
    run_gemv_case(workloads.lm_head_m1(n=n, k=k, rows=1), dev)


def test_gemv_two_segment_concat_bf16_out(dev):
    run_gemv_case(workloads.fc_combiner(n=640, k_seg=512, m=5), dev, with_bf16=True)


def test_gemv_strided_activations(dev):
    m = nd()
    case = workloads.propose_m8(n=300, k=256, m=4)
    p, s, g, _ = oracle.quantize(workloads.bits(case.w))
    wq = upload_weight(p, s, g, dev)
    x = case.segments[0][0]
    big = torch.zeros((4, 264), dtype=torch.bfloat16)
    big[:, :256] = x
    y, sabs = oracle.gemv(workloads.bits(x), p, s, g)
    out = torch.full((4, 320), float("nan"), device=dev)
    m.w4a16_gemv([(big.to(dev)[:, :256], None)], wq, out=out[:, :300])
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    check_logits(o[:, :300], y, sabs)
    assert np.all(np.isnan(o[:, 300:])), "wrote outside the output rows"


@pytest.mark.parametrize("m_rows,n,k1,k2", [(2, 300, 1056, 0), (3, 1000, 512, 544), (8, 257, 2048, 1024)])
def test_prepared_activations_match_in_kernel_prologue(dev, m_rows, n, k1, k2):
    """The once-per-call activation grid (large workspace) and the per-CTA
    prologue (small or no workspace) both match the oracle.  (Their sums of
    squares may add partials in different orders, so the two are compared to
    the oracle, not to each other bit for bit.)"""
    m = nd()
    g = torch.Generator().manual_seed(n + k1 + k2)
    k = k1 + k2
    w = (torch.randn((n, k), generator=g) * 0.02).to(torch.bfloat16)
    wq, _ = m.nvfp4_quantize(w.to(dev))
    segs = []
    for ks in (k1, k2):
        if ks == 0:
            continue
        x = (torch.randn((m_rows, ks + 16), generator=g) * 3).to(torch.bfloat16)[:, 8:8 + ks]
        gamma = (1 + 0.05 * torch.randn(ks, generator=g)).to(torch.bfloat16)
        segs.append((x.to(dev), gamma.to(dev), 1e-6))
    big = torch.zeros(m.gemv_workspace_bytes(m_rows, k), dtype=torch.uint8, device=dev)
    small = torch.zeros(m.ARGMAX_WS_BYTES, dtype=torch.uint8, device=dev)
    lg_p, idx_p = m.w4a16_gemv_argmax(segs, wq, workspace=big)
    lg_k, idx_k = m.w4a16_gemv_argmax(segs, wq, workspace=small)
    y_p = m.w4a16_gemv(segs, wq, out_dtype=torch.bfloat16, workspace=big)
    y_k = m.w4a16_gemv(segs, wq, out_dtype=torch.bfloat16, prepare=False)
    torch.cuda.synchronize()
    a = oracle.rmsnorm_concat([(workloads.bits(x.cpu()), workloads.bits(gm.cpu()), e) for x, gm, e in segs],
                              m_rows)
    y, sabs = oracle.gemv(a, wq.packed.cpu().numpy(), wq.scales.cpu().numpy(),
                          np.float32(wq.global_scale.item()))
    for lg, idx in ((lg_p, idx_p), (lg_k, idx_k)):
        check_logits(lg.cpu().numpy(), y, sabs)
        check_argmax(idx.cpu().numpy(), lg.cpu().numpy(), y, sabs)
    for yb in (y_p, y_k):
        got = yb.float().cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - y) <= TOL_REL * sabs + TOL_ABS + np.abs(y) * 2.0 ** -8)


def test_argmax_ties_pick_lowest_index(dev):
    m = nd()
    case = workloads.propose_m8(n=700, k=256, m=2)
    p, s, g, _ = oracle.quantize(workloads.bits(case.w))
    x = case.segments[0][0]
    y, _ = oracle.gemv(workloads.bits(x), p, s, g)
    for r in range(2):
        j = oracle.argmax(y[r])
        lo = 5 if j > 5 else j + 1
        hi = 650 if j < 650 else j - 1
        p2, s2 = p.copy(), s.copy()
        for tgt in (lo, hi):
            p2[tgt], s2[tgt] = p[j], s[j]
        wq = upload_weight(p2, s2, g, dev)
        logits, idx = m.w4a16_gemv_argmax([(x.to(dev), None)], wq)
        torch.cuda.synchronize()
        lg = logits.cpu().numpy()
        assert lg[r, lo] == lg[r, j] == lg[r, hi], "duplicated rows must give bit-equal logits"
        assert idx[r].item() == min(lo, j, hi)


def test_argmax_workspace_returns_to_zero_and_repeats(dev):
    m = nd()
    case = workloads.tiny(n=512, k=256, m=3)
    p, s, g, _ = oracle.quantize(workloads.bits(case.w))
    wq = upload_weight(p, s, g, dev)
    ws = torch.zeros(m.ARGMAX_WS_BYTES, dtype=torch.uint8, device=dev)
    x = case.segments[0][0].to(dev)
    outs = []
    for _ in range(3):
        _, idx = m.w4a16_gemv_argmax([(x, None)], wq, logits=False, workspace=ws)
        outs.append(idx.cpu().numpy())
    torch.cuda.synchronize()
    assert not ws.any().item()
    assert all(np.array_equal(o, outs[0]) for o in outs)
    y, sabs = oracle.gemv(workloads.bits(case.segments[0][0]), p, s, g)
    logits, _ = m.w4a16_gemv_argmax([(x, None)], wq, workspace=ws)
    torch.cuda.synchronize()
    check_argmax(outs[0], logits.cpu().numpy(), y, sabs)


def test_argmax_all_negative_infinity_and_nan_logits(dev):
    # a zero weight gives y = 0 everywhere: the first index wins
    m = nd()
    wq = upload_weight(np.zeros((64, 32), np.uint8), np.zeros((64, 4), np.uint8), 1.0, dev)
    x = torch.ones((1, 64), dtype=torch.bfloat16, device=dev)
    _, idx = m.w4a16_gemv_argmax([(x, None)], wq, logits=False)
    torch.cuda.synchronize()
    assert idx.item() == 0


# --------------------------------------------------------------------- GEMM

def check_gemm(a, wq_oracle, c_gpu, rows, cols):
    p, s, g = wq_oracle
    exact, sabs = oracle.gemm_pairs(workloads.bits(a), p, s, g, rows, cols)
    got = c_gpu[rows, cols].astype(np.float64)
    ulp = np.abs(exact) * 2.0 ** -8
    err = np.abs(got - exact)
    bad = np.nonzero(err > TOL_REL * sabs + TOL_ABS + ulp)[0]
    assert bad.size == 0, f"{bad.size} outputs off, first ({rows[bad[0]]},{cols[bad[0]]}): " \
                          f"gpu {got[bad[0]]} oracle {exact[bad[0]]}"


@pytest.mark.parametrize("staged", [False, True], ids=["bf16", "f16_staged"])
@pytest.mark.parametrize("m_rows,n,k", [(128, 128, 64), (200, 256, 320), (1, 384, 128),
                                        (257, 128, 1024)])
def test_gemm_small_all_outputs(dev, m_rows, n, k, staged):
    m = nd()
    case = workloads.prefill_gemm(m=m_rows, n=n, k=k)
    p, s, g, _ = oracle.quantize(workloads.bits(case.w))
    wq = upload_weight(p, s, g, dev)
    ws = (torch.empty(m.gemm_workspace_bytes(m_rows, k), dtype=torch.uint8, device=dev)
          if staged else None)
    c = m.w4a16_gemm(case.a.to(dev), wq, workspace=ws)
    torch.cuda.synchronize()
    cg = c.float().cpu().numpy()
    rows = np.repeat(np.arange(m_rows), n)
    cols = np.tile(np.arange(n), m_rows)
    check_gemm(case.a, (p, s, g), cg, rows, cols)


def test_gemm_strided_output(dev):
    m = nd()
    case = workloads.prefill_gemm(m=130, n=256, k=192)
    p, s, g, _ = oracle.quantize(workloads.bits(case.w))
    wq = upload_weight(p, s, g, dev)
    out = torch.full((130, 264), float("nan"), dtype=torch.bfloat16, device=dev)
    m.w4a16_gemm(case.a.to(dev), wq, out=out[:, :256])
    torch.cuda.synchronize()
    o = out.float().cpu().numpy()
    assert np.all(np.isnan(o[:, 256:]))
    rows = np.repeat(np.arange(130), 256)
    cols = np.tile(np.arange(256), 130)
    check_gemm(case.a, (p, s, g), o, rows, cols)


def test_gemm_staged_rows_of_very_different_scales(dev):
    """Rows whose magnitudes differ by up to 2^60: each row gets its own FP16
    staging scale, so both paths stay within tolerance of the oracle."""
    m = nd()
    case = workloads.prefill_gemm(m=130, n=256, k=192)
    a = case.a.float()
    a *= torch.exp2(torch.linspace(-30, 30, 130)).unsqueeze(1)
    a = a.to(torch.bfloat16)
    a[7] = 0
    p, s, g, _ = oracle.quantize(workloads.bits(case.w))
    wq = upload_weight(p, s, g, dev)
    rows = np.repeat(np.arange(130), 256)
    cols = np.tile(np.arange(256), 130)
    for staged in (False, True):
        ws = (torch.empty(m.gemm_workspace_bytes(130, 192), dtype=torch.uint8, device=dev)
              if staged else None)
        c = m.w4a16_gemm(a.to(dev), wq, workspace=ws)
        torch.cuda.synchronize()
        check_gemm(a, (p, s, g), c.float().cpu().numpy(), rows, cols)


def test_quantize_exact_midpoint_ties(dev):
    """Quotients that land exactly on E2M1 rounding midpoints (ties to even)
    and one BF16 ulp either side: g = 2^e exactly (global max 2688 * 2^e) and
    block scales on the E4M3 grid make every quotient exact."""
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    rows = []
    for e in (-12, -3, 0):
        for s in (448.0, 288.0, 40.0, 0.875):
            for sign in (1.0, -1.0):
                blk = [6.0 * s] + [sign * m * s for m in mids] + [sign * m * s for m in mids] + [0.0]
                rows.append([v * 2.0 ** e for v in blk])
    w = torch.tensor(rows, dtype=torch.float64)
    wb = w.to(torch.bfloat16)
    assert wb.double().eq(w).all()                        # the ties are exact in BF16
    bits = wb.view(torch.int16)
    nz = (bits & 0x7FFF) != 0                              # zeros stay zeros
    up = torch.where(nz, bits + 1, bits).view(torch.bfloat16)  # one BF16 ulp either side
    down = torch.where(nz, bits - 1, bits).view(torch.bfloat16)
    up[:, 0], down[:, 0] = wb[:, 0], wb[:, 0]              # keep each block's maximum
    blocks = torch.cat([wb, up, down, torch.zeros_like(wb)], dim=1)
    blocks[0, 63] = 2688.0  # the global maximum: g = 2688 / 2688 = 1 exactly
    quantize_both(blocks, dev)


def near_tie_blocks(amax):
    """Blocks whose quotients fl32(x / d) fall within two binary32 ulps of an
    E2M1 rounding midpoint while x / d itself is not the midpoint (d = fl32(
    dec(s) * g) with g = fl32(amax / 2688) inexact), plus the global maximum:
    there the correctly rounded quotient, not the exact one, decides the code.
    Each block holds its scale-setting maximum, the near-tie element and its
    negation."""
    g = np.float32(amax) / np.float32(2688)
    dec = torch.arange(1, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    d = (dec * g).astype(np.float32)
    blocks = []
    for mid in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0):
        near = torch.from_numpy(mid * d.astype(np.float64)).to(torch.bfloat16).view(torch.int16)
        for off in (-2, -1, 0, 1, 2):
            x = (near + off).view(torch.bfloat16).float().numpy()
            q = (x / d).astype(np.float32)
            hit = ((np.abs(q.astype(np.float64) - mid) <= 2 * np.spacing(np.float32(mid)))
                   & (x.astype(np.float64) != mid * d.astype(np.float64)))
            for i in np.nonzero(hit)[0]:
                bmax = float(torch.tensor(6.0 * float(d[i])).to(torch.bfloat16))
                blocks.append([bmax, float(x[i]), -float(x[i])] + [0.0] * 13)
    blocks.append([amax] + [0.0] * 15)
    if len(blocks) % 2:
        blocks.append([0.0] * 16)
    return torch.tensor(blocks, dtype=torch.float32).view(-1, 32).to(torch.bfloat16), len(blocks)


@pytest.mark.parametrize("amax", [1.0, 1.03125, 1.453125, 1.78125])
def test_quantize_near_tie_quotients(dev, amax):
    """Codes where the quotient's binary32 rounding lands on or next to an
    E2M1 midpoint (double rounding): each must equal the oracle's."""
    w, nblk = near_tie_blocks(amax)
    assert nblk > 100, "the construction should find many near-tie quotients"
    assert float(w.float().abs().max()) == amax
    quantize_both(w, dev)


def test_quantize_scale_array_at_odd_address(dev):
    """The scale array may start at any byte: an odd start takes the
    byte-wise scale stores, with the same bytes as the oracle's and the bytes
    around the array untouched."""
    import ctypes
    m = nd()
    w = workloads.propose_m8(n=300, k=512).w
    p, s, g, _ = oracle.quantize(workloads.bits(w))
    n, k = w.shape
    wd = w.to(dev).contiguous()
    packed = torch.empty((n, k // 2), dtype=torch.uint8, device=dev)
    buf = torch.full((n * (k // 16) + 2,), 0xA5, dtype=torch.uint8, device=dev)
    gs = torch.empty(1, dtype=torch.float32, device=dev)
    amax = torch.empty(1, dtype=torch.float32, device=dev)
    ex = m._exec(None, None, None, dev)
    rc = m.load().nvfp4_quantize(wd.data_ptr(), n, k, packed.data_ptr(), buf.data_ptr() + 1,
                                 gs.data_ptr(), amax.data_ptr(), ctypes.byref(ex))
    assert rc == 0
    torch.cuda.synchronize()
    got = buf.cpu().numpy()
    assert got[0] == 0xA5 and got[-1] == 0xA5
    assert np.array_equal(got[1:-1].reshape(s.shape), s)
    assert np.array_equal(packed.cpu().numpy(), p)
    assert gs.item() == float(g)


def test_quantize_repeatable_at_full_size(dev):
    """The 17408 x 5120 weight quantised eight times (half of them after an L2
    flush) gives the same bytes every time, equal to the oracle on sampled
    rows: the staged pass's ring turns over thousands of times, so a stage
    read before its copy lands, or refilled before its readers are done,
    shows up as differing blocks."""
    m = nd()
    case = workloads.prefill_gemm(m=16, device=dev)
    first, _ = m.nvfp4_quantize(case.w)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for i in range(8):
        if i % 2:
            flush.fill_(i)
        wq, _ = m.nvfp4_quantize(case.w)
        torch.cuda.synchronize()
        assert torch.equal(wq.scales, first.scales), f"run {i}: scale bytes differ between runs"
        assert torch.equal(wq.packed, first.packed), f"run {i}: codes differ between runs"
    wb = workloads.bits(case.w)
    rows = np.random.default_rng(5).choice(wb.shape[0], 256, replace=False)
    g = oracle.global_scale(oracle.global_absmax(wb))
    for r in rows[:64]:
        p, s = oracle.quantize_rows(wb, np.array([r]), g)
        assert np.array_equal(first.scales[int(r)].cpu().numpy(), s[0])
        assert np.array_equal(first.packed[int(r)].cpu().numpy(), p[0])


@pytest.mark.parametrize("m_rows,n,k,width", [(2048, 4864, 128, 256), (300, 512, 256, 240)])
def test_gemm_both_tile_widths(dev, m_rows, n, k, width):
    """The GEMM picks 256- or 240-wide tiles by the waves they fill (whole
    waves of one CTA per SM, each tile costed as its width + 16).  2048 x 4864
    is 152 tiles of 256 (one wave) and takes 256; 300 x 512 takes 240, whose
    last tile holds 32 valid columns.  A full output row in every 256-row M
    tile, a full column in every tile of the chosen width, and random samples
    against the oracle."""
    m = nd()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mt = -(-m_rows // 256)
    cost = {bn: -(-(mt * -(-n // bn)) // sms) * (bn + 16) for bn in (256, 240)}
    if (240 if cost[240] < cost[256] else 256) != width:
        pytest.skip(f"on {sms} SMs this shape does not select the {width}-wide tiles")
    case = workloads.prefill_gemm(m=m_rows, n=n, k=k)
    p, s, g, _ = oracle.quantize(workloads.bits(case.w))
    wq = upload_weight(p, s, g, dev)
    c = m.w4a16_gemm(case.a.to(dev), wq)
    torch.cuda.synchronize()
    cg = c.float().cpu().numpy()
    rng = np.random.default_rng(width)
    full_rows = np.minimum(256 * np.arange(mt) + rng.integers(0, 256, mt), m_rows - 1)
    nt = -(-n // width)
    full_cols = np.minimum(width * np.arange(nt) + rng.integers(0, width, nt), n - 1)
    full_cols = np.concatenate([full_cols, [n - 1]])
    rows = np.concatenate([rng.integers(0, m_rows, 4096), np.repeat(full_rows, n),
                           np.tile(np.arange(m_rows), full_cols.size)])
    cols = np.concatenate([rng.integers(0, n, 4096), np.tile(np.arange(n), full_rows.size),
                           np.repeat(full_cols, m_rows)])
    check_gemm(case.a, (p, s, g), cg, rows, cols)
