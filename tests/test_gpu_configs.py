"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times, against the CPU oracle (run on all host cores from here; the
oracle's own code is unchanged).  Where the oracle cannot cover every output
in seconds, outputs are sampled (seeded) and checked one by one.

Bars as in test_gpu_parity: codes/scales/absmax/g bit-exact; FP32 logits
within 1e-3 * S + 1e-6; BF16 outputs the same plus one BF16 ulp; argmax equal
to the first maximum of the GPU's own logits and to the oracle's index when
the oracle's top-2 gap exceeds the tolerances.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

TOL_REL, TOL_ABS = 1e-3, 1e-6
THREADS = max(1, min(32, os.cpu_count() or 1))


def nd():
    import nvfp4_speculative_draft_gb300 as m
    return m


def par_quantize_rows(wb, rows, g):
    chunks = np.array_split(np.asarray(rows), THREADS)
    with ThreadPoolExecutor(THREADS) as ex:
        parts = list(ex.map(lambda r: oracle.quantize_rows(wb, r, g), [c for c in chunks if len(c)]))
    return np.concatenate([p for p, _ in parts]), np.concatenate([s for _, s in parts])


def par_gemv(a, packed, scales, g):
    n = packed.shape[0]
    bounds = np.linspace(0, n, THREADS + 1).astype(int)
    jobs = [(bounds[i], bounds[i + 1] - bounds[i]) for i in range(THREADS) if bounds[i + 1] > bounds[i]]
    with ThreadPoolExecutor(THREADS) as ex:
        res = list(ex.map(lambda j: oracle.gemv(a, packed, scales, g, n0=j[0], nn=j[1]), jobs))
    return np.concatenate([y for y, _ in res], axis=1), np.concatenate([s for _, s in res], axis=1)


def check_gpu_quant(wq, amax, wb, sample_rows=None):
    """GPU quantisation vs the oracle: absmax and g exactly, then every row
    (or the sampled rows) bit-exact."""
    a_ref = oracle.global_absmax(wb)
    g_ref = oracle.global_scale(a_ref)
    assert amax.item() == a_ref
    assert wq.global_scale.item() == float(g_ref)
    rows = np.arange(wb.shape[0]) if sample_rows is None else np.asarray(sample_rows)
    p_ref, s_ref = par_quantize_rows(wb, rows, g_ref)
    gp = wq.packed[torch.from_numpy(rows).to(wq.packed.device)].cpu().numpy()
    gs = wq.scales[torch.from_numpy(rows).to(wq.scales.device)].cpu().numpy()
    assert np.array_equal(gs, s_ref), "scale bytes differ"
    assert np.array_equal(gp, p_ref), "packed codes differ"
    return g_ref


def check_logits_and_argmax(lg, idx, y, sabs):
    err = np.abs(lg.astype(np.float64) - y)
    tol = TOL_REL * sabs + TOL_ABS
    assert np.all(err <= tol), f"{int((err > tol).sum())} logits out of tolerance"
    for r in range(y.shape[0]):
        i = int(idx[r])
        assert i == oracle.argmax(lg[r].astype(np.float64))
        j = oracle.argmax(y[r])
        top = np.partition(-y[r], 1)[:2]
        if (-top[0]) - (-top[1]) > 2 * tol[r].max():
            assert i == j
        else:
            assert y[r, i] >= y[r, j] - tol[r, j] - tol[r, i]


def half_mask(m_rows, n, seed):
    """Grammar bitmask words [m, ceil(n/32)] with about half the tokens allowed."""
    rng = np.random.default_rng(seed)
    return rng.integers(-2 ** 31, 2 ** 31, size=(m_rows, (n + 31) // 32), dtype=np.int64).astype(np.int32)


def mask_bits(words, n):
    b = words.view(np.uint32)
    j = np.arange(n)
    return ((b[j // 32] >> (j % 32).astype(np.uint32)) & 1).astype(bool)


def lse64(v):
    v = np.asarray(v, dtype=np.float64)
    mx = v.max()
    return mx + np.log(np.exp(v - mx).sum())


def test_tiny_config(dev):
    m = nd()
    case = workloads.tiny()
    wq, amax = m.nvfp4_quantize(case.w.to(dev))
    wb = workloads.bits(case.w)
    g = check_gpu_quant(wq, amax, wb)
    x = case.segments[0][0]
    logits, idx = m.w4a16_gemv_argmax([(x.to(dev), None)], wq)
    torch.cuda.synchronize()
    y, sabs = oracle.gemv(workloads.bits(x), wq.packed.cpu().numpy(), wq.scales.cpu().numpy(), g)
    check_logits_and_argmax(logits.cpu().numpy(), idx.cpu().numpy(), y, sabs)


def test_lm_head_config_full(dev):
    """32768 x 4096 reduced-vocab head with 1% outlier rows; RMSNorm + GEMV +
    argmax at M=1 for three of the seeded hidden rows."""
    m = nd()
    case = workloads.lm_head_m1(rows=3, device=dev)
    wq, amax = m.nvfp4_quantize(case.w)
    wb = workloads.bits(case.w)
    g = check_gpu_quant(wq, amax, wb)
    h, gamma = case.segments[0]
    pk, sc = wq.packed.cpu().numpy(), wq.scales.cpu().numpy()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for r in range(3):
        logits, idx = m.w4a16_gemv_argmax([(h[r:r + 1], gamma, 1e-6)], wq, dev_status=status)
        torch.cuda.synchronize()
        assert status.item() == 0  # no bounded wait ran out, no index reported
        a = oracle.rmsnorm_concat([(workloads.bits(h[r:r + 1]), workloads.bits(gamma), 1e-6)], 1)
        y, sabs = par_gemv(a, pk, sc, g)
        check_logits_and_argmax(logits.cpu().numpy(), idx.cpu().numpy(), y, sabs)


def test_propose_config_full_width(dev):
    """151936 x 5120 head: quantiser on sampled rows; M = 1, 2, 4, 8 logits
    over every row and the argmax against the oracle; grammar mask + top-1
    log-probability at every width."""
    m = nd()
    case = workloads.propose_m8(device=dev)
    wq, amax = m.nvfp4_quantize(case.w)
    wb = workloads.bits(case.w)
    rng = np.random.default_rng(11)
    rows = np.unique(np.concatenate([rng.integers(0, 151936, 3000), [0, 1, 151935]]))
    g = check_gpu_quant(wq, amax, wb, sample_rows=rows)
    del wb
    x = case.segments[0][0]
    pk, sc = wq.packed.cpu().numpy(), wq.scales.cpu().numpy()
    logits, idx = m.w4a16_gemv_argmax([(x[:1], None)], wq)
    torch.cuda.synchronize()
    y, sabs = par_gemv(workloads.bits(x[:1]), pk, sc, g)
    check_logits_and_argmax(logits.cpu().numpy(), idx.cpu().numpy(), y, sabs)
    lg1 = logits.cpu().numpy()
    # grammar mask + top-1 log-probability at full width (M=1 against the exact
    # logits, the larger batches against the GPU's own logits)
    mask = half_mask(8, 151936, seed=21)
    _, idx, lp = m.w4a16_gemv_argmax_ex([(x[:1], None)], wq, mask=torch.from_numpy(mask[:1]).to(dev),
                                        logits=False)
    torch.cuda.synchronize()
    i = int(idx[0])
    assert i == oracle.argmax_masked(lg1[0].astype(np.float64), mask[0])
    j = oracle.argmax_masked(y[0], mask[0])
    tol = TOL_REL * sabs[0] + TOL_ABS
    assert y[0, i] >= y[0, j] - tol[i] - tol[j]
    allowed = mask_bits(mask[0], 151936)
    lp_ref = oracle.top1_logprob(y[0], j, mask[0])
    assert abs(float(lp[0]) - lp_ref) <= tol[i] + tol[allowed].max() + 1e-5 * (1 + abs(float(lg1[0, i])))
    for mm in (2, 4, 8):
        # every logit of every batch row against the oracle, and the argmax by
        # the top-2-gap rule against the oracle's index
        logits, idx = m.w4a16_gemv_argmax([(x[:mm].contiguous(), None)], wq)
        torch.cuda.synchronize()
        lg = logits.cpu().numpy()
        ys, ss = par_gemv(workloads.bits(x[:mm]), pk, sc, g)
        check_logits_and_argmax(lg, idx.cpu().numpy(), ys, ss)
        _, idx, lp = m.w4a16_gemv_argmax_ex([(x[:mm].contiguous(), None)], wq,
                                            mask=torch.from_numpy(mask[:mm]).to(dev), logits=False)
        torch.cuda.synchronize()
        for r in range(mm):
            i = int(idx[r])
            assert i == oracle.argmax_masked(lg[r].astype(np.float64), mask[r])
            allowed = mask_bits(mask[r], 151936)
            own = float(lg[r, i]) - lse64(lg[r, allowed])
            assert abs(float(lp[r]) - own) <= 1e-5 * (1 + abs(float(lg[r, i])))


def test_propose_16_rows_full_width(dev):
    """The 151936 x 5120 head at 16 batch rows (the draft width the benchmark
    times: two MMA column groups, 63 whole tiles per CTA shared by the warps):
    every logit of every row against the oracle, and each row's argmax by the
    top-2-gap rule."""
    m = nd()
    case = workloads.propose_m8(m=16, device=dev)
    wq, _ = m.nvfp4_quantize(case.w)
    del case.w
    x = case.segments[0][0]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    logits, idx = m.w4a16_gemv_argmax([(x, None)], wq, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    g = np.float32(wq.global_scale.item())
    ys, ss = par_gemv(workloads.bits(x), wq.packed.cpu().numpy(), wq.scales.cpu().numpy(), g)
    check_logits_and_argmax(logits.cpu().numpy(), idx.cpu().numpy(), ys, ss)


@pytest.mark.parametrize("mm", [1, 4, 8])
def test_fc_combiner_config_full(dev, mm):
    """5120 x 10240 fc over RMSNorm(e) ++ RMSNorm(h), BF16 output, every output."""
    m = nd()
    case = workloads.fc_combiner(device=dev)
    wq, amax = m.nvfp4_quantize(case.w)
    g = float(wq.global_scale.item())
    (e, ge), (h, gh) = case.segments
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = m.w4a16_gemv([(e[:mm].contiguous(), ge, 1e-6), (h[:mm].contiguous(), gh, 1e-6)], wq,
                       out_dtype=torch.bfloat16, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    a = oracle.rmsnorm_concat([(workloads.bits(e[:mm]), workloads.bits(ge), 1e-6),
                               (workloads.bits(h[:mm]), workloads.bits(gh), 1e-6)], mm)
    y, sabs = par_gemv(a, wq.packed.cpu().numpy(), wq.scales.cpu().numpy(), np.float32(g))
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - y) <= TOL_REL * sabs + TOL_ABS + np.abs(y) * 2.0 ** -8)


def test_prefill_gemm_config_sampled(dev):
    """2048 x 17408 x 5120 prefill GEMM: quantiser bit-exact on every row;
    8192 sampled outputs, a full row in every M tile and a full column in every
    N tile (about 320 000 outputs), on both operand paths."""
    m = nd()
    case = workloads.prefill_gemm(device=dev)
    wq, amax = m.nvfp4_quantize(case.w)
    wb = workloads.bits(case.w)
    g = check_gpu_quant(wq, amax, wb)
    ws = torch.empty(m.gemm_workspace_bytes(2048, 5120), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    c = m.w4a16_gemm(case.a, wq, workspace=ws, dev_status=status)  # FP16 staging path
    c_bf16 = m.w4a16_gemm(case.a, wq, dev_status=status)            # the launch the benchmark times
    torch.cuda.synchronize()
    assert status.item() == 0  # no bounded wait ran out
    rng = np.random.default_rng(12)
    # 8192 random outputs, one full output row inside every 256-row M tile and
    # one full column inside every 256-column N tile (so each tile of the
    # persistent schedule is checked along a whole row and a whole column),
    # plus the first and last row and column
    mt, nt = 2048 // 256, 17408 // 256
    full_rows = np.concatenate([256 * np.arange(mt) + rng.integers(0, 256, mt), [0, 2047]])
    full_cols = np.concatenate([256 * np.arange(nt) + rng.integers(0, 256, nt), [0, 17407]])
    rows = np.concatenate([rng.integers(0, 2048, 8192), np.repeat(full_rows, 17408),
                           np.tile(np.arange(2048), full_cols.size)])
    cols = np.concatenate([rng.integers(0, 17408, 8192), np.tile(np.arange(17408), full_rows.size),
                           np.repeat(full_cols, 2048)])
    ab = workloads.bits(case.a)
    pk, sc = wq.packed.cpu().numpy(), wq.scales.cpu().numpy()
    parts = np.array_split(np.arange(rows.size), THREADS)
    with ThreadPoolExecutor(THREADS) as ex:
        res = list(ex.map(lambda ix: oracle.gemm_pairs(ab, pk, sc, g, rows[ix], cols[ix]), parts))
    exact = np.concatenate([e for e, _ in res])
    sabs = np.concatenate([s for _, s in res])
    for out in (c, c_bf16):
        got = out.float().cpu().numpy()[rows, cols].astype(np.float64)
        bad = np.abs(got - exact) > TOL_REL * sabs + TOL_ABS + np.abs(exact) * 2.0 ** -8
        assert not bad.any(), f"{int(bad.sum())} sampled outputs out of tolerance"


def test_fp8_propose_full_width(dev):
    """FP8 weight variant on the 151936 x 5120 head: per-row codes and scales
    bit-exact on sampled rows, M=1 logits over every row and the argmax."""
    m = nd()
    case = workloads.propose_m8(device=dev)
    wq = m.fp8w_quantize(case.w)
    wb = workloads.bits(case.w)
    rng = np.random.default_rng(13)
    rows = np.unique(np.concatenate([rng.integers(0, 151936, 2000), [0, 151935]]))
    codes_s, scales_s = oracle.fp8_quantize(wb, rows)
    del wb
    torch.cuda.synchronize()
    assert np.array_equal(wq.row_scale.cpu().numpy()[rows], scales_s)
    assert np.array_equal(wq.codes[torch.from_numpy(rows).to(dev)].cpu().numpy(), codes_s)
    codes, scales = wq.codes.cpu().numpy(), wq.row_scale.cpu().numpy()
    x = case.segments[0][0][:1].contiguous()
    logits, idx = m.fp8w_gemv_argmax([(x, None)], wq)
    torch.cuda.synchronize()
    a = workloads.bits(x)
    bounds = np.linspace(0, 151936, THREADS + 1).astype(int)
    jobs = [(bounds[i], bounds[i + 1] - bounds[i]) for i in range(THREADS) if bounds[i + 1] > bounds[i]]
    with ThreadPoolExecutor(THREADS) as ex:
        res = list(ex.map(lambda j: oracle.fp8_gemv(a, codes, scales, n0=j[0], nn=j[1]), jobs))
    y = np.concatenate([r[0] for r in res], axis=1)
    sabs = np.concatenate([r[1] for r in res], axis=1)
    check_logits_and_argmax(logits.cpu().numpy(), idx.cpu().numpy(), y, sabs)
