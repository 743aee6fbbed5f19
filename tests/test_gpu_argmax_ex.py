"""GPU parity of the fused grammar mask and top-1 log-probability
(w4a16_gemv_argmax_ex) against the oracle's masked scan and log-sum-exp.

Bars:
  * logits: bit-equal to w4a16_gemv_argmax on the same inputs (the mask does
    not touch them), and within 1e-3 * S + 1e-6 of the oracle;
  * argmax: equal to the oracle's masked scan over the GPU's own FP32 logits
    (same precision), and to the oracle's index over exact logits whenever
    the top-2 allowed gap exceeds both tolerances; 0 when nothing is allowed;
  * log-probability: log-sum-exp is 1-Lipschitz in the max norm, so against
    the oracle's value on exact logits the error is at most tol[argmax] plus
    the largest tolerance among the allowed logits, plus FP32 exp/log/sum
    rounding (1e-5 * (1 + |y_max|)); against a binary64 log-sum-exp of the
    GPU's own logits only the FP32 rounding term remains.  NaN when nothing
    is allowed, exactly 0 when one token is.
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


def random_mask(m_rows, n, density, seed, pad_words=0):
    """int32 words [m, ceil(n/32) + pad_words]; bits past n and pad words set
    to 1 (never read: tokens past n do not exist)."""
    rng = np.random.default_rng(seed)
    nw = (n + 31) // 32
    allowed = rng.random((m_rows, nw * 32)) < density
    allowed[:, n:] = True
    words = np.zeros((m_rows, nw + pad_words), dtype=np.uint32)
    for b in range(32):
        words[:, :nw] |= allowed[:, b::32].astype(np.uint32) << np.uint32(b)
    words[:, nw:] = 0xFFFFFFFF
    return words.view(np.int32)


def lse64(v):
    v = np.asarray(v, dtype=np.float64)
    mx = v.max()
    return mx + np.log(np.exp(v - mx).sum())


def check_row(r, lg, idx, lp, y, sabs, mask):
    """One batch row: argmax and log-probability against the oracle."""
    n = y.shape[1]
    mrow = None if mask is None else mask[r]
    i = int(idx[r])
    assert i == oracle.argmax_masked(lg[r].astype(np.float64), mrow), "not the masked scan of GPU logits"
    j = oracle.argmax_masked(y[r], mrow)
    tol = TOL_REL * sabs[r] + TOL_ABS
    if mrow is None:
        allowed = np.ones(n, dtype=bool)
    else:
        bits = mrow.view(np.uint32)
        allowed = ((bits[np.arange(n) // 32] >> (np.arange(n) % 32).astype(np.uint32)) & 1).astype(bool)
    if not allowed.any():
        assert i == 0 and np.isnan(lp[r])
        return
    ya = np.where(allowed, y[r], -np.inf)
    order = np.argsort(-ya, kind="stable")
    second = order[1] if order[0] == j else order[0]
    if allowed.sum() == 1 or ya[j] - ya[second] > tol[j] + tol[second]:
        assert i == j
    else:
        assert y[r, i] >= y[r, j] - tol[j] - tol[i]
    if allowed.sum() == 1:
        assert lp[r] == 0.0
    lp_ref = oracle.top1_logprob(y[r], j, mrow)
    fp32 = 1e-5 * (1.0 + abs(float(lg[r, i])))
    assert abs(float(lp[r]) - lp_ref) <= tol[i] + tol[allowed].max() + fp32, (r, lp[r], lp_ref)
    own = float(lg[r, i]) - lse64(lg[r, allowed])
    assert abs(float(lp[r]) - own) <= fp32, (r, lp[r], own)


def run(case, dev, mask=None, logits=True):
    m = nd()
    p, s, g, _ = oracle.quantize(workloads.bits(case.w))
    wq = upload_weight(p, s, g, dev)
    x = case.segments[0][0]
    y, sabs = oracle.gemv(workloads.bits(x), p, s, g)
    dm = None if mask is None else torch.from_numpy(mask).to(dev)
    lg_ref, idx_ref = m.w4a16_gemv_argmax([(x.to(dev), None)], wq)
    lg, idx, lp = m.w4a16_gemv_argmax_ex([(x.to(dev), None)], wq, mask=dm, logits=logits)
    torch.cuda.synchronize()
    lg_ref = lg_ref.cpu().numpy()
    if logits:
        assert np.array_equal(lg.cpu().numpy(), lg_ref), "logits changed by the ex epilogue"
    if mask is None:
        assert np.array_equal(idx.cpu().numpy(), idx_ref.cpu().numpy())
    idx, lp = idx.cpu().numpy(), lp.cpu().numpy()
    for r in range(y.shape[0]):
        check_row(r, lg_ref, idx, lp, y, sabs, mask)
    return idx, lp


@pytest.mark.parametrize("m_rows", [1, 3, 8])
def test_logprob_unmasked(dev, m_rows):
    run(workloads.propose_m8(n=3001, k=512, m=m_rows), dev)


@pytest.mark.parametrize("m_rows,density", [(1, 0.5), (4, 0.05), (8, 0.3), (16, 0.3)])
def test_masked_argmax_and_logprob(dev, m_rows, density):
    case = workloads.propose_m8(n=4100, k=256, m=m_rows)
    mask = random_mask(m_rows, 4100, density, seed=100 + m_rows, pad_words=3)
    assert case.segments[0][0].shape[0] == m_rows
    idx, _ = run(case, dev, mask=mask)
    # the mask matters: some row's unmasked winner is barred
    y, _ = oracle.gemv(workloads.bits(case.segments[0][0]), *oracle.quantize(workloads.bits(case.w))[:3])
    assert any(oracle.argmax(y[r]) != idx[r] for r in range(m_rows))


def test_mask_edge_rows(dev):
    """Row 0 allows nothing, row 1 one token, row 2 only the last token, row 3
    everything; logits not written."""
    n = 1000
    case = workloads.tiny(n=n, k=512, m=4)
    nw = (n + 31) // 32
    words = np.zeros((4, nw), dtype=np.uint32)
    words[1, 517 // 32] = np.uint32(1) << np.uint32(517 % 32)
    words[2, (n - 1) // 32] = np.uint32(1) << np.uint32((n - 1) % 32)
    words[3, :] = 0xFFFFFFFF
    idx, lp = run(case, dev, mask=words.view(np.int32), logits=False)
    assert idx[0] == 0 and np.isnan(lp[0])
    assert idx[1] == 517 and lp[1] == 0.0
    assert idx[2] == n - 1 and lp[2] == 0.0
    assert lp[3] < 0.0


def test_repeat_is_bitwise_identical_and_workspace_returns_to_zero(dev):
    m = nd()
    case = workloads.propose_m8(n=20000, k=1024, m=8)
    p, s, g, _ = oracle.quantize(workloads.bits(case.w))
    wq = upload_weight(p, s, g, dev)
    x = case.segments[0][0].to(dev)
    mask = torch.from_numpy(random_mask(8, 20000, 0.4, seed=7)).to(dev)
    ws = torch.zeros(m.ARGMAX_EX_WS_BYTES, dtype=torch.uint8, device=dev)
    outs = [m.w4a16_gemv_argmax_ex([(x, None)], wq, mask=mask, logits=False, workspace=ws)
            for _ in range(3)]
    torch.cuda.synchronize()
    assert not ws[:m.ARGMAX_WS_BYTES].any().item()
    for _, idx, lp in outs[1:]:
        assert torch.equal(idx, outs[0][1])
        assert torch.equal(lp.view(torch.int32), outs[0][2].view(torch.int32))


@pytest.mark.parametrize("m_rows", [1, 4])
def test_fp8_masked_argmax_and_logprob(dev, m_rows):
    """The same fused epilogue on the FP8 weight path."""
    m = nd()
    case = workloads.propose_m8(n=2600, k=384, m=m_rows)
    codes, scales = oracle.fp8_quantize(workloads.bits(case.w))
    wq = m.Fp8Weight(torch.from_numpy(codes).to(dev), torch.from_numpy(scales).to(dev), 2600, 384)
    x = case.segments[0][0]
    y, sabs = oracle.fp8_gemv(workloads.bits(x), codes, scales)
    mask = random_mask(m_rows, 2600, 0.3, seed=200 + m_rows, pad_words=1)
    lg, idx, lp = m.fp8w_gemv_argmax_ex([(x.to(dev), None)], wq, mask=torch.from_numpy(mask).to(dev))
    torch.cuda.synchronize()
    lg, idx, lp = lg.cpu().numpy(), idx.cpu().numpy(), lp.cpu().numpy()
    for r in range(m_rows):
        check_row(r, lg, idx, lp, y, sabs, mask)
