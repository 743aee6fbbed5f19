"""Pins of the CPU oracle against what the number format and mathematics fix.

None of these compare the oracle with itself: each checks it against a
library routine (torch's FP8 conversion, numpy matmul / argmax), a closed
form, a hand-worked fixture under tests/golden/, an invariant, or brute force.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
CODEBOOK = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _torch_e4m3_decode_all():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def _torch_e4m3_encode(values_f32):
    t = torch.from_numpy(np.asarray(values_f32, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _f32(x):
    return float(np.float32(x))


# ------------------------------------------------------------------ format

def test_e2m1_codebook_closed_form():
    # Codebook {0, 0.5, 1, 1.5, 2, 3, 4, 6}; bit 3 is the sign.
    for c in range(8):
        assert oracle.e2m1_value(c) == CODEBOOK[c]
        neg = oracle.e2m1_value(c | 8)
        assert neg == -CODEBOOK[c] and math.copysign(1.0, neg) == -1.0


def test_e4m3_decode_matches_torch_all_bytes():
    ref = _torch_e4m3_decode_all()
    for b in range(256):
        v = oracle.e4m3_value(b)
        if math.isnan(ref[b]):
            assert math.isnan(v), hex(b)
        else:
            assert v == ref[b], hex(b)
            assert math.copysign(1.0, v) == math.copysign(1.0, ref[b])


def _golden_e4m3():
    dec, enc = [], []
    with open(os.path.join(GOLDEN, "e4m3_points.txt")) as f:
        for line in f:
            line = line.split("#")[0].split()
            if not line:
                continue
            if line[0] == "decode":
                dec.append((int(line[1], 16), float(line[2])))
            else:
                enc.append((float(line[1]), int(line[2], 16)))
    return dec, enc


def test_e4m3_golden_points():
    dec, enc = _golden_e4m3()
    assert len(dec) > 10 and len(enc) > 10
    for b, v in dec:
        got = oracle.e4m3_value(b)
        assert got == v and math.copysign(1, got) == math.copysign(1, v), hex(b)
    for v, b in enc:
        assert oracle.e4m3_encode(v) == b, v


def test_e4m3_encode_matches_torch_rne():
    # Every finite value, every midpoint, and the floats just either side of
    # each midpoint, plus random floats, within the finite range [0, 448].
    vals = np.array([oracle.e4m3_value(b) for b in range(0x7F)], dtype=np.float64)
    mids = (vals[:-1] + vals[1:]) / 2
    pts = np.concatenate([vals, mids]).astype(np.float32)
    up = np.nextafter(pts, np.float32(np.inf))
    dn = np.nextafter(pts, np.float32(0))
    rng = np.random.default_rng(0)
    rnd = (rng.random(20000) * 448).astype(np.float32)
    tiny = (rng.random(5000) * 0.02).astype(np.float32)
    allp = np.concatenate([pts, up, dn, rnd, tiny])
    allp = allp[(allp >= 0) & (allp <= 448)]
    ref = _torch_e4m3_encode(allp)
    got = np.array([oracle.e4m3_encode(float(x)) for x in allp])
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(allp[i]), got[i], ref[i]) for i in bad[:5]]


def test_e4m3_encode_saturates():
    for v in [448.0, 448.5, 463.9, 464.0, 480.0, 1e6, 3.0e38]:
        assert oracle.e4m3_encode(v) == 0x7E
    assert oracle.e4m3_encode(-1.0) == -1
    assert oracle.e4m3_encode(float("nan")) == -1


def _golden_e2m1():
    rows = []
    with open(os.path.join(GOLDEN, "e2m1_rounding.txt")) as f:
        for line in f:
            line = line.split("#")[0].split()
            if line:
                rows.append((float(line[0]), int(line[1])))
    return rows


def test_e2m1_golden_rounding():
    rows = _golden_e2m1()
    assert len(rows) > 20
    for q, code in rows:
        assert oracle.e2m1_encode(q) == code, q


def test_e2m1_rounding_either_side_of_every_midpoint():
    for c in range(7):
        mid = np.float32((CODEBOOK[c] + CODEBOOK[c + 1]) / 2)
        below = float(np.nextafter(mid, np.float32(0)))
        above = float(np.nextafter(mid, np.float32(10)))
        assert oracle.e2m1_encode(below) == c
        assert oracle.e2m1_encode(above) == c + 1
        assert oracle.e2m1_encode(-below) == c | 8
        assert oracle.e2m1_encode(-above) == (c + 1) | 8
        tie = oracle.e2m1_encode(float(mid))
        assert tie == (c if c % 2 == 0 else c + 1)


def test_brute_force_codes_times_scales_exact_in_bf16():
    # All 16 codes x 256 scale bytes: the product e2m1 * e4m3 equals the value
    # assembled from the bit fields, and BF16 holds it exactly.
    ref = _torch_e4m3_decode_all()
    for c in range(16):
        e2 = oracle.e2m1_value(c)
        s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
        e2_fields = (-1) ** s * ((m / 2) if e == 0 else 2 ** (e - 1) * (1 + m / 2))
        assert e2 == e2_fields
        for b in range(256):
            if math.isnan(ref[b]):
                continue
            p = e2 * oracle.e4m3_value(b)
            assert p == e2_fields * ref[b]
            pb = torch.tensor([p], dtype=torch.float64).to(torch.bfloat16).double().item()
            assert pb == p, (c, b)


def test_bf16_rounding_single_step_from_double():
    rng = np.random.default_rng(1)
    f = rng.standard_normal(2000).astype(np.float32) * np.float32(3.0)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_round(f.astype(np.float64))
    assert np.array_equal(got, ref)
    # A double just above a BF16 midpoint must round up, which a detour
    # through binary32 would get wrong (it lands on the midpoint, then ties).
    lo = 1.0                       # BF16 neighbours 1.0 and 1.0078125
    mid = lo + 2.0 ** -8
    assert oracle.bf16_from_double(mid) == 0x3F80          # tie -> even (1.0)
    assert oracle.bf16_from_double(mid + 2.0 ** -40) == 0x3F81
    assert oracle.bf16_from_double(mid - 2.0 ** -40) == 0x3F80
    assert oracle.bf16_from_double(-(mid + 2.0 ** -40)) == 0xBF81
    assert oracle.bf16_from_double(1e-45) == 0x0000
    assert oracle.bf16_from_double(3 * 2.0 ** -134) == 0x0002  # subnormal tie -> even


# --------------------------------------------------------------- quantiser

def _bf16_bits_from_f64(v):
    t = torch.from_numpy(np.asarray(v, dtype=np.float64)).to(torch.bfloat16)
    assert np.array_equal(t.double().numpy(), v), "construction must be exact in BF16"
    return t.view(torch.int16).numpy().view(np.uint16)


def test_quantize_lossless_round_trip_of_representable_blocks():
    rng = np.random.default_rng(2)
    n, k = 24, 96
    g = 2.0 ** -10
    codes = rng.integers(0, 16, size=(n, k))
    codes.reshape(n, k // 16, 16)[:, :, 0] = 7 | (rng.integers(0, 2, size=(n, k // 16)) * 8)
    scales = rng.integers(0x20, 0x7E, size=(n, k // 16)).astype(np.uint8)
    scales[0, 0] = 0x7E                           # amax = 6 * 448 * g = 2688 g
    val = np.vectorize(lambda c: oracle.e2m1_value(int(c)))(codes)
    sv = np.vectorize(lambda b: oracle.e4m3_value(int(b)))(scales)
    x = val * np.repeat(sv, 16, axis=1) * g
    wb = _bf16_bits_from_f64(x)
    packed, sc, gq, amax = oracle.quantize(wb)
    assert amax == 2688.0 * g and gq == np.float32(g)
    assert np.array_equal(sc, scales)
    exp_packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    assert np.array_equal(packed, exp_packed)
    assert np.array_equal(oracle.dequant(packed, sc, gq), x)


def test_quantize_all_zero_tensor_and_blocks():
    wb = np.zeros((4, 64), dtype=np.uint16)
    wb[1, 5] = 0x8000                             # -0.0 is still zero
    packed, sc, g, amax = oracle.quantize(wb)
    assert g == 0 and amax == 0
    assert not packed.any() and not sc.any()
    # A zero block inside a non-zero tensor: scale 0 and +0 codes, -0.0 included.
    x = np.zeros((2, 32))
    x[0, 20] = 1.5
    wb = _bf16_bits_from_f64(x)
    wb[1, 3] = 0x8000
    packed, sc, g, amax = oracle.quantize(wb)
    assert sc[0, 0] == 0 and sc[1, 0] == 0 and sc[1, 1] == 0 and sc[0, 1] != 0
    assert not packed[1].any() and not packed[0, :8].any()


def test_global_absmax_against_numpy():
    """The largest magnitude, whatever its sign: each matrix has one planted
    extreme, negative or positive, at a random position."""
    rng = np.random.default_rng(8)
    for trial in range(6):
        x = rng.standard_normal((17, 48)) * 0.02
        r, c = rng.integers(0, 17), rng.integers(0, 48)
        x[r, c] = (-1.0 if trial % 2 == 0 else 1.0) * 0.5
        wb = workloads.bits(torch.from_numpy(x).to(torch.bfloat16))
        xf = oracle.bf16_bits_to_f32(wb)
        assert oracle.global_absmax(wb) == np.abs(xf).max() == np.float32(0.5)
        assert oracle.quantize(wb)[3] == np.float32(0.5)


def test_quantize_sign_symmetry():
    case = workloads.tiny(n=32, k=128)
    wb = workloads.bits(case.w)
    p1, s1, g1, _ = oracle.quantize(wb)
    p2, s2, g2, _ = oracle.quantize(wb ^ np.uint16(0x8000))
    assert g1 == g2 and np.array_equal(s1, s2)
    assert np.array_equal(p2, p1 ^ np.uint8(0x88))


def test_quantize_scales_and_codes_against_library_rounding():
    # Scales: torch's RNE FP8 conversion of t = amax_b / (6 g), formed with
    # numpy binary32 arithmetic.  Codes: nearest codebook entry by brute force,
    # even code on ties.  Error: within half the local codebook gap.
    case = workloads.propose_m8(n=40, k=256)
    wb = workloads.bits(case.w)
    packed, sc, g, amax = oracle.quantize(wb)
    x = oracle.bf16_bits_to_f32(wb)
    assert amax == np.abs(x).max() and g == np.float32(amax) / np.float32(2688)
    amax_b = np.abs(x).reshape(40, -1, 16).max(-1)
    t = amax_b / (np.float32(6) * np.float32(g))
    assert t.dtype == np.float32
    exp_sc = _torch_e4m3_encode(np.minimum(t, np.float32(448)))
    assert np.array_equal(sc, exp_sc)
    dec = _torch_e4m3_decode_all().astype(np.float32)
    d = (dec[sc] * np.float32(g)).astype(np.float32)
    q = x.reshape(40, -1, 16) / d[:, :, None]
    codes = np.empty((40, 256), dtype=np.int64)
    codes[:, 0::2] = packed & 15
    codes[:, 1::2] = packed >> 4
    cb = np.array(CODEBOOK)
    dist = np.abs(np.abs(q.reshape(40, 256, 1).astype(np.float64)) - cb)
    best = dist.min(-1)
    mag = codes & 7
    chosen = dist[np.arange(40)[:, None], np.arange(256)[None], mag]
    assert np.all(chosen == best)
    ties = (dist == best[..., None]).sum(-1) > 1
    assert np.all(mag[ties] % 2 == 0)
    assert np.all(((codes >> 3) == 1) == np.signbit(x))


def test_quantize_quotients_at_codebook_midpoints():
    """Rows whose quotients x / d land exactly on an E2M1 midpoint whose lower
    neighbour is odd (0.75, 1.75, 3.5), so that ties-to-even decides the code
    -- and where x * fl32(1 / d) would land one ulp below instead.  The
    quantiser divides with a correctly rounded binary32 '/', reproduced here
    by numpy's IEEE division; the codes must follow it."""
    cases = [  # (global amax, block amax, values at a midpoint after division)
        (1.109375, 0.6953125, [0.2080078125, 0.416015625]),
        (1.109375, 0.0849609375, [0.0260009765625, 0.052001953125]),
        (1.1640625, 1.1484375, [0.1455078125]),
        (1.3828125, 1.1484375, [0.345703125, 0.69140625]),
    ]
    dec = _torch_e4m3_decode_all().astype(np.float32)
    for amax, amax_b, xs in cases:
        row = np.zeros(32)
        row[0] = amax                                   # block 0 sets the global amax
        row[16] = amax_b                                # block 1: its amax, then the values
        row[17:17 + len(xs)] = xs
        wb = _bf16_bits_from_f64(row[None, :])
        packed, sc, g, _ = oracle.quantize(wb)
        assert g == np.float32(amax) / np.float32(2688)
        t = np.float32(amax_b) / (np.float32(6) * g)
        assert sc[0, 1] == _torch_e4m3_encode([t])[0]
        d = np.float32(dec[sc[0, 1]] * g)
        q = (np.asarray(xs, dtype=np.float32) / d).astype(np.float32)   # IEEE binary32 division
        assert np.all(np.isin(q, [0.75, 1.75, 3.5])), "the fixture must hit exact midpoints"
        codes = np.empty(32, dtype=np.int64)
        codes[0::2], codes[1::2] = packed[0] & 15, packed[0] >> 4
        expect = {0.75: 2, 1.75: 4, 3.5: 6}             # ties go to the even code
        assert [int(c) for c in codes[17:17 + len(xs)]] == [expect[float(v)] for v in q]


# ---------------------------------------------------------------- RMSNorm

def test_rmsnorm_textbook_and_constant_rows():
    rng = np.random.default_rng(3)
    m, ks = 3, 200
    x = torch.from_numpy(rng.standard_normal((m, ks)).astype(np.float32)).to(torch.bfloat16)
    gamma = torch.from_numpy((1 + 0.05 * rng.standard_normal(ks)).astype(np.float32)).to(torch.bfloat16)
    out = oracle.rmsnorm_concat([(workloads.bits(x), workloads.bits(gamma), 1e-6)], m)
    xd, gd = x.double().numpy(), gamma.double().numpy()
    ref = xd / np.sqrt((xd ** 2).mean(1, keepdims=True) + 1e-6) * gd
    got = oracle.bf16_bits_to_f32(out).astype(np.float64)
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-30)
    # Constant rows: a_i = bf16(gamma_i * sign(c) / sqrt(1 + eps / c^2)).
    c = torch.full((1, ks), -0.75).to(torch.bfloat16)
    out = oracle.rmsnorm_concat([(workloads.bits(c), workloads.bits(gamma), 1e-6)], 1)
    ref = -gd / np.sqrt(1 + 1e-6 / 0.5625)
    assert np.array_equal(out[0], oracle.bf16_round(ref))
    # A row small enough that eps is not negligible: c = 2^-10, c^2 ~ eps.
    c2 = torch.full((1, ks), 2.0 ** -10).to(torch.bfloat16)
    out2 = oracle.rmsnorm_concat([(workloads.bits(c2), workloads.bits(gamma), 1e-6)], 1)
    ref2 = gd / np.sqrt(1 + 1e-6 / 2.0 ** -20)
    assert np.array_equal(out2[0], oracle.bf16_round(ref2))
    # No gamma: copy; segments concatenated in argument order.
    out = oracle.rmsnorm_concat([(workloads.bits(x), None, 0.0),
                                 (workloads.bits(c.expand(m, ks)), workloads.bits(gamma), 1e-6)], m)
    assert np.array_equal(out[:, :ks], workloads.bits(x))
    assert np.array_equal(out[0, ks:], oracle.bf16_round(ref))


# ------------------------------------------------------------------ GEMV

def _numpy_dequant(packed, scales, g):
    codes = np.empty((packed.shape[0], packed.shape[1] * 2), dtype=np.int64)
    codes[:, 0::2] = packed & 15
    codes[:, 1::2] = packed >> 4
    table = np.array(CODEBOOK + [-v for v in CODEBOOK])
    sv = _torch_e4m3_decode_all()[scales]
    return table[codes] * np.repeat(sv, 16, axis=1) * np.float64(g)


def test_gemv_matches_numpy_matmul():
    case = workloads.propose_m8(n=48, k=160, m=5)
    wb = workloads.bits(case.w)
    packed, sc, g, _ = oracle.quantize(wb)
    a = workloads.bits(case.segments[0][0])
    y, s = oracle.gemv(a, packed, sc, g)
    wd = _numpy_dequant(packed, sc, g)
    ad = oracle.bf16_bits_to_f32(a).astype(np.float64)
    ref = ad @ wd.T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-300)
    assert np.allclose(s, np.abs(ad) @ np.abs(wd).T, rtol=1e-12)
    # a sub-range of rows
    y2, _ = oracle.gemv(a, packed, sc, g, n0=7, nn=11)
    assert np.array_equal(y2, y[:, 7:18])


def test_gemv_one_hot_returns_the_dequantised_weight():
    case = workloads.tiny(n=16, k=64)
    packed, sc, g, _ = oracle.quantize(workloads.bits(case.w))
    for i in [0, 1, 17, 63]:
        a = np.zeros((1, 64), dtype=np.uint16)
        a[0, i] = 0x3F80                           # 1.0
        y, _ = oracle.gemv(a, packed, sc, g)
        code = (packed[:, i // 2] >> (4 * (i % 2))) & 15
        exp = [float(g) * oracle.e4m3_value(int(sc[r, i // 16])) * CODEBOOK[code[r] & 7]
               * (-1 if code[r] & 8 else 1) for r in range(16)]
        assert np.array_equal(y[0], np.array(exp))


def test_argmax_scan_semantics():
    rng = np.random.default_rng(4)
    for _ in range(20):
        y = rng.integers(-5, 5, size=50).astype(np.float64)
        assert oracle.argmax(y) == int(np.argmax(y))       # first occurrence
    nan, inf = float("nan"), float("inf")
    assert oracle.argmax(np.array([nan, 1.0, 1.0])) == 1
    assert oracle.argmax(np.array([-inf, -inf])) == 0
    assert oracle.argmax(np.array([nan, -inf, nan])) == 0
    assert oracle.argmax(np.array([-inf, 2.0, nan, 3.0, 3.0])) == 3


def test_gemm_pairs_match_numpy():
    case = workloads.prefill_gemm(m=9, n=20, k=96)
    packed, sc, g, _ = oracle.quantize(workloads.bits(case.w))
    a = workloads.bits(case.a)
    rows = np.repeat(np.arange(9), 20)
    cols = np.tile(np.arange(20), 9)
    exact, sabs = oracle.gemm_pairs(a, packed, sc, g, rows, cols)
    wd = _numpy_dequant(packed, sc, g)
    ad = oracle.bf16_bits_to_f32(a).astype(np.float64)
    assert np.allclose(exact.reshape(9, 20), ad @ wd.T, rtol=1e-12)
    assert np.allclose(sabs.reshape(9, 20), np.abs(ad) @ np.abs(wd).T, rtol=1e-12)


def test_workloads_are_seeded_and_shaped():
    a = workloads.lm_head_m1(n=300, k=64, rows=4)
    b = workloads.lm_head_m1(n=300, k=64, rows=4)
    assert torch.equal(a.w, b.w) and torch.equal(a.segments[0][0], b.segments[0][0])
    assert a.extra["outlier_rows"].numel() == 3
    c = workloads.fc_combiner(n=32, k_seg=48, m=3)
    assert c.w.shape == (32, 96) and len(c.segments) == 2


# ------------------------------------------- masked argmax and top-1 log-prob

def _bits_to_mask(allowed):
    n = len(allowed)
    words = np.zeros((n + 31) // 32, dtype=np.int64)
    for i, a in enumerate(allowed):
        if a:
            words[i // 32] |= 1 << (i % 32)
    return words.astype(np.uint32).view(np.int32)


def test_masked_argmax_brute_force_and_scan_rules():
    rng = np.random.default_rng(21)
    for _ in range(50):
        n = int(rng.integers(1, 200))
        y = rng.integers(-4, 4, size=n).astype(np.float64)
        allowed = rng.random(n) < 0.3
        mask = _bits_to_mask(allowed)
        idxs = np.nonzero(allowed)[0]
        exp = int(idxs[np.argmax(y[idxs])]) if idxs.size else 0   # first max among allowed
        assert oracle.argmax_masked(y, mask) == exp
    assert oracle.argmax_masked(np.array([5.0, 1.0]), _bits_to_mask([False, False])) == 0
    # words past the mask's length disallow their tokens
    y = np.zeros(40); y[35] = 9.0
    assert oracle.argmax_masked(y, _bits_to_mask([True] * 32)) == 0
    assert oracle.argmax_masked(np.array([np.nan, 2.0, 7.0]), _bits_to_mask([True, True, False])) == 1


def test_top1_logprob_against_scipy_logsumexp():
    from scipy.special import logsumexp
    rng = np.random.default_rng(22)
    for _ in range(30):
        n = int(rng.integers(1, 3000))
        y = rng.standard_normal(n) * 8
        i = int(np.argmax(y))
        assert abs(oracle.top1_logprob(y, i) - (y[i] - logsumexp(y))) < 1e-12 * (1 + abs(y[i]))
        allowed = rng.random(n) < 0.5
        allowed[i] = True
        mask = _bits_to_mask(allowed)
        exp = y[i] - logsumexp(y[allowed])
        assert abs(oracle.top1_logprob(y, i, mask) - exp) < 1e-12 * (1 + abs(y[i]))
    assert np.isnan(oracle.top1_logprob(np.array([1.0, 2.0]), 0, _bits_to_mask([False, False])))
    # a single allowed token has probability one
    assert oracle.top1_logprob(np.array([3.0, 50.0]), 0, _bits_to_mask([True, False])) == 0.0
    # uniform logits: log(1/n)
    assert abs(oracle.top1_logprob(np.zeros(64), 5) - np.log(1 / 64)) < 1e-15


# ------------------------------------------------------------ FP8 weights

def _fp8_decode(codes, scales):
    """Independent dequantisation: torch's E4M3 decode times the row scale."""
    vals = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64)
    return vals.numpy() * scales.astype(np.float64)[:, None]


def test_fp8_value_matches_torch_all_bytes():
    allb = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for b in range(256):
        if (b & 0x7F) == 0x7F:
            continue  # NaN encodings, never produced
        assert oracle.fp8_value(b) == allb[b], b


def test_fp8_quantize_lossless_round_trip_of_representable_rows():
    """Rows s * v with s a power of two, v on the E4M3 grid and one |v| = 448:
    the row scale comes out as s exactly and every code reproduces v."""
    rng = np.random.default_rng(31)
    grid = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for s_exp in (-14, -9, -3, 0):
        v = rng.choice(grid, size=(3, 64)) * rng.choice([-1.0, 1.0], size=(3, 64))
        v[:, 5] = 448.0
        s = 2.0 ** s_exp
        x = torch.tensor(v * s, dtype=torch.float64).to(torch.bfloat16)
        assert np.array_equal(x.double().numpy(), v * s)  # exact in BF16 (4 significant bits)
        codes, scales = oracle.fp8_quantize(workloads.bits(x))
        assert np.all(scales == np.float32(s))
        assert np.array_equal(_fp8_decode(codes, scales), v * s)


def test_fp8_codes_match_torch_rne_of_binary32_quotients():
    g = torch.Generator().manual_seed(32)
    w = (torch.randn((16, 256), generator=g) * torch.exp2(torch.randint(-8, 4, (16, 1), generator=g).float()))
    w = w.to(torch.bfloat16)
    codes, scales = oracle.fp8_quantize(workloads.bits(w))
    x = w.float().numpy()
    amax = np.abs(x).max(axis=1).astype(np.float32)
    s = (amax / np.float32(448.0)).astype(np.float32)
    assert np.array_equal(scales, s)
    q = (x / s[:, None]).astype(np.float32)
    ref = torch.from_numpy(np.clip(q, -448.0, 448.0)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)


def test_fp8_zero_row_and_signs():
    w = torch.zeros((3, 32), dtype=torch.bfloat16)
    w[1, 3] = -0.5
    w[1, 5] = -0.0                                 # the code keeps the sign of x
    w[2] = torch.linspace(-1, 1, 32).to(torch.bfloat16)
    codes, scales = oracle.fp8_quantize(workloads.bits(w))
    assert scales[0] == 0.0 and not codes[0].any()
    assert codes[1, 3] == 0xFE and scales[1] == np.float32(0.5) / np.float32(448.0)
    assert codes[1, 5] == 0x80 and codes[1, 4] == 0x00
    neg, pos = codes[2, :16], codes[2, 16:][::-1]
    assert np.array_equal(neg & 0x7F, pos & 0x7F) and np.all(neg & 0x80) and not np.any(pos & 0x80)


def test_fp8_gemv_matches_numpy_matmul():
    g = torch.Generator().manual_seed(33)
    w = (torch.randn((40, 96), generator=g) * 0.02).to(torch.bfloat16)
    a = torch.randn((3, 96), generator=g).to(torch.bfloat16)
    codes, scales = oracle.fp8_quantize(workloads.bits(w))
    y, sabs = oracle.fp8_gemv(workloads.bits(a), codes, scales)
    wd = _fp8_decode(codes, scales)
    ref = a.double().numpy() @ wd.T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-15)
    assert np.allclose(sabs, np.abs(a.double().numpy()) @ np.abs(wd).T, rtol=1e-12)
    y2, _ = oracle.fp8_gemv(workloads.bits(a), codes, scales, n0=7, nn=5)
    assert np.array_equal(y2, y[:, 7:12])
