"""The oracle's Python wrapper refuses arguments its C code would read past
(the C functions trust their sizes): row ranges, indices and shapes."""
import numpy as np
import pytest

import oracle


def _weight(n=8, k=64):
    rng = np.random.default_rng(0)
    return (rng.integers(0, 256, (n, k // 2)).astype(np.uint8),
            rng.integers(0, 0x7E, (n, k // 16)).astype(np.uint8))


def test_gemv_and_dequant_ranges():
    p, s = _weight()
    a = np.zeros((2, 64), dtype=np.uint16)
    oracle.gemv(a, p, s, 1.0, n0=6, nn=2)
    with pytest.raises(ValueError):
        oracle.gemv(a, p, s, 1.0, n0=6, nn=3)
    with pytest.raises(ValueError):
        oracle.gemv(a, p, s, 1.0, n0=-1, nn=1)
    with pytest.raises(ValueError):
        oracle.gemv(np.zeros((2, 32), dtype=np.uint16), p, s, 1.0)     # K mismatch
    with pytest.raises(ValueError):
        oracle.gemv(a, p, s[:, :3], 1.0)                               # scales too narrow
    with pytest.raises(ValueError):
        oracle.dequant(p, s, 1.0, row0=7, nrows=2)


def test_gemm_pairs_indices():
    p, s = _weight()
    a = np.zeros((3, 64), dtype=np.uint16)
    oracle.gemm_pairs(a, p, s, 1.0, [0, 2], [7, 0])
    for rows, cols in (([3], [0]), ([0], [8]), ([-1], [0]), ([0, 1], [0])):
        with pytest.raises(ValueError):
            oracle.gemm_pairs(a, p, s, 1.0, rows, cols)


def test_rows_indices_and_segments():
    w = np.zeros((4, 32), dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle.quantize_rows(w, [4], np.float32(1.0))
    with pytest.raises(ValueError):
        oracle.fp8_quantize(w, rows=[-1])
    with pytest.raises(ValueError):
        oracle.rmsnorm_concat([(w, np.zeros(16, dtype=np.uint16), 1e-6)], 4)   # gamma too short
    with pytest.raises(ValueError):
        oracle.rmsnorm_concat([(w, None, 0.0)], 5)                              # too few rows
    with pytest.raises(ValueError):
        oracle.top1_logprob(np.zeros(4), 4)
    codes, scales = oracle.fp8_quantize(w)
    with pytest.raises(ValueError):
        oracle.fp8_gemv(np.zeros((1, 32), dtype=np.uint16), codes, scales, n0=3, nn=2)
    with pytest.raises(ValueError):
        oracle.fp8_gemv(np.zeros((1, 32), dtype=np.uint16), codes, scales[:3])
