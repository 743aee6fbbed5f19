"""CPU oracle for NVFP4 W4A16 projection -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct restatement of the hot path in C
(``nvfp4_oracle.c``), wrapped with ctypes and numpy.  Only ``tests/``, the
package smoke check and the benchmark's CPU-baseline leg may import this
module; the product library never does, and the two share no code.

Every function works on numpy arrays of raw bits: BF16 as ``uint16``, packed
E2M1 codes and E4M3 scales as ``uint8``.

What each function follows is stated in the C source; in short:
  * quantise: global absmax, g = absmax/2688, per-16 E4M3 block scale,
    E2M1 codes, RNE with saturation (load-time quantisation in
    "spark_model/layers/mtp_head/new.rs", MtpHead::new);
  * dequantise: g * dec(s) * e2m1(c), exact;
  * rmsnorm: weight applied as stored ("spark_model/layers/deepseek_v4_mtp.rs",
    constructor), output rounded to BF16;
  * gemv/gemm: binary64 dot products over the dequantised matrix;
  * argmax: strict '>' ascending scan from -inf
    ("spark_model/layers/deepseek_v4_mtp.rs", argmax_grammar_masked).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)
_i64 = ctypes.c_int64


# A different build of the oracle to load instead of the in-tree one: the
# mutation test points this at deliberately broken copies of the C source to
# check that the pins in tests/test_oracle.py catch each mistake.
LIB_OVERRIDE_ENV = "NVFP4_ORACLE_LIB"


def lib():
    """Build (if needed) and load the oracle's shared library."""
    global _LIB
    if _LIB is None:
        path = os.environ.get(LIB_OVERRIDE_ENV) or _build.build()
        L = ctypes.CDLL(path)
        L.oracle_e2m1_value.argtypes = [ctypes.c_int]
        L.oracle_e2m1_value.restype = ctypes.c_double
        L.oracle_e4m3_value.argtypes = [ctypes.c_int]
        L.oracle_e4m3_value.restype = ctypes.c_double
        L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        L.oracle_e4m3_encode.restype = ctypes.c_int
        L.oracle_e2m1_encode.argtypes = [ctypes.c_float]
        L.oracle_e2m1_encode.restype = ctypes.c_int
        L.oracle_bf16_from_double.argtypes = [ctypes.c_double]
        L.oracle_bf16_from_double.restype = ctypes.c_uint16
        L.oracle_global_absmax.argtypes = [_u16p, _i64, _f32p]
        L.oracle_global_absmax.restype = ctypes.c_int
        L.oracle_global_scale.argtypes = [ctypes.c_float]
        L.oracle_global_scale.restype = ctypes.c_float
        L.oracle_quantize_rows.argtypes = [_u16p, _i64, _i64, _i64, ctypes.c_float,
                                           _u8p, _u8p]
        L.oracle_quantize_rows.restype = ctypes.c_int
        L.oracle_quantize.argtypes = [_u16p, _i64, _i64, _u8p, _u8p, _f32p, _f32p]
        L.oracle_quantize.restype = ctypes.c_int
        L.oracle_dequant_rows.argtypes = [_u8p, _u8p, ctypes.c_float, _i64, _i64,
                                          _i64, _f64p]
        L.oracle_dequant_rows.restype = None
        L.oracle_rmsnorm_row.argtypes = [_u16p, _i64, _u16p, ctypes.c_float, _u16p]
        L.oracle_rmsnorm_row.restype = None
        L.oracle_gemv_rows.argtypes = [_u16p, _i64, _i64, _u8p, _u8p, ctypes.c_float,
                                       _i64, _i64, _i64, _f64p, _f64p]
        L.oracle_gemv_rows.restype = None
        L.oracle_argmax.argtypes = [_f64p, _i64]
        L.oracle_argmax.restype = _i64
        L.oracle_gemm_pairs.argtypes = [_u16p, _i64, _u8p, _u8p, ctypes.c_float, _i64,
                                        _i64p, _i64p, _i64, _f64p, _f64p]
        L.oracle_gemm_pairs.restype = None
        _i32p = ctypes.POINTER(ctypes.c_int32)
        L.oracle_argmax_masked.argtypes = [_f64p, _i64, _i32p, _i64]
        L.oracle_argmax_masked.restype = _i64
        L.oracle_top1_logprob.argtypes = [_f64p, _i64, _i32p, _i64, _i64]
        L.oracle_top1_logprob.restype = ctypes.c_double
        L.oracle_fp8_value.argtypes = [ctypes.c_int]
        L.oracle_fp8_value.restype = ctypes.c_double
        L.oracle_fp8_quantize_rows.argtypes = [_u16p, _i64, _i64, _i64, _u8p, _f32p]
        L.oracle_fp8_quantize_rows.restype = ctypes.c_int
        L.oracle_fp8_gemv_rows.argtypes = [_u16p, _i64, _i64, _u8p, _f32p, _i64, _i64, _i64,
                                           _f64p, _f64p]
        L.oracle_fp8_gemv_rows.restype = None
        _LIB = L
    return _LIB


def _ptr(a, ty):
    return a.ctypes.data_as(ty)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


class OracleError(RuntimeError):
    pass


def _need(cond, msg):
    """Argument check before a call into C (which trusts its sizes)."""
    if not cond:
        raise ValueError(msg)


def _check_weight(packed, scales, k=None):
    """packed [n, k/2] and scales [n, k/16] of one weight (k given or implied)."""
    _need(packed.ndim == 2 and scales.ndim == 2, "packed and scales must be 2-D")
    n, kh = packed.shape
    _need(k is None or kh * 2 == k, f"packed has {kh * 2} columns of codes, activations {k}")
    _need((kh * 2) % 16 == 0 and scales.shape == (n, kh * 2 // 16),
          f"scales must be [{n}, {kh * 2 // 16}], got {list(scales.shape)}")


def _check_range(n0, nn, n):
    _need(0 <= n0 and 0 <= nn and n0 + nn <= n, f"rows [{n0}, {n0 + nn}) outside [0, {n})")


# ----------------------------------------------------------------- format

def e2m1_value(code: int) -> float:
    return lib().oracle_e2m1_value(int(code))


def e4m3_value(byte: int) -> float:
    return lib().oracle_e4m3_value(int(byte))


def e4m3_encode(t: float) -> int:
    return lib().oracle_e4m3_encode(float(np.float32(t)))


def e2m1_encode(q: float) -> int:
    return lib().oracle_e2m1_encode(float(np.float32(q)))


def bf16_from_double(v: float) -> int:
    return int(lib().oracle_bf16_from_double(float(v)))


def bf16_round(values) -> np.ndarray:
    """Round an array of binary64 values to BF16 bits (uint16), RNE."""
    v = np.asarray(values, dtype=np.float64).ravel()
    out = np.empty(v.shape, dtype=np.uint16)
    f = lib().oracle_bf16_from_double
    for i, x in enumerate(v):
        out[i] = f(float(x))
    return out.reshape(np.shape(values))


def bf16_bits_to_f32(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


# -------------------------------------------------------------- quantiser

def global_absmax(w_bits) -> float:
    w = _c(w_bits, np.uint16)
    out = ctypes.c_float()
    rc = lib().oracle_global_absmax(_ptr(w, _u16p), w.size, ctypes.byref(out))
    if rc:
        raise OracleError(f"oracle_global_absmax rc={rc}")
    return out.value


def global_scale(amax: float) -> np.float32:
    return np.float32(lib().oracle_global_scale(float(np.float32(amax))))


def quantize(w_bits):
    """Quantise BF16 bits w[n, k] -> (packed [n, k/2], scales [n, k/16], g, amax)."""
    w = _c(w_bits, np.uint16)
    n, k = w.shape
    packed = np.empty((n, k // 2), dtype=np.uint8)
    scales = np.empty((n, k // 16), dtype=np.uint8)
    g = ctypes.c_float()
    amax = ctypes.c_float()
    rc = lib().oracle_quantize(_ptr(w, _u16p), n, k, _ptr(packed, _u8p),
                               _ptr(scales, _u8p), ctypes.byref(g), ctypes.byref(amax))
    if rc:
        raise OracleError(f"oracle_quantize rc={rc}")
    return packed, scales, np.float32(g.value), np.float32(amax.value)


def quantize_rows(w_bits, rows, g):
    """Quantise selected rows of w[n, k] with a given global scale g."""
    w = _c(w_bits, np.uint16)
    _need(w.ndim == 2, "w must be 2-D")
    n, k = w.shape
    rows = np.asarray(rows, dtype=np.int64).ravel()
    _need(np.all((rows >= 0) & (rows < n)), "row index outside the weight")
    packed = np.empty((len(rows), k // 2), dtype=np.uint8)
    scales = np.empty((len(rows), k // 16), dtype=np.uint8)
    for j, r in enumerate(rows):
        rc = lib().oracle_quantize_rows(_ptr(w, _u16p), k, int(r), 1, float(g),
                                        _ptr(packed[j], _u8p), _ptr(scales[j], _u8p))
        if rc:
            raise OracleError(f"oracle_quantize_rows rc={rc}")
    return packed, scales


def dequant(packed, scales, g, row0=0, nrows=None) -> np.ndarray:
    packed = _c(packed, np.uint8)
    scales = _c(scales, np.uint8)
    _check_weight(packed, scales)
    n, kh = packed.shape
    k = kh * 2
    if nrows is None:
        nrows = n - row0
    _check_range(row0, nrows, n)
    out = np.empty((nrows, k), dtype=np.float64)
    lib().oracle_dequant_rows(_ptr(packed, _u8p), _ptr(scales, _u8p), float(g), k,
                              row0, nrows, _ptr(out, _f64p))
    return out


# ---------------------------------------------------------------- RMSNorm

def rmsnorm_concat(segments, m):
    """Normalise and concatenate activation segments.

    ``segments`` is a list of (x_bits [m, k_seg] uint16, gamma_bits [k_seg] or
    None, eps).  Returns BF16 bits [m, sum k_seg]; segment order is kept.
    """
    parts = []
    for x, gamma, eps in segments:
        x = _c(x, np.uint16)
        _need(x.ndim == 2 and x.shape[0] >= m, f"a segment needs {m} rows")
        ks = x.shape[1]
        out = np.empty((m, ks), dtype=np.uint16)
        gp = None
        if gamma is not None:
            gamma = _c(gamma, np.uint16).ravel()
            _need(gamma.size >= ks, f"gamma needs {ks} elements")
            gp = _ptr(gamma, _u16p)
        for r in range(m):
            lib().oracle_rmsnorm_row(_ptr(x[r], _u16p), ks, gp, float(eps),
                                     _ptr(out[r], _u16p))
        parts.append(out)
    return np.concatenate(parts, axis=1)


# ------------------------------------------------------------ GEMV / GEMM

def gemv(a_bits, packed, scales, g, n0=0, nn=None):
    """Exact y[m, nn] and sabs[m, nn] for activation bits a[m, k]."""
    a = _c(a_bits, np.uint16)
    _need(a.ndim == 2, "activations must be 2-D")
    m, k = a.shape
    packed = _c(packed, np.uint8)
    scales = _c(scales, np.uint8)
    _check_weight(packed, scales, k)
    if nn is None:
        nn = packed.shape[0] - n0
    _check_range(n0, nn, packed.shape[0])
    y = np.empty((m, nn), dtype=np.float64)
    s = np.empty((m, nn), dtype=np.float64)
    lib().oracle_gemv_rows(_ptr(a, _u16p), m, k, _ptr(packed, _u8p), _ptr(scales, _u8p),
                           float(g), k, n0, nn, _ptr(y, _f64p), _ptr(s, _f64p))
    return y, s


def argmax(y) -> int:
    y = _c(y, np.float64)
    return int(lib().oracle_argmax(_ptr(y, _f64p), y.size))


def gemm_pairs(a_bits, packed, scales, g, rows, cols):
    """Exact C[rows[p], cols[p]] and sabs for sampled output positions."""
    a = _c(a_bits, np.uint16)
    _need(a.ndim == 2, "A must be 2-D")
    k = a.shape[1]
    packed = _c(packed, np.uint8)
    scales = _c(scales, np.uint8)
    _check_weight(packed, scales, k)
    rows = _c(rows, np.int64).ravel()
    cols = _c(cols, np.int64).ravel()
    _need(rows.size == cols.size, "rows and cols must pair up")
    _need(np.all((rows >= 0) & (rows < a.shape[0])), "a row index is outside A")
    _need(np.all((cols >= 0) & (cols < packed.shape[0])), "a column index is outside the weight")
    exact = np.empty(rows.shape, dtype=np.float64)
    sabs = np.empty(rows.shape, dtype=np.float64)
    lib().oracle_gemm_pairs(_ptr(a, _u16p), k, _ptr(packed, _u8p), _ptr(scales, _u8p),
                            float(g), k, _ptr(rows, _i64p), _ptr(cols, _i64p), rows.size,
                            _ptr(exact, _f64p), _ptr(sabs, _f64p))
    return exact, sabs


def argmax_masked(y, mask=None) -> int:
    """Grammar-masked argmax (mask: int32 words, bit i%32 of word i/32)."""
    y = _c(y, np.float64)
    if mask is None:
        return int(lib().oracle_argmax_masked(_ptr(y, _f64p), y.size, None, 0))
    mask = _c(mask, np.int32)
    return int(lib().oracle_argmax_masked(_ptr(y, _f64p), y.size,
                                          _ptr(mask, ctypes.POINTER(ctypes.c_int32)), mask.size))


def top1_logprob(y, idx, mask=None) -> float:
    """y[idx] - logsumexp over the allowed tokens; NaN when none is allowed."""
    y = _c(y, np.float64)
    _need(0 <= int(idx) < y.size, "idx outside y")
    if mask is None:
        return float(lib().oracle_top1_logprob(_ptr(y, _f64p), y.size, None, 0, int(idx)))
    mask = _c(mask, np.int32)
    return float(lib().oracle_top1_logprob(_ptr(y, _f64p), y.size,
                                           _ptr(mask, ctypes.POINTER(ctypes.c_int32)), mask.size,
                                           int(idx)))


# ------------------------------------------------------------ FP8 weights

def fp8_value(byte: int) -> float:
    return lib().oracle_fp8_value(int(byte))


def fp8_quantize(w_bits, rows=None):
    """Per-row FP8 E4M3 quantisation of BF16 bits w[n, k] (all rows or the
    given ones) -> (codes [r, k] u8, row scales [r] f32)."""
    w = _c(w_bits, np.uint16)
    _need(w.ndim == 2, "w must be 2-D")
    n, k = w.shape
    rows = np.arange(n) if rows is None else np.asarray(rows, dtype=np.int64).ravel()
    _need(np.all((rows >= 0) & (rows < n)), "row index outside the weight")
    codes = np.empty((len(rows), k), dtype=np.uint8)
    scales = np.empty(len(rows), dtype=np.float32)
    for j, r in enumerate(rows):
        rc = lib().oracle_fp8_quantize_rows(_ptr(w, _u16p), k, int(r), 1, _ptr(codes[j], _u8p),
                                            _ptr(scales[j:j + 1], _f32p))
        if rc:
            raise OracleError(f"oracle_fp8_quantize_rows rc={rc}")
    return codes, scales


def fp8_gemv(a_bits, codes, scales, n0=0, nn=None):
    """Exact y[m, nn] and sabs[m, nn] for activation bits a[m, k]."""
    a = _c(a_bits, np.uint16)
    m, k = a.shape
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.float32).ravel()
    _need(a.ndim == 2 and codes.ndim == 2 and codes.shape[1] == k, "codes must be [n, k]")
    _need(scales.size == codes.shape[0], "one scale per weight row")
    if nn is None:
        nn = codes.shape[0] - n0
    _check_range(n0, nn, codes.shape[0])
    y = np.empty((m, nn), dtype=np.float64)
    s = np.empty((m, nn), dtype=np.float64)
    lib().oracle_fp8_gemv_rows(_ptr(a, _u16p), m, k, _ptr(codes, _u8p), _ptr(scales, _f32p), k,
                               n0, nn, _ptr(y, _f64p), _ptr(s, _f64p))
    return y, s
