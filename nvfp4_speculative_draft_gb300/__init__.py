"""Python binding of the NVFP4 W4A16 projection library (sm_103a).

Argument marshalling only: every step of the hot path runs in the CUDA
library ``_build/libnvfp4draft.so`` behind the C ABI of
``include/nvfp4draft.h``.  PyTorch supplies device memory and streams.  If
the library has not been built, :func:`load` raises -- there is no CPU
fallback.

The calls keep the C names:

* :func:`nvfp4_quantize`     BF16 [n, k] -> NVFP4 (packed, scales, g, absmax)
* :func:`w4a16_gemv`         y[m, n] = g * a . w~   (m <= 16, RMSNorm/concat fused)
* :func:`w4a16_gemv_argmax`  the same, FP32 logits + fused greedy argmax
  (:func:`w4a16_gemv_argmax_noalloc`: the same without a workspace)
* :func:`w4a16_gemv_argmax_ex`  + grammar bitmask and top-1 log-probability
* :func:`w4a16_gemm`         prefill C[m, n] = bf16(g * A . w~^T)
* :func:`fp8w_quantize`, :func:`fp8w_gemv`, :func:`fp8w_gemv_argmax`,
  :func:`fp8w_gemv_argmax_ex`: the same contracts for per-row FP8 weights

The C library checks what it can see (null pointers, sizes, leading
dimensions, alignment); the extents, dtypes and devices of the tensors are
checked here, before anything is passed down, and a mismatch raises
ValueError.

Example (one draft step's LM head and the prefill GEMM; every tensor on the
GPU, BF16 unless stated)::

    import nvfp4_speculative_draft_gb300 as nd
    head, _ = nd.nvfp4_quantize(w_lm_head)             # [n, k] -> NVFP4, load time
    logits, token = nd.w4a16_gemv_argmax([(hidden, norm_weight, 1e-6)], head)
    _, token, logprob = nd.w4a16_gemv_argmax_ex([(hidden, norm_weight, 1e-6)], head,
                                                mask=nd.pack_mask(allowed), logits=False)
    fc, _ = nd.nvfp4_quantize(w_fc)
    h = nd.w4a16_gemv([(embed_table, g_e, 1e-6, token), (hidden, g_h, 1e-6)], fc,
                      out_dtype=torch.bfloat16)         # embedding gathered by token
    c = nd.w4a16_gemm(prefill_activations, fc)          # [m, k] x [n, k]^T -> [m, n]
"""
import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libnvfp4draft.so")

NVFP4_OK = 0
NVFP4_ERR_INDEX = 9
STATUS_NAMES = {0: "OK", 1: "ERR_NULL", 2: "ERR_SHAPE", 3: "ERR_ALIGN", 4: "ERR_WORKSPACE",
                5: "ERR_CUDA", 6: "ERR_TIMEOUT", 7: "ERR_NONFINITE", 8: "ERR_DTYPE", 9: "ERR_INDEX"}
DTYPE_F32 = 0
DTYPE_BF16 = 1
GEMV_MAX_M = 32
GEMV_MAX_K = 16384
ARGMAX_WS_BYTES = 256
GEMV_MAX_CTAS = 1024
ARGMAX_EX_WS_BYTES = ARGMAX_WS_BYTES + GEMV_MAX_CTAS * GEMV_MAX_M * 8
GEMV_PREP_OFFSET = ARGMAX_EX_WS_BYTES


def gemv_workspace_bytes(m: int, k: int) -> int:
    """W4A16_GEMV_WS_BYTES: argmax / log-prob area plus prepared activations."""
    return GEMV_PREP_OFFSET + 256 + (k + 255) // 256 * 512 * (m if m <= 8 else GEMV_MAX_M)


QUANTIZE_WS_BYTES = 16
EXPORTED = ("nvfp4_quantize", "w4a16_gemv", "w4a16_gemv_argmax", "w4a16_gemv_argmax_ex",
            "w4a16_gemm", "fp8w_quantize", "fp8w_gemv", "fp8w_gemv_argmax", "fp8w_gemv_argmax_ex")


class Nvfp4Error(RuntimeError):
    def __init__(self, call, status):
        super().__init__(f"{call} failed: {STATUS_NAMES.get(status, status)}")
        self.status = status


def _need(cond, msg: str):
    if not cond:
        raise ValueError(msg)


def _check_tensor(t, name: str, dtype, device, min_shape=None, contiguous: bool = False):
    """t is a tensor of `dtype` on `device`; with min_shape, of that rank and
    at least that extent in every dimension; 2-D tensors have unit column
    stride (rows may be padded), or are fully contiguous when asked."""
    _need(isinstance(t, torch.Tensor), f"{name} must be a torch.Tensor")
    _need(t.dtype == dtype, f"{name} must be {dtype}, got {t.dtype}")
    _need(t.device == device, f"{name} must be on {device}, got {t.device}")
    if min_shape is not None:
        _need(t.dim() == len(min_shape) and all(a >= b for a, b in zip(t.shape, min_shape)),
              f"{name} must have shape >= {tuple(min_shape)}, got {tuple(t.shape)}")
    if contiguous:
        _need(t.is_contiguous(), f"{name} must be contiguous")
    elif t.dim() == 2:
        _need(t.stride(1) == 1 or t.shape[1] <= 1, f"{name} must have unit column stride")
        _need(t.stride(0) >= t.shape[1] or t.shape[0] <= 1, f"{name} rows must not overlap")
    elif t.dim() == 1:
        _need(t.stride(0) == 1 or t.numel() <= 1, f"{name} must be contiguous")


def _cuda_device(t, name: str):
    _need(isinstance(t, torch.Tensor) and t.is_cuda, f"{name} must be a CUDA tensor")
    return t.device


def _check_workspace(ws, device):
    if ws is not None:
        _need(isinstance(ws, torch.Tensor) and ws.device == device and ws.is_contiguous(),
              f"workspace must be a contiguous tensor on {device}")


class _Weight(ctypes.Structure):
    _fields_ = [("packed", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("global_scale", ctypes.c_void_p), ("n", ctypes.c_int64), ("k", ctypes.c_int64)]


class _Segment(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("k_seg", ctypes.c_int64), ("ld", ctypes.c_int64),
                ("gamma", ctypes.c_void_p), ("eps", ctypes.c_float),
                ("row_index", ctypes.c_void_p), ("index_rows", ctypes.c_int64)]


class _Fp8Weight(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("row_scale", ctypes.c_void_p),
                ("n", ctypes.c_int64), ("k", ctypes.c_int64)]


class _Exec(ctypes.Structure):
    _fields_ = [("stream", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("dev_status", ctypes.c_void_p)]


_LIB = None


def load(path: str = LIB_PATH):
    """Load the CUDA library (raises if it was not built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(path):
        raise ImportError(f"NVFP4 CUDA library not built: {path} is missing "
                          "(run __graft_entry__.build() or python -m "
                          "nvfp4_speculative_draft_gb300.build)")
    L = ctypes.CDLL(path)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    P = ctypes.POINTER
    L.nvfp4_quantize.argtypes = [vp, i64, i64, vp, vp, vp, vp, P(_Exec)]
    L.w4a16_gemv.argtypes = [P(_Segment), i32, i32, P(_Weight), vp, i32, i64, P(_Exec)]
    L.w4a16_gemv_argmax.argtypes = [P(_Segment), i32, i32, P(_Weight), vp, i64, vp, P(_Exec)]
    L.w4a16_gemv_argmax_ex.argtypes = [P(_Segment), i32, i32, P(_Weight), vp, i64, vp, vp, vp,
                                       i64, P(_Exec)]
    L.w4a16_gemm.argtypes = [vp, i64, i64, P(_Weight), vp, i64, P(_Exec)]
    L.fp8w_quantize.argtypes = [vp, i64, i64, vp, vp, P(_Exec)]
    L.fp8w_gemv.argtypes = [P(_Segment), i32, i32, P(_Fp8Weight), vp, i32, i64, P(_Exec)]
    L.fp8w_gemv_argmax.argtypes = [P(_Segment), i32, i32, P(_Fp8Weight), vp, i64, vp, P(_Exec)]
    L.fp8w_gemv_argmax_ex.argtypes = [P(_Segment), i32, i32, P(_Fp8Weight), vp, i64, vp, vp, vp,
                                      i64, P(_Exec)]
    L.w4a16_gemv_argmax_noalloc.argtypes = [P(_Segment), i32, i32, P(_Weight), vp, i64, vp, vp,
                                            vp]
    for f in EXPORTED + ("w4a16_gemv_argmax_noalloc",):
        getattr(L, f).restype = ctypes.c_int
    _LIB = L
    return L


@dataclass
class Nvfp4Weight:
    """Device tensors of one quantised weight."""
    packed: torch.Tensor   # uint8 [n, k/2]
    scales: torch.Tensor   # uint8 [n, k/16]
    global_scale: torch.Tensor  # float32 [1]
    n: int
    k: int

    def check(self) -> torch.device:
        """Tensors consistent with (n, k) on one CUDA device; returns it."""
        dev = _cuda_device(self.packed, "weight.packed")
        _need(self.k % 16 == 0, "weight.k must be a multiple of 16")
        _check_tensor(self.packed, "weight.packed", torch.uint8, dev, (self.n, self.k // 2), True)
        _check_tensor(self.scales, "weight.scales", torch.uint8, dev, (self.n, self.k // 16), True)
        _need(tuple(self.packed.shape) == (self.n, self.k // 2), "weight.packed must be [n, k/2]")
        _need(tuple(self.scales.shape) == (self.n, self.k // 16), "weight.scales must be [n, k/16]")
        _check_tensor(self.global_scale, "weight.global_scale", torch.float32, dev, (1,))
        return dev

    def c(self) -> _Weight:
        return _Weight(self.packed.data_ptr(), self.scales.data_ptr(),
                       self.global_scale.data_ptr(), self.n, self.k)


@dataclass
class Fp8Weight:
    """Device tensors of one per-row FP8 (E4M3) weight."""
    codes: torch.Tensor      # uint8 [n, k]
    row_scale: torch.Tensor  # float32 [n]
    n: int
    k: int

    def check(self) -> torch.device:
        """Tensors consistent with (n, k) on one CUDA device; returns it."""
        dev = _cuda_device(self.codes, "weight.codes")
        _check_tensor(self.codes, "weight.codes", torch.uint8, dev, (self.n, self.k), True)
        _need(tuple(self.codes.shape) == (self.n, self.k), "weight.codes must be [n, k]")
        _check_tensor(self.row_scale, "weight.row_scale", torch.float32, dev, (self.n,), True)
        return dev

    def c(self) -> _Fp8Weight:
        return _Fp8Weight(self.codes.data_ptr(), self.row_scale.data_ptr(), self.n, self.k)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _exec(stream=None, workspace: Optional[torch.Tensor] = None,
          dev_status: Optional[torch.Tensor] = None, device=None) -> _Exec:
    if device is not None:
        _check_workspace(workspace, device)
        if dev_status is not None:
            _check_tensor(dev_status, "dev_status", torch.int32, device, (1,))
    return _Exec(_stream(stream),
                 workspace.data_ptr() if workspace is not None else None,
                 workspace.numel() * workspace.element_size() if workspace is not None else 0,
                 dev_status.data_ptr() if dev_status is not None else None)


_WS = {}


def argmax_workspace(device) -> torch.Tensor:
    """A zeroed GEMV workspace per device (each completed call re-zeroes its
    argmax area), large enough for every GEMV call at any m <= 16 and k <= 16384
    (argmax, log-probability and the once-per-call activation preparation).
    Calls on concurrent streams must pass their own workspace instead."""
    device = torch.device(device)
    key = ("argmax", device.index)
    if key not in _WS:
        _WS[key] = torch.zeros(gemv_workspace_bytes(GEMV_MAX_M, GEMV_MAX_K), dtype=torch.uint8,
                               device=device)
    return _WS[key]


def _check(call, rc):
    if rc != NVFP4_OK:
        raise Nvfp4Error(call, rc)


def nvfp4_quantize(w: torch.Tensor, out: Optional[Nvfp4Weight] = None, absmax: Optional[torch.Tensor] = None,
                   stream=None, dev_status: Optional[torch.Tensor] = None):
    """Quantise a BF16 [n, k] device matrix.  Returns (Nvfp4Weight, absmax tensor)."""
    dev = _cuda_device(w, "w")
    _check_tensor(w, "w", torch.bfloat16, dev, (0, 0), contiguous=True)
    n, k = w.shape
    if out is None:
        out = Nvfp4Weight(torch.empty((n, k // 2), dtype=torch.uint8, device=dev),
                          torch.empty((n, k // 16), dtype=torch.uint8, device=dev),
                          torch.empty(1, dtype=torch.float32, device=dev), n, k)
    _need(out.n == n and out.k == k, "out must be a weight of the same [n, k]")
    _need(out.check() == dev, f"out must be on {dev}")
    if absmax is None:
        absmax = torch.empty(1, dtype=torch.float32, device=dev)
    _check_tensor(absmax, "absmax", torch.float32, dev, (1,))
    ex = _exec(stream, None, dev_status, dev)
    rc = load().nvfp4_quantize(w.data_ptr(), n, k, out.packed.data_ptr(), out.scales.data_ptr(),
                               out.global_scale.data_ptr(), absmax.data_ptr(), ctypes.byref(ex))
    _check("nvfp4_quantize", rc)
    return out, absmax


def _segments(segments: Sequence, device=None, m: Optional[int] = None) -> tuple:
    """segments: [(x, gamma or None, eps[, row_index]), ...], on `device`
    (default: the first x's).

    x is BF16 [m, k_seg] with unit column stride; or, with ``row_index`` (a
    device int32 tensor of m indices, e.g. the argmax output of the previous
    call), a BF16 table [rows, k_seg] whose rows row_index[r] are gathered.
    gamma is BF16 with at least k_seg contiguous elements."""
    _need(len(segments) >= 1, "at least one segment")
    arr = (_Segment * len(segments))()
    for i, s in enumerate(segments):
        s = tuple(s)
        x = s[0]
        gamma = s[1] if len(s) > 1 else None
        eps = s[2] if len(s) > 2 else 1e-6
        ridx = s[3] if len(s) > 3 else None
        if device is None:
            device = _cuda_device(x, "segment x")
        _check_tensor(x, f"segment {i} x", torch.bfloat16, device, (0, 0))
        if gamma is not None:
            _check_tensor(gamma, f"segment {i} gamma", torch.bfloat16, device, None, contiguous=True)
            _need(gamma.numel() >= x.shape[1], f"segment {i} gamma needs {x.shape[1]} elements")
        if ridx is not None:
            _check_tensor(ridx, f"segment {i} row_index", torch.int32, device, (0,), contiguous=True)
            rows = ridx.shape[0]
        else:
            rows = x.shape[0]
        arr[i] = _Segment(x.data_ptr(), x.shape[1], x.stride(0),
                          gamma.data_ptr() if gamma is not None else None, float(eps),
                          ridx.data_ptr() if ridx is not None else None,
                          x.shape[0] if ridx is not None else 0)
        m = rows if m is None else m
        _need(rows == m, "every segment needs the same number of rows")
    return arr, m


def w4a16_gemv(segments: Sequence, weight: Nvfp4Weight, out_dtype=torch.float32,
               out: Optional[torch.Tensor] = None, stream=None,
               dev_status: Optional[torch.Tensor] = None,
               workspace: Optional[torch.Tensor] = None, prepare: bool = True) -> torch.Tensor:
    """``prepare``: use the per-device workspace (or ``workspace``) so the
    activations are normalised once per call rather than in every CTA."""
    dev = weight.check()
    segs, m = _segments(segments, dev)
    if out is None:
        out = torch.empty((m, weight.n), dtype=out_dtype, device=dev)
    _need(out.dtype in (torch.float32, torch.bfloat16), "out must be float32 or bfloat16")
    _check_tensor(out, "out", out.dtype, dev, (m, weight.n))
    dt = DTYPE_F32 if out.dtype == torch.float32 else DTYPE_BF16
    if workspace is None and prepare:
        workspace = argmax_workspace(dev)
    ex = _exec(stream, workspace, dev_status, dev)
    w = weight.c()
    rc = load().w4a16_gemv(segs, len(segments), m, ctypes.byref(w), out.data_ptr(), dt,
                           out.stride(0), ctypes.byref(ex))
    _check("w4a16_gemv", rc)
    return out


def w4a16_gemv_argmax(segments: Sequence, weight: Nvfp4Weight, logits: bool = True,
                      out_logits: Optional[torch.Tensor] = None,
                      out_argmax: Optional[torch.Tensor] = None,
                      workspace: Optional[torch.Tensor] = None, stream=None,
                      dev_status: Optional[torch.Tensor] = None):
    """Returns (logits FP32 [m, n] or None, argmax int32 [m])."""
    dev = weight.check()
    segs, m = _segments(segments, dev)
    out_logits, out_argmax, _ = _argmax_outputs(m, weight.n, dev, logits, out_logits, out_argmax,
                                                False, None)
    if workspace is None:
        workspace = argmax_workspace(dev)
    ex = _exec(stream, workspace, dev_status, dev)
    w = weight.c()
    rc = load().w4a16_gemv_argmax(segs, len(segments), m, ctypes.byref(w),
                                  out_logits.data_ptr() if out_logits is not None else None,
                                  out_logits.stride(0) if out_logits is not None else 0,
                                  out_argmax.data_ptr(), ctypes.byref(ex))
    _check("w4a16_gemv_argmax", rc)
    return out_logits, out_argmax


def pack_mask(allowed: torch.Tensor) -> torch.Tensor:
    """Bool [m, n] -> int32 words [m, ceil(n/32)], bit j%32 of word j/32 = allowed[:, j]."""
    m, n = allowed.shape
    nw = (n + 31) // 32
    bits = torch.zeros((m, nw * 32), dtype=torch.int64, device=allowed.device)
    bits[:, :n] = allowed.to(torch.int64)
    words = (bits.view(m, nw, 32) << torch.arange(32, device=allowed.device)).sum(-1)
    return torch.where(words >= 2 ** 31, words - 2 ** 32, words).to(torch.int32)


def _argmax_outputs(m, n, dev, logits, out_logits, out_argmax, logprob, out_logprob):
    """Allocate the outputs not passed in; check the ones that were."""
    if logits and out_logits is None:
        out_logits = torch.empty((m, n), dtype=torch.float32, device=dev)
    if out_logits is not None:
        _check_tensor(out_logits, "out_logits", torch.float32, dev, (m, n))
    if out_argmax is None:
        out_argmax = torch.empty(m, dtype=torch.int32, device=dev)
    _check_tensor(out_argmax, "out_argmax", torch.int32, dev, (m,), contiguous=True)
    if logprob and out_logprob is None:
        out_logprob = torch.empty(m, dtype=torch.float32, device=dev)
    if out_logprob is not None:
        _check_tensor(out_logprob, "out_logprob", torch.float32, dev, (m,), contiguous=True)
    return out_logits, out_argmax, out_logprob


def _argmax_ex(call, segments, weight, n, dev, mask, logprob, logits, out_logits, out_argmax,
               out_logprob, workspace, stream, dev_status):
    segs, m = _segments(segments, dev)
    out_logits, out_argmax, out_logprob = _argmax_outputs(m, n, dev, logits, out_logits, out_argmax,
                                                          logprob, out_logprob)
    if workspace is None:
        workspace = argmax_workspace(dev)
    if mask is not None:
        _check_tensor(mask, "mask", torch.int32, dev, (m, (n + 31) // 32))
    ex = _exec(stream, workspace, dev_status, dev)
    w = weight.c()
    rc = getattr(load(), call)(segs, len(segments), m, ctypes.byref(w),
                               out_logits.data_ptr() if out_logits is not None else None,
                               out_logits.stride(0) if out_logits is not None else 0,
                               out_argmax.data_ptr(),
                               out_logprob.data_ptr() if out_logprob is not None else None,
                               mask.data_ptr() if mask is not None else None,
                               mask.stride(0) if mask is not None else 0, ctypes.byref(ex))
    _check(call, rc)
    return out_logits, out_argmax, out_logprob


def w4a16_gemv_argmax_ex(segments: Sequence, weight: Nvfp4Weight, mask: Optional[torch.Tensor] = None,
                         logprob: bool = True, logits: bool = True,
                         out_logits: Optional[torch.Tensor] = None,
                         out_argmax: Optional[torch.Tensor] = None,
                         out_logprob: Optional[torch.Tensor] = None,
                         workspace: Optional[torch.Tensor] = None, stream=None,
                         dev_status: Optional[torch.Tensor] = None):
    """Returns (logits FP32 [m, n] or None, argmax int32 [m], logprob FP32 [m] or None).

    ``mask`` is int32 words [m, >= ceil(n/32)] (see :func:`pack_mask`) or None."""
    return _argmax_ex("w4a16_gemv_argmax_ex", segments, weight, weight.n, weight.check(), mask,
                      logprob, logits, out_logits, out_argmax, out_logprob, workspace, stream,
                      dev_status)


def w4a16_gemv_argmax_noalloc(segments: Sequence, weight: Nvfp4Weight,
                              out_logits: Optional[torch.Tensor] = None,
                              out_argmax: Optional[torch.Tensor] = None, logits: bool = True,
                              stream=None, dev_status: Optional[torch.Tensor] = None):
    """w4a16_gemv_argmax without a workspace: the library's own fixed device
    scratch holds the argmax keys (for callers that cannot allocate).  Calls
    that overlap on the GPU share that scratch and race.  Output tensors are
    allocated here only when not passed in."""
    dev = weight.check()
    segs, m = _segments(segments, dev)
    out_logits, out_argmax, _ = _argmax_outputs(m, weight.n, dev, logits, out_logits, out_argmax,
                                                False, None)
    if dev_status is not None:
        _check_tensor(dev_status, "dev_status", torch.int32, dev, (1,))
    w = weight.c()
    # the library takes the scratch of the current device: make it the
    # weight's, and default to that device's current stream
    with torch.cuda.device(dev):
        rc = load().w4a16_gemv_argmax_noalloc(
            segs, len(segments), m, ctypes.byref(w),
            out_logits.data_ptr() if out_logits is not None else None,
            out_logits.stride(0) if out_logits is not None else 0, out_argmax.data_ptr(),
            _stream(torch.cuda.current_stream(dev) if stream is None else stream),
            dev_status.data_ptr() if dev_status is not None else None)
    _check("w4a16_gemv_argmax_noalloc", rc)
    return out_logits, out_argmax


def gemm_workspace_bytes(m: int, k: int) -> int:
    """Bytes of the optional w4a16_gemm workspace (FP16 staging path)."""
    return m * k * 2 + m * 4 + 256


def w4a16_gemm(a: torch.Tensor, weight: Nvfp4Weight, out: Optional[torch.Tensor] = None,
               workspace: Optional[torch.Tensor] = None, stream=None,
               dev_status: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Prefill GEMM.  Pass a workspace of gemm_workspace_bytes(m, k) bytes for
    the FP16 staging path (see the header); without one the BF16 path runs."""
    dev = weight.check()
    _check_tensor(a, "a", torch.bfloat16, dev, (0, weight.k))
    _need(a.shape[1] == weight.k, f"a must have k = {weight.k} columns, got {a.shape[1]}")
    m = a.shape[0]
    if out is None:
        out = torch.empty((m, weight.n), dtype=torch.bfloat16, device=dev)
    _check_tensor(out, "out", torch.bfloat16, dev, (m, weight.n))
    ex = _exec(stream, workspace, dev_status, dev)
    w = weight.c()
    rc = load().w4a16_gemm(a.data_ptr(), m, a.stride(0), ctypes.byref(w), out.data_ptr(),
                           out.stride(0), ctypes.byref(ex))
    _check("w4a16_gemm", rc)
    return out


# ------------------------------------------------------------ FP8 weights

def fp8w_quantize(w: torch.Tensor, out: Optional[Fp8Weight] = None, stream=None,
                  dev_status: Optional[torch.Tensor] = None) -> Fp8Weight:
    """BF16 [n, k] -> per-row FP8 E4M3 codes [n, k] + row scales [n]."""
    dev = _cuda_device(w, "w")
    _check_tensor(w, "w", torch.bfloat16, dev, (0, 0), contiguous=True)
    n, k = w.shape
    if out is None:
        out = Fp8Weight(torch.empty((n, k), dtype=torch.uint8, device=dev),
                        torch.empty(n, dtype=torch.float32, device=dev), n, k)
    _need(out.n == n and out.k == k, "out must be a weight of the same [n, k]")
    _need(out.check() == dev, f"out must be on {dev}")
    ex = _exec(stream, None, dev_status, dev)
    rc = load().fp8w_quantize(w.data_ptr(), n, k, out.codes.data_ptr(), out.row_scale.data_ptr(),
                              ctypes.byref(ex))
    _check("fp8w_quantize", rc)
    return out


def fp8w_gemv(segments: Sequence, weight: Fp8Weight, out_dtype=torch.float32,
              out: Optional[torch.Tensor] = None, stream=None,
              dev_status: Optional[torch.Tensor] = None,
              workspace: Optional[torch.Tensor] = None, prepare: bool = True) -> torch.Tensor:
    """:func:`w4a16_gemv` with the FP8 weight."""
    dev = weight.check()
    segs, m = _segments(segments, dev)
    if out is None:
        out = torch.empty((m, weight.n), dtype=out_dtype, device=dev)
    _need(out.dtype in (torch.float32, torch.bfloat16), "out must be float32 or bfloat16")
    _check_tensor(out, "out", out.dtype, dev, (m, weight.n))
    dt = DTYPE_F32 if out.dtype == torch.float32 else DTYPE_BF16
    if workspace is None and prepare:
        workspace = argmax_workspace(dev)
    ex = _exec(stream, workspace, dev_status, dev)
    w = weight.c()
    rc = load().fp8w_gemv(segs, len(segments), m, ctypes.byref(w), out.data_ptr(), dt,
                          out.stride(0), ctypes.byref(ex))
    _check("fp8w_gemv", rc)
    return out


def fp8w_gemv_argmax(segments: Sequence, weight: Fp8Weight, logits: bool = True,
                     out_logits: Optional[torch.Tensor] = None,
                     out_argmax: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None, stream=None,
                     dev_status: Optional[torch.Tensor] = None):
    """Returns (logits FP32 [m, n] or None, argmax int32 [m])."""
    dev = weight.check()
    segs, m = _segments(segments, dev)
    out_logits, out_argmax, _ = _argmax_outputs(m, weight.n, dev, logits, out_logits, out_argmax,
                                                False, None)
    if workspace is None:
        workspace = argmax_workspace(dev)
    ex = _exec(stream, workspace, dev_status, dev)
    w = weight.c()
    rc = load().fp8w_gemv_argmax(segs, len(segments), m, ctypes.byref(w),
                                 out_logits.data_ptr() if out_logits is not None else None,
                                 out_logits.stride(0) if out_logits is not None else 0,
                                 out_argmax.data_ptr(), ctypes.byref(ex))
    _check("fp8w_gemv_argmax", rc)
    return out_logits, out_argmax


def fp8w_gemv_argmax_ex(segments: Sequence, weight: Fp8Weight, mask: Optional[torch.Tensor] = None,
                        logprob: bool = True, logits: bool = True,
                        out_logits: Optional[torch.Tensor] = None,
                        out_argmax: Optional[torch.Tensor] = None,
                        out_logprob: Optional[torch.Tensor] = None,
                        workspace: Optional[torch.Tensor] = None, stream=None,
                        dev_status: Optional[torch.Tensor] = None):
    """:func:`w4a16_gemv_argmax_ex` with the FP8 weight."""
    return _argmax_ex("fp8w_gemv_argmax_ex", segments, weight, weight.n, weight.check(), mask,
                      logprob, logits, out_logits, out_argmax, out_logprob, workspace, stream,
                      dev_status)
