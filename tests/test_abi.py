"""Host-side tests of the C ABI: the library builds, loads without a GPU,
exports every call the header declares, and rejects bad arguments on the
host with the documented status codes before anything is launched."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4draft.h")


@pytest.fixture(scope="module")
def L():
    from nvfp4_speculative_draft_gb300 import build
    build.build()
    import nvfp4_speculative_draft_gb300 as nd
    return nd.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*int\s+(\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_four_calls():
    assert set(declared_functions()) >= {"nvfp4_quantize", "w4a16_gemv", "w4a16_gemv_argmax",
                                         "w4a16_gemm"}


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_library_links_no_oracle_code():
    import nvfp4_speculative_draft_gb300 as nd
    data = open(nd.LIB_PATH, "rb").read()
    assert b"oracle_" not in data


def _weight(nd, packed=0x1000, scales=0x2000, g=0x3000, n=256, k=512):
    return nd._Weight(packed, scales, g, n, k)


def _seg(nd, x=0x4000, k_seg=512, ld=512, gamma=None, eps=1e-6):
    return nd._Segment(x, k_seg, ld, gamma, eps)


def test_quantize_argument_checks(L):
    import nvfp4_speculative_draft_gb300 as nd
    ex = nd._Exec(None, None, 0, None)
    q = L.nvfp4_quantize
    assert q(None, 4, 64, 0x1000, 0x2000, 0x3000, 0x3010, ctypes.byref(ex)) == 1
    assert q(0x1000, 4, 48, 0x1000, 0x2000, 0x3000, 0x3010, ctypes.byref(ex)) == 2
    assert q(0x1000, 0, 64, 0x1000, 0x2000, 0x3000, 0x3010, ctypes.byref(ex)) == 2
    assert q(0x1008, 4, 64, 0x1000, 0x2000, 0x3000, 0x3010, ctypes.byref(ex)) == 3
    assert q(0x1000, 4, 64, 0x1000, 0x2000, 0x3000, None, ctypes.byref(ex)) == 4
    ex_small = nd._Exec(None, 0x5000, 8, None)
    assert q(0x1000, 4, 64, 0x1000, 0x2000, 0x3000, None, ctypes.byref(ex_small)) == 4


def test_gemv_argument_checks(L):
    import nvfp4_speculative_draft_gb300 as nd
    ex = nd._Exec(None, None, 0, None)
    w = _weight(nd)
    seg = (nd._Segment * 1)(_seg(nd))
    f = L.w4a16_gemv
    assert f(seg, 1, 1, ctypes.byref(w), None, 0, 256, ctypes.byref(ex)) == 1
    assert f(seg, 1, 0, ctypes.byref(w), 0x6000, 0, 256, ctypes.byref(ex)) == 2
    assert f(seg, 1, 33, ctypes.byref(w), 0x6000, 0, 256, ctypes.byref(ex)) == 2
    assert f(seg, 3, 1, ctypes.byref(w), 0x6000, 0, 256, ctypes.byref(ex)) == 2
    assert f(seg, 1, 1, ctypes.byref(w), 0x6000, 5, 256, ctypes.byref(ex)) == 8
    assert f(seg, 1, 1, ctypes.byref(w), 0x6000, 0, 255, ctypes.byref(ex)) == 2
    bad_k = (nd._Segment * 1)(_seg(nd, k_seg=480, ld=480))
    assert f(bad_k, 1, 1, ctypes.byref(w), 0x6000, 0, 256, ctypes.byref(ex)) == 2
    bad_ld = (nd._Segment * 1)(_seg(nd, ld=516))
    assert f(bad_ld, 1, 1, ctypes.byref(w), 0x6000, 0, 256, ctypes.byref(ex)) == 3
    bad_x = (nd._Segment * 1)(_seg(nd, x=0x4004))
    assert f(bad_x, 1, 1, ctypes.byref(w), 0x6000, 0, 256, ctypes.byref(ex)) == 3
    two = (nd._Segment * 2)(_seg(nd, k_seg=256, ld=256), _seg(nd, k_seg=128, ld=128))
    assert f(two, 2, 1, ctypes.byref(w), 0x6000, 0, 256, ctypes.byref(ex)) == 2  # 384 != 512
    w_bad = _weight(nd, k=520)
    assert f(seg, 1, 1, ctypes.byref(w_bad), 0x6000, 0, 256, ctypes.byref(ex)) == 2
    w_align = _weight(nd, packed=0x1001)
    assert f(seg, 1, 1, ctypes.byref(w_align), 0x6000, 0, 256, ctypes.byref(ex)) == 3
    w_big = _weight(nd, k=32768)
    seg_big = (nd._Segment * 1)(_seg(nd, k_seg=32768, ld=32768))
    assert f(seg_big, 1, 1, ctypes.byref(w_big), 0x6000, 0, 256, ctypes.byref(ex)) == 2


def test_gemv_argmax_needs_workspace(L):
    import nvfp4_speculative_draft_gb300 as nd
    w = _weight(nd)
    seg = (nd._Segment * 1)(_seg(nd))
    f = L.w4a16_gemv_argmax
    ex = nd._Exec(None, None, 0, None)
    assert f(seg, 1, 1, ctypes.byref(w), 0x6000, 256, 0x7000, ctypes.byref(ex)) == 4
    ex = nd._Exec(None, 0x8000, 64, None)
    assert f(seg, 1, 1, ctypes.byref(w), 0x6000, 256, 0x7000, ctypes.byref(ex)) == 4
    ex = nd._Exec(None, 0x8008, 128, None)
    assert f(seg, 1, 1, ctypes.byref(w), 0x6000, 256, 0x7000, ctypes.byref(ex)) == 4
    ex = nd._Exec(None, 0x8000, 128, None)
    assert f(seg, 1, 1, ctypes.byref(w), 0x6000, 256, None, ctypes.byref(ex)) == 1
    assert f(seg, 1, 1, ctypes.byref(w), 0x6002, 256, 0x7000, ctypes.byref(ex)) == 3


def test_gemv_argmax_ex_argument_checks(L):
    import nvfp4_speculative_draft_gb300 as nd
    w = _weight(nd)                      # n = 256 -> 8 mask words
    seg = (nd._Segment * 1)(_seg(nd))
    f = L.w4a16_gemv_argmax_ex
    ok = nd._Exec(None, 0x10000, nd.ARGMAX_EX_WS_BYTES, None)
    small = nd._Exec(None, 0x10000, nd.ARGMAX_WS_BYTES, None)
    assert f(seg, 1, 1, ctypes.byref(w), 0x6000, 256, 0x7000, 0x7100, 0x7200, 8,
             ctypes.byref(small)) == 4
    assert f(seg, 1, 1, ctypes.byref(w), 0x6000, 256, None, 0x7100, 0x7200, 8,
             ctypes.byref(ok)) == 1
    assert f(seg, 1, 1, ctypes.byref(w), 0x6000, 256, 0x7000, 0x7100, 0x7200, 7,
             ctypes.byref(ok)) == 2
    assert f(seg, 1, 1, ctypes.byref(w), 0x6000, 256, 0x7000, 0x7102, 0x7200, 8,
             ctypes.byref(ok)) == 3
    assert f(seg, 1, 1, ctypes.byref(w), 0x6000, 256, 0x7000, 0x7100, 0x7201, 8,
             ctypes.byref(ok)) == 3
    assert f(seg, 1, 33, ctypes.byref(w), 0x6000, 256, 0x7000, 0x7100, 0x7200, 8,
             ctypes.byref(ok)) == 2


def test_gather_segment_argument_checks(L):
    import nvfp4_speculative_draft_gb300 as nd
    w = _weight(nd)
    ex = nd._Exec(None, None, 0, None)
    f = L.w4a16_gemv
    bad_align = (nd._Segment * 1)(nd._Segment(0x4000, 512, 512, None, 1e-6, 0x7002, 100))
    assert f(bad_align, 1, 1, ctypes.byref(w), 0x6000, 0, 256, ctypes.byref(ex)) == 3
    no_rows = (nd._Segment * 1)(nd._Segment(0x4000, 512, 512, None, 1e-6, 0x7000, 0))
    assert f(no_rows, 1, 1, ctypes.byref(w), 0x6000, 0, 256, ctypes.byref(ex)) == 2


def test_fp8w_argument_checks(L):
    import nvfp4_speculative_draft_gb300 as nd
    ex = nd._Exec(None, None, 0, None)
    q = L.fp8w_quantize
    assert q(None, 4, 64, 0x2000, 0x3000, ctypes.byref(ex)) == 1
    assert q(0x1000, 4, 48, 0x2000, 0x3000, ctypes.byref(ex)) == 2
    assert q(0x1008, 4, 64, 0x2000, 0x3000, ctypes.byref(ex)) == 3
    assert q(0x1000, 4, 64, 0x2000, 0x3002, ctypes.byref(ex)) == 3
    seg = (nd._Segment * 1)(_seg(nd))
    w = nd._Fp8Weight(0x1000, 0x3000, 256, 512)
    f = L.fp8w_gemv
    assert f(seg, 1, 1, ctypes.byref(nd._Fp8Weight(0x1000, None, 256, 512)), 0x6000, 0, 256,
             ctypes.byref(ex)) == 1
    assert f(seg, 1, 1, ctypes.byref(nd._Fp8Weight(0x1004, 0x3000, 256, 512)), 0x6000, 0, 256,
             ctypes.byref(ex)) == 3
    assert f(seg, 1, 1, ctypes.byref(w), 0x6000, 0, 200, ctypes.byref(ex)) == 2
    a = L.fp8w_gemv_argmax
    assert a(seg, 1, 1, ctypes.byref(w), 0x6000, 256, 0x7000, ctypes.byref(ex)) == 4
    e = L.fp8w_gemv_argmax_ex
    small = nd._Exec(None, 0x10000, nd.ARGMAX_WS_BYTES, None)
    assert e(seg, 1, 1, ctypes.byref(w), 0x6000, 256, 0x7000, 0x7100, 0x7200, 16,
             ctypes.byref(small)) == 4
    ok = nd._Exec(None, 0x10000, nd.ARGMAX_EX_WS_BYTES, None)
    assert e(seg, 1, 1, ctypes.byref(w), 0x6000, 256, 0x7000, 0x7100, 0x7200, 7,
             ctypes.byref(ok)) == 2


def test_gemm_argument_checks(L):
    import nvfp4_speculative_draft_gb300 as nd
    ex = nd._Exec(None, None, 0, None)
    f = L.w4a16_gemm
    w = _weight(nd, n=256, k=512)
    assert f(None, 128, 512, ctypes.byref(w), 0x9000, 256, ctypes.byref(ex)) == 1
    assert f(0x4000, 0, 512, ctypes.byref(w), 0x9000, 256, ctypes.byref(ex)) == 2
    assert f(0x4000, 128, 500, ctypes.byref(w), 0x9000, 256, ctypes.byref(ex)) == 2
    assert f(0x4000, 128, 512, ctypes.byref(w), 0x9000, 200, ctypes.byref(ex)) == 2
    w_n = _weight(nd, n=200, k=512)
    assert f(0x4000, 128, 512, ctypes.byref(w_n), 0x9000, 256, ctypes.byref(ex)) == 2
    w_k = _weight(nd, n=256, k=480)
    assert f(0x4000, 128, 512, ctypes.byref(w_k), 0x9000, 256, ctypes.byref(ex)) == 2
    assert f(0x4002, 128, 512, ctypes.byref(w), 0x9000, 256, ctypes.byref(ex)) == 3
    assert f(0x4000, 128, 516, ctypes.byref(w), 0x9000, 256, ctypes.byref(ex)) == 3


def test_product_path_fails_loudly_without_library(tmp_path):
    import nvfp4_speculative_draft_gb300 as nd
    saved = nd._LIB
    nd._LIB = None
    try:
        with pytest.raises(ImportError):
            nd.load(str(tmp_path / "missing.so"))
    finally:
        nd._LIB = saved
