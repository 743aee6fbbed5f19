"""Host-side argument checks of the Python binding (no GPU, no library call).

The C library sees raw pointers, so the extents, dtypes and devices of the
tensors are checked in the binding; a mismatch must raise ValueError before
anything is passed down (and must not depend on Python's assert)."""
import pytest
import torch

import nvfp4_speculative_draft_gb300 as nd

CPU = torch.device("cpu")


def bf16(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def test_check_tensor_accepts_valid_views():
    nd._check_tensor(torch.zeros((4, 8)), "t", torch.float32, CPU, (4, 8))
    nd._check_tensor(torch.zeros((4, 16))[:, :8], "t", torch.float32, CPU, (4, 8))  # padded rows
    nd._check_tensor(torch.zeros((6, 9)), "t", torch.float32, CPU, (4, 8))          # larger is fine
    nd._check_tensor(torch.zeros(5, dtype=torch.int32), "t", torch.int32, CPU, (5,), contiguous=True)


@pytest.mark.parametrize("t,dtype,shape,contig", [
    (torch.zeros((4, 8)), torch.float64, (4, 8), False),                     # dtype
    (torch.zeros((3, 8)), torch.float32, (4, 8), False),                     # too few rows
    (torch.zeros((4, 7)), torch.float32, (4, 8), False),                     # too few columns
    (torch.zeros((4, 8, 1)), torch.float32, (4, 8), False),                  # rank
    (torch.zeros((8, 4)).t(), torch.float32, (4, 8), False),                 # column stride 4
    (torch.zeros(16).as_strided((4, 8), (2, 1)), torch.float32, (4, 8), False),  # overlapping rows
    (torch.zeros(10)[::2], torch.float32, (5,), False),                      # strided vector
    (torch.zeros((4, 16))[:, :8], torch.float32, (4, 8), True),              # not contiguous
    ("not a tensor", torch.float32, (1,), False),
])
def test_check_tensor_rejects(t, dtype, shape, contig):
    with pytest.raises(ValueError):
        nd._check_tensor(t, "t", dtype, CPU, shape, contiguous=contig)


def test_check_tensor_rejects_other_device():
    meta = torch.empty((4, 8), device="meta")
    with pytest.raises(ValueError, match="must be on"):
        nd._check_tensor(meta, "t", torch.float32, CPU, (4, 8))


def test_segments_checks():
    segs, m = nd._segments([(bf16(3, 64), bf16(64), 1e-6)], CPU)
    assert m == 3 and segs[0].k_seg == 64 and segs[0].ld == 64 and segs[0].index_rows == 0
    # gathered segment: m from the index vector, table rows passed down
    idx = torch.zeros(2, dtype=torch.int32)
    segs, m = nd._segments([(bf16(100, 32), None, 1e-6, idx), (bf16(2, 32), None)], CPU)
    assert m == 2 and segs[0].index_rows == 100
    with pytest.raises(ValueError, match="same number of rows"):
        nd._segments([(bf16(3, 64), None), (bf16(2, 64), None)], CPU)
    with pytest.raises(ValueError, match="gamma needs"):
        nd._segments([(bf16(3, 64), bf16(32), 1e-6)], CPU)
    with pytest.raises(ValueError):
        nd._segments([(torch.zeros((3, 64)), None)], CPU)           # FP32 activations
    with pytest.raises(ValueError):
        nd._segments([(bf16(3, 64), None, 1e-6, torch.zeros(2, dtype=torch.int64))], CPU)
    with pytest.raises(ValueError):
        nd._segments([], CPU)


def test_argmax_outputs_checks():
    lg, idx, lp = nd._argmax_outputs(2, 100, CPU, True, None, None, True, None)
    assert lg.shape == (2, 100) and idx.shape == (2,) and lp.shape == (2,)
    assert nd._argmax_outputs(2, 100, CPU, False, None, None, False, None)[0] is None
    with pytest.raises(ValueError):   # logits buffer one column short
        nd._argmax_outputs(2, 100, CPU, True, torch.zeros((2, 99)), None, False, None)
    with pytest.raises(ValueError):   # argmax buffer too short
        nd._argmax_outputs(2, 100, CPU, False, None, torch.zeros(1, dtype=torch.int32), False, None)
    with pytest.raises(ValueError):   # log-probabilities of the wrong type
        nd._argmax_outputs(2, 100, CPU, False, None, None, True, torch.zeros(2, dtype=torch.float64))


def test_public_calls_reject_host_tensors_before_the_library():
    w = nd.Nvfp4Weight(torch.zeros((16, 32), dtype=torch.uint8), torch.zeros((16, 4), dtype=torch.uint8),
                       torch.ones(1), 16, 64)
    x = bf16(1, 64)
    for call in (lambda: nd.w4a16_gemv([(x, None)], w), lambda: nd.w4a16_gemv_argmax([(x, None)], w),
                 lambda: nd.w4a16_gemv_argmax_ex([(x, None)], w), lambda: nd.w4a16_gemm(x, w),
                 lambda: nd.nvfp4_quantize(bf16(16, 64)), lambda: nd.fp8w_quantize(bf16(16, 64))):
        with pytest.raises(ValueError, match="CUDA tensor"):
            call()
