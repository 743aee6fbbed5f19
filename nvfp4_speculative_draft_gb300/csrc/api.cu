// api.cu -- the C ABI: argument validation on the host, then the launchers.
// Nothing here allocates, synchronises or keeps state beyond a cached SM count.

#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace nvfp4 {

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

namespace {
struct OccEntry {
  int dev;
  const void* func;
  int threads;
  size_t smem;
  int occ;
};
std::mutex g_occ_mutex;
OccEntry g_occ[256];
int g_nocc = 0;
}  // namespace

int occupancy(const void* func, int threads, size_t smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(g_occ_mutex);
  for (int i = 0; i < g_nocc; ++i)
    if (g_occ[i].dev == dev && g_occ[i].func == func && g_occ[i].threads == threads &&
        g_occ[i].smem == smem)
      return g_occ[i].occ;
  int maxopt = 0;
  if (cudaDeviceGetAttribute(&maxopt, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return 0;
  cudaFuncAttributes attr;
  if (cudaFuncGetAttributes(&attr, func) != cudaSuccess) return 0;
  const int limit = maxopt - (int)attr.sharedSizeBytes;  // dynamic + static <= opt-in maximum
  if (limit < 0 || smem > (size_t)limit) return 0;
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, limit) != cudaSuccess)
    return 0;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, func, threads, smem) != cudaSuccess)
    return 0;
  if (g_nocc < 256) g_occ[g_nocc++] = OccEntry{dev, func, threads, smem, occ};
  return occ;
}

}  // namespace nvfp4

namespace nvfp4 {

int check_weight(const nvfp4_weight* w) {
  if (w == nullptr || w->packed == nullptr || w->scales == nullptr || w->global_scale == nullptr)
    return NVFP4_ERR_NULL;
  if (w->n < 1 || w->k < 32 || w->k % 32 != 0) return NVFP4_ERR_SHAPE;
  if (w->n * (w->k / 2) >= (int64_t)1 << 32) return NVFP4_ERR_SHAPE;  // 32-bit offsets
  if (!aligned16(w->packed) || (reinterpret_cast<uintptr_t>(w->scales) & 1u) ||
      (reinterpret_cast<uintptr_t>(w->global_scale) & 3u))
    return NVFP4_ERR_ALIGN;
  return NVFP4_OK;
}

int check_fp8_weight(const fp8w_weight* w) {
  if (w == nullptr || w->codes == nullptr || w->row_scale == nullptr) return NVFP4_ERR_NULL;
  if (w->n < 1 || w->k < 32 || w->k % 32 != 0) return NVFP4_ERR_SHAPE;
  if (w->n * w->k >= (int64_t)1 << 32) return NVFP4_ERR_SHAPE;  // 32-bit offsets
  if (!aligned16(w->codes) || (reinterpret_cast<uintptr_t>(w->row_scale) & 3u)) return NVFP4_ERR_ALIGN;
  return NVFP4_OK;
}

int check_segments(const w4a16_act_segment* seg, int nseg, int m, int64_t k) {
  if (seg == nullptr) return NVFP4_ERR_NULL;
  if (nseg < 1 || nseg > 2) return NVFP4_ERR_SHAPE;
  if (m < 1 || m > W4A16_GEMV_MAX_M) return NVFP4_ERR_SHAPE;
  if (k > W4A16_GEMV_MAX_K) return NVFP4_ERR_SHAPE;
  int64_t total = 0;
  for (int s = 0; s < nseg; ++s) {
    if (seg[s].x == nullptr) return NVFP4_ERR_NULL;
    if (seg[s].k_seg < 32 || seg[s].k_seg % 32 != 0) return NVFP4_ERR_SHAPE;
    if (seg[s].ld < seg[s].k_seg) return NVFP4_ERR_SHAPE;
    if (seg[s].ld % 8 != 0 || !aligned16(seg[s].x)) return NVFP4_ERR_ALIGN;
    if (seg[s].gamma != nullptr && !aligned16(seg[s].gamma)) return NVFP4_ERR_ALIGN;
    if (seg[s].gamma != nullptr && !(seg[s].eps >= 0.0f)) return NVFP4_ERR_SHAPE;
    if (seg[s].row_index != nullptr) {
      if (reinterpret_cast<uintptr_t>(seg[s].row_index) & 3u) return NVFP4_ERR_ALIGN;
      if (seg[s].index_rows < 1) return NVFP4_ERR_SHAPE;
    }
    total += seg[s].k_seg;
  }
  if (total != k) return NVFP4_ERR_SHAPE;
  return NVFP4_OK;
}

bool encode_tiled(CUtensorMap* map, CUtensorMapDataType type, cuuint32_t rank, void* addr,
                  const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                  const cuuint32_t* elem_strides, CUtensorMapSwizzle swizzle) {
  static std::mutex mu;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (fn == nullptr) {
      void* ptr = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                           &q) == cudaSuccess &&
          q == cudaDriverEntryPointSuccess)
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
  }
  if (fn == nullptr) return false;
  return fn(map, type, rank, addr, dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace nvfp4

namespace {

using nvfp4::aligned16;
using nvfp4::check_fp8_weight;
using nvfp4::check_segments;
using nvfp4::check_weight;

cudaStream_t stream_of(const nvfp4_exec* ex) {
  return ex ? reinterpret_cast<cudaStream_t>(ex->stream) : nullptr;
}
int32_t* status_of(const nvfp4_exec* ex) { return ex ? ex->dev_status : nullptr; }

// Argument checks and launch shared by the two weight formats' _ex calls.
int gemv_argmax_ex(const w4a16_act_segment* seg, int nseg, int m, const WeightRef& wr, float* logits,
                   int64_t ld_logits, int32_t* argmax, float* logprob, const int32_t* mask,
                   int64_t ld_mask, const nvfp4_exec* ex) {
  const WeightRef* w = &wr;
  int rc = check_segments(seg, nseg, m, w->k);
  if (rc) return rc;
  if (argmax == nullptr) return NVFP4_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(argmax) & 3u) ||
      (logits != nullptr && (reinterpret_cast<uintptr_t>(logits) & 3u)) ||
      (logprob != nullptr && (reinterpret_cast<uintptr_t>(logprob) & 3u)) ||
      (mask != nullptr && (reinterpret_cast<uintptr_t>(mask) & 3u)))
    return NVFP4_ERR_ALIGN;
  if (logits != nullptr && ld_logits < w->n) return NVFP4_ERR_SHAPE;
  if (mask != nullptr && ld_mask < (w->n + 31) / 32) return NVFP4_ERR_SHAPE;
  if (w->n > 0x7FFFFFFFLL) return NVFP4_ERR_SHAPE;
  if (ex == nullptr || ex->workspace == nullptr || ex->workspace_bytes < W4A16_ARGMAX_EX_WS_BYTES ||
      !aligned16(ex->workspace))
    return NVFP4_ERR_WORKSPACE;
  return launch_gemv(seg, nseg, m, wr, logits, NVFP4_DTYPE_F32, ld_logits, true, argmax,
                     ex->workspace, ex->workspace_bytes, status_of(ex), stream_of(ex), logprob, mask,
                     ld_mask);
}

}  // namespace

extern "C" {

int nvfp4_quantize(const void* w_bf16, int64_t n, int64_t k, uint8_t* packed, uint8_t* scales,
                   float* global_scale, float* absmax, const nvfp4_exec* ex) {
  if (w_bf16 == nullptr || packed == nullptr || scales == nullptr || global_scale == nullptr)
    return NVFP4_ERR_NULL;
  if (n < 1 || k < 32 || k % 32 != 0) return NVFP4_ERR_SHAPE;
  if (!aligned16(w_bf16) || !aligned16(packed) || (reinterpret_cast<uintptr_t>(global_scale) & 3u))
    return NVFP4_ERR_ALIGN;
  uint32_t* word = reinterpret_cast<uint32_t*>(absmax);
  if (word == nullptr) {
    if (ex == nullptr || ex->workspace == nullptr || ex->workspace_bytes < NVFP4_QUANTIZE_WS_BYTES ||
        !aligned16(ex->workspace))
      return NVFP4_ERR_WORKSPACE;
    word = reinterpret_cast<uint32_t*>(ex->workspace);
  } else if (reinterpret_cast<uintptr_t>(absmax) & 3u) {
    return NVFP4_ERR_ALIGN;
  }
  return launch_quantize(w_bf16, n, k, packed, scales, global_scale, word, status_of(ex),
                         stream_of(ex));
}

int w4a16_gemv(const w4a16_act_segment* seg, int nseg, int m, const nvfp4_weight* w, void* y,
               int y_dtype, int64_t ldy, const nvfp4_exec* ex) {
  int rc = check_weight(w);
  if (rc) return rc;
  rc = check_segments(seg, nseg, m, w->k);
  if (rc) return rc;
  if (y == nullptr) return NVFP4_ERR_NULL;
  if (y_dtype != NVFP4_DTYPE_F32 && y_dtype != NVFP4_DTYPE_BF16) return NVFP4_ERR_DTYPE;
  if (ldy < w->n) return NVFP4_ERR_SHAPE;
  const uintptr_t ya = reinterpret_cast<uintptr_t>(y);
  if ((y_dtype == NVFP4_DTYPE_F32 && (ya & 3u)) || (ya & 1u)) return NVFP4_ERR_ALIGN;
  return launch_gemv(seg, nseg, m, ref_of(w), y, y_dtype, ldy, false, nullptr,
                     ex != nullptr ? ex->workspace : nullptr, ex != nullptr ? ex->workspace_bytes : 0,
                     status_of(ex), stream_of(ex));
}

int w4a16_gemv_argmax(const w4a16_act_segment* seg, int nseg, int m, const nvfp4_weight* w,
                      float* logits, int64_t ld_logits, int32_t* argmax, const nvfp4_exec* ex) {
  int rc = check_weight(w);
  if (rc) return rc;
  rc = check_segments(seg, nseg, m, w->k);
  if (rc) return rc;
  if (argmax == nullptr) return NVFP4_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(argmax) & 3u) ||
      (logits != nullptr && (reinterpret_cast<uintptr_t>(logits) & 3u)))
    return NVFP4_ERR_ALIGN;
  if (logits != nullptr && ld_logits < w->n) return NVFP4_ERR_SHAPE;
  if (w->n > 0x7FFFFFFFLL) return NVFP4_ERR_SHAPE;
  if (ex == nullptr || ex->workspace == nullptr || ex->workspace_bytes < W4A16_ARGMAX_WS_BYTES ||
      !aligned16(ex->workspace))
    return NVFP4_ERR_WORKSPACE;
  return launch_gemv(seg, nseg, m, ref_of(w), logits, NVFP4_DTYPE_F32, ld_logits, true, argmax,
                     ex->workspace, ex->workspace_bytes, status_of(ex), stream_of(ex));
}

int w4a16_gemv_argmax_ex(const w4a16_act_segment* seg, int nseg, int m, const nvfp4_weight* w,
                         float* logits, int64_t ld_logits, int32_t* argmax, float* logprob,
                         const int32_t* mask, int64_t ld_mask, const nvfp4_exec* ex) {
  int rc = check_weight(w);
  if (rc) return rc;
  return gemv_argmax_ex(seg, nseg, m, ref_of(w), logits, ld_logits, argmax, logprob, mask, ld_mask, ex);
}

int fp8w_gemv_argmax_ex(const w4a16_act_segment* seg, int nseg, int m, const fp8w_weight* w,
                        float* logits, int64_t ld_logits, int32_t* argmax, float* logprob,
                        const int32_t* mask, int64_t ld_mask, const nvfp4_exec* ex) {
  int rc = check_fp8_weight(w);
  if (rc) return rc;
  return gemv_argmax_ex(seg, nseg, m, ref_of(w), logits, ld_logits, argmax, logprob, mask, ld_mask, ex);
}

int w4a16_gemm(const void* a_bf16, int64_t m, int64_t lda, const nvfp4_weight* w, void* c_bf16,
               int64_t ldc, const nvfp4_exec* ex) {
  int rc = check_weight(w);
  if (rc) return rc;
  if (a_bf16 == nullptr || c_bf16 == nullptr) return NVFP4_ERR_NULL;
  if (m < 1 || w->n % 128 != 0 || w->k % 64 != 0 || lda < w->k || ldc < w->n)
    return NVFP4_ERR_SHAPE;
  if (!aligned16(a_bf16) || !aligned16(c_bf16) || lda % 8 != 0 || ldc % 8 != 0 ||
      (reinterpret_cast<uintptr_t>(w->scales) & 3u))
    return NVFP4_ERR_ALIGN;
  return launch_gemm(a_bf16, m, lda, w, c_bf16, ldc, ex ? ex->workspace : nullptr,
                     ex ? ex->workspace_bytes : 0, status_of(ex), stream_of(ex));
}

int fp8w_quantize(const void* w_bf16, int64_t n, int64_t k, uint8_t* codes, float* row_scale,
                  const nvfp4_exec* ex) {
  if (w_bf16 == nullptr || codes == nullptr || row_scale == nullptr) return NVFP4_ERR_NULL;
  if (n < 1 || k < 32 || k % 32 != 0 || n * k >= (int64_t)1 << 32) return NVFP4_ERR_SHAPE;
  if (!aligned16(w_bf16) || !aligned16(codes) || (reinterpret_cast<uintptr_t>(row_scale) & 3u))
    return NVFP4_ERR_ALIGN;
  return launch_fp8_quantize(w_bf16, n, k, codes, row_scale, status_of(ex), stream_of(ex));
}

int fp8w_gemv(const w4a16_act_segment* seg, int nseg, int m, const fp8w_weight* w, void* y,
              int y_dtype, int64_t ldy, const nvfp4_exec* ex) {
  int rc = check_fp8_weight(w);
  if (rc) return rc;
  rc = check_segments(seg, nseg, m, w->k);
  if (rc) return rc;
  if (y == nullptr) return NVFP4_ERR_NULL;
  if (y_dtype != NVFP4_DTYPE_F32 && y_dtype != NVFP4_DTYPE_BF16) return NVFP4_ERR_DTYPE;
  if (ldy < w->n) return NVFP4_ERR_SHAPE;
  const uintptr_t ya = reinterpret_cast<uintptr_t>(y);
  if ((y_dtype == NVFP4_DTYPE_F32 && (ya & 3u)) || (ya & 1u)) return NVFP4_ERR_ALIGN;
  return launch_gemv(seg, nseg, m, ref_of(w), y, y_dtype, ldy, false, nullptr,
                     ex != nullptr ? ex->workspace : nullptr, ex != nullptr ? ex->workspace_bytes : 0,
                     status_of(ex), stream_of(ex));
}

int fp8w_gemv_argmax(const w4a16_act_segment* seg, int nseg, int m, const fp8w_weight* w,
                     float* logits, int64_t ld_logits, int32_t* argmax, const nvfp4_exec* ex) {
  int rc = check_fp8_weight(w);
  if (rc) return rc;
  rc = check_segments(seg, nseg, m, w->k);
  if (rc) return rc;
  if (argmax == nullptr) return NVFP4_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(argmax) & 3u) ||
      (logits != nullptr && (reinterpret_cast<uintptr_t>(logits) & 3u)))
    return NVFP4_ERR_ALIGN;
  if (logits != nullptr && ld_logits < w->n) return NVFP4_ERR_SHAPE;
  if (w->n > 0x7FFFFFFFLL) return NVFP4_ERR_SHAPE;
  if (ex == nullptr || ex->workspace == nullptr || ex->workspace_bytes < W4A16_ARGMAX_WS_BYTES ||
      !aligned16(ex->workspace))
    return NVFP4_ERR_WORKSPACE;
  return launch_gemv(seg, nseg, m, ref_of(w), logits, NVFP4_DTYPE_F32, ld_logits, true,
                     argmax, ex->workspace, ex->workspace_bytes, status_of(ex), stream_of(ex));
}

}  // extern "C"
