// common.cuh -- small shared pieces of the CUDA library (status codes come from
// the public header; nothing here is shared with the CPU oracle).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "nvfp4draft.h"

namespace nvfp4 {

// Record a device-detected condition in the caller's status word (if any).
__device__ __forceinline__ void report(int32_t* dev_status, int32_t code) {
  if (dev_status != nullptr) atomicCAS(reinterpret_cast<int*>(dev_status), 0, code);
}

// Debug builds (-DNVFP4_DEBUG_BOUNDS) check the GEMV's activation loads,
// fragment stores and output stores against the extents its arguments imply;
// a failed check records 1000 + tag in the caller's status word and the access
// is skipped.  Release builds compile the checks away.
#ifdef NVFP4_DEBUG_BOUNDS
__device__ __forceinline__ bool guard(bool ok, int tag, int32_t* st) {
  if (!ok) report(st, 1000 + tag);
  return ok;
}
#define NVFP4_GUARD(cond, tag, st) (::nvfp4::guard((cond), (tag), (st)))
#else
#define NVFP4_GUARD(cond, tag, st) true
#endif

// Test build (-DNVFP4_TEST_WITHHOLD, the library the timeout tests load): CTA 0
// never issues one copy -- the GEMV's warp 0 its first weight stage, the
// GEMM's producer its first A tile -- so the bounded wait on it runs out (the
// limit is 20 ms there) and the unwinding after a timeout runs.  Nothing of
// the withheld copy is ever in flight.
#ifdef NVFP4_TEST_WITHHOLD
constexpr unsigned long long kWaitLimit = 20000000ull;  // ns of globaltimer
constexpr bool kWithhold = true;
#else
constexpr unsigned long long kWaitLimit = 2000000000ull;
constexpr bool kWithhold = false;
#endif

__host__ __device__ __forceinline__ int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Number of SMs of the current device (cached per device ordinal).
int sm_count();

// Resident CTAs per SM of `func` at `threads` threads and `smem` dynamic shared
// bytes on the current device.  The first query per (device, func, smem) raises
// the function's dynamic shared memory limit to the device maximum and asks the
// runtime; later queries are served from a table, so calls made while a stream
// is being captured into a CUDA graph issue no CUDA API calls here.
int occupancy(const void* func, int threads, size_t smem);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda);
// false if the entry point is unavailable or the encoder rejects the map.
// Interleave none, 256-byte L2 promotion, out-of-bounds elements read as zero.
bool encode_tiled(CUtensorMap* map, CUtensorMapDataType type, cuuint32_t rank, void* addr,
                  const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                  const cuuint32_t* elem_strides, CUtensorMapSwizzle swizzle);

// Host-side argument checks shared by the entry points (status codes of
// nvfp4draft.h).
int check_weight(const nvfp4_weight* w);
int check_fp8_weight(const fp8w_weight* w);
int check_segments(const w4a16_act_segment* seg, int nseg, int m, int64_t k);

}  // namespace nvfp4

// Launchers implemented in the kernel translation units.
int launch_quantize(const void* w, int64_t n, int64_t k, uint8_t* packed, uint8_t* scales,
                    float* global_scale, uint32_t* amax_word, int32_t* dev_status,
                    cudaStream_t stream);
// The GEMV's view of a weight: NVFP4 (packed codes, block scales, global
// scale) or FP8 (E4M3 codes, one scale per row).
struct WeightRef {
  const uint8_t* codes;
  const uint8_t* scales;
  const float* gscale;
  const float* row_scale;
  int64_t n, k;
  bool fp8;
};
inline WeightRef ref_of(const nvfp4_weight* w) {
  return WeightRef{w->packed, w->scales, w->global_scale, nullptr, w->n, w->k, false};
}
inline WeightRef ref_of(const fp8w_weight* w) {
  return WeightRef{w->codes, nullptr, nullptr, w->row_scale, w->n, w->k, true};
}
int launch_fp8_quantize(const void* w, int64_t n, int64_t k, uint8_t* codes, float* row_scale,
                        int32_t* dev_status, cudaStream_t stream);
int launch_gemv(const w4a16_act_segment* seg, int nseg, int m, const WeightRef& w,
                void* y, int y_dtype, int64_t ldy, bool want_argmax, int32_t* argmax,
                void* workspace, size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream,
                float* logprob = nullptr, const int32_t* mask = nullptr, int64_t ld_mask = 0);
int launch_gemm(const void* a, int64_t m, int64_t lda, const nvfp4_weight* w, void* c,
                int64_t ldc, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                cudaStream_t stream);
size_t gemm_f16_workspace_bytes(int64_t m, int64_t k);
