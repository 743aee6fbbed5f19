// fp8.cu -- per-row FP8 (E4M3) weight quantisation for the FP8 weight
// variant of the GEMV path (quantize_bf16_to_fp8 of "spark_model/layers/
// mtp_head/new.rs", MtpHead::new):
//     s_n = fl32(amax_n / 448),   c = E4M3_RNE_SATFINITE(fl32(x / s_n))
// with the sign of x and all codes +0 for an all-zero row.  One CTA per row:
// 16-byte loads, a max over the row's BF16 magnitudes, then the quotients
// (correctly rounded binary32 division) through the hardware conversion.

#include <cuda_fp8.h>

#include "common.cuh"

namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) fp8_quantize_kernel(const uint4* __restrict__ w,
                                                                int64_t n, int64_t k,
                                                                uint2* __restrict__ codes,
                                                                float* __restrict__ row_scale,
                                                                int32_t* dev_status) {
  __shared__ unsigned int wmax[kThreads / 32];
  const int64_t nvec = k / 8;  // 8 BF16 per 16-byte load
  for (int64_t row = blockIdx.x; row < n; row += gridDim.x) {
    const uint4* src = w + row * nvec;
    unsigned int mx = 0u;
    for (int64_t i = threadIdx.x; i < nvec; i += kThreads) {
      const uint4 v = src[i];
      mx = __vmaxu2(mx, __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                                 __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu)));
    }
    mx = __reduce_max_sync(0xFFFFFFFFu, max(mx & 0xFFFFu, mx >> 16));
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = mx;
    __syncthreads();
    unsigned int m = 0u;
#pragma unroll
    for (int j = 0; j < kThreads / 32; ++j) m = max(m, wmax[j]);
    __syncthreads();  // wmax is reused by the next row
    if (m >= 0x7F80u) nvfp4::report(dev_status, NVFP4_ERR_NONFINITE);
    const float amax = __uint_as_float(m << 16);
    const float s = __fdiv_rn(amax, 448.0f);
    if (threadIdx.x == 0) row_scale[row] = s;
    uint2* dst = codes + row * nvec;
    for (int64_t i = threadIdx.x; i < nvec; i += kThreads) {
      const uint4 v = src[i];
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
      uint32_t out[2] = {0u, 0u};
      if (s != 0.0f) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t b = (j & 1) ? (u[j >> 1] & 0xFFFF0000u) : (u[j >> 1] << 16);
          const float q = __fdiv_rn(__uint_as_float(b), s);
          const uint32_t c = (uint32_t)__nv_cvt_float_to_fp8(q, __NV_SATFINITE, __NV_E4M3);
          out[j >> 2] |= c << (8 * (j & 3));
        }
      }
      dst[i] = make_uint2(out[0], out[1]);
    }
  }
  // The GEMV reads its weights before its grid-dependency wait (they are
  // load-time constants): make this kernel's output visible device-wide
  // before a dependent launch may start.
  __threadfence();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace

int launch_fp8_quantize(const void* w, int64_t n, int64_t k, uint8_t* codes, float* row_scale,
                        int32_t* dev_status, cudaStream_t stream) {
  const int64_t cap = (int64_t)nvfp4::sm_count() * 8;
  const int64_t grid = n < cap ? n : cap;
  fp8_quantize_kernel<<<(unsigned)grid, kThreads, 0, stream>>>(
      reinterpret_cast<const uint4*>(w), n, k, reinterpret_cast<uint2*>(codes), row_scale,
      dev_status);
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}
