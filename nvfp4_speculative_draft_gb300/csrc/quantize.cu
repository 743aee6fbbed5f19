// quantize.cu -- load-time BF16 -> NVFP4 quantisation on sm_103a.
//
// The load path of "spark_model/layers/mtp_head/new.rs" (MtpHead::new) runs two
// kernels per projection: a global |w| maximum, then the block quantiser.  Both
// are HBM-bound streams over the BF16 weight; the design keeps them that way:
//   absmax_kernel   grid-stride, 4 x 16-byte loads in flight per thread, a
//                   packed 16x2 integer max on (bits & 0x7FFF) (magnitude order
//                   of finite BF16 values is integer order), warp + block
//                   reduction, one atomicMax per CTA on the float bits.
//   quantize_kernel one thread per 16-element block: 2 x 16-byte loads, the
//                   block scale from a correctly rounded binary32 division,
//                   E4M3 and E2M1 by the hardware round-to-nearest-even
//                   conversions, 8 bytes of codes + 1 scale byte stored
//                   (coalesced: consecutive threads own consecutive blocks).
// Every arithmetic step is one IEEE binary32 operation in a fixed order, so
// codes, scales, absmax and g match a scalar CPU restatement bit for bit.
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace {

__device__ __forceinline__ uint4 ld_stream_u4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// max over the eight BF16 magnitudes of a 16-byte vector, as 16x2 lanes
__device__ __forceinline__ uint32_t mag_max8(uint4 v) {
  uint32_t a = __vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu);
  uint32_t b = __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu);
  return __vmaxu2(a, b);
}

constexpr int kAbsmaxThreads = 256;
constexpr int kAbsmaxUnroll = 4;

__global__ void __launch_bounds__(kAbsmaxThreads)
absmax_kernel(const uint4* __restrict__ w, int64_t nvec, uint32_t* __restrict__ amax_word,
              int32_t* dev_status) {
  uint32_t m2 = 0;
  const int64_t stride = (int64_t)gridDim.x * kAbsmaxThreads;
  int64_t i = (int64_t)blockIdx.x * kAbsmaxThreads + threadIdx.x;
  for (; i + (kAbsmaxUnroll - 1) * stride < nvec; i += kAbsmaxUnroll * stride) {
    uint4 v[kAbsmaxUnroll];
#pragma unroll
    for (int u = 0; u < kAbsmaxUnroll; ++u) v[u] = ld_stream_u4(w + i + u * stride);
#pragma unroll
    for (int u = 0; u < kAbsmaxUnroll; ++u) m2 = __vmaxu2(m2, mag_max8(v[u]));
  }
  for (; i < nvec; i += stride) m2 = __vmaxu2(m2, mag_max8(ld_stream_u4(w + i)));
  uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  __shared__ uint32_t red[kAbsmaxThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (warp == 0) {
    m = lane < kAbsmaxThreads / 32 ? red[lane] : 0u;
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if (lane == 0) {
      if (m >= 0x7F80u) nvfp4::report(dev_status, NVFP4_ERR_NONFINITE);
      atomicMax(amax_word, m << 16);  // float bits of |w|max; monotone for x >= 0
    }
  }
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// E2M1 code of x / d: magnitude by the hardware RNE satfinite conversion of
// |q|, sign bit copied from x (a negative x whose magnitude rounds to zero
// keeps its sign, -0.0 included).
__device__ __forceinline__ uint32_t e2m1_code(float x, float d) {
  float q = __fdiv_rn(x, d);
  uint32_t mag = (uint32_t)__nv_cvt_float_to_fp4(fabsf(q), __NV_E2M1, cudaRoundNearest) & 7u;
  return mag | ((__float_as_uint(x) >> 28) & 8u);
}

constexpr int kQuantThreads = 256;

__global__ void __launch_bounds__(kQuantThreads)
quantize_kernel(const uint4* __restrict__ w, int64_t nblocks, const uint32_t* __restrict__ amax_word,
                uint2* __restrict__ packed, uint8_t* __restrict__ scales,
                float* __restrict__ global_scale) {
  const float amax = __uint_as_float(*amax_word);
  const float g = __fdiv_rn(amax, 2688.0f);  // absmax / (6 * 448)
  if (blockIdx.x == 0 && threadIdx.x == 0) *global_scale = g;
  const float six_g = __fmul_rn(6.0f, g);
  const int64_t stride = (int64_t)gridDim.x * kQuantThreads;
  for (int64_t b = (int64_t)blockIdx.x * kQuantThreads + threadIdx.x; b < nblocks; b += stride) {
    const uint4 v0 = ld_stream_u4(w + 2 * b);
    const uint4 v1 = ld_stream_u4(w + 2 * b + 1);
    const uint32_t u[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    uint32_t m2 = __vmaxu2(mag_max8(v0), mag_max8(v1));
    const float amax_b = __uint_as_float(max(m2 & 0xFFFFu, m2 >> 16) << 16);
    uint32_t s = 0;
    if (g != 0.0f && amax_b != 0.0f) {
      const float t = __fdiv_rn(amax_b, six_g);
      s = (uint32_t)__nv_cvt_float_to_fp8(t, __NV_SATFINITE, __NV_E4M3);
    }
    const __half_raw sh = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)s, __NV_E4M3);
    const float d = __fmul_rn(__half2float(__half(sh)), g);
    uint32_t lo = 0, hi = 0;
    if (d != 0.0f) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        lo |= e2m1_code(bf16_lo(u[j]), d) << (8 * j);
        lo |= e2m1_code(bf16_hi(u[j]), d) << (8 * j + 4);
        hi |= e2m1_code(bf16_lo(u[j + 4]), d) << (8 * j);
        hi |= e2m1_code(bf16_hi(u[j + 4]), d) << (8 * j + 4);
      }
    }
    packed[b] = make_uint2(lo, hi);
    scales[b] = (uint8_t)s;
  }
  // The GEMV reads its weights before its grid-dependency wait (they are
  // load-time constants): make this kernel's output visible device-wide
  // before a dependent launch may start.
  __threadfence();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace

int launch_quantize(const void* w, int64_t n, int64_t k, uint8_t* packed, uint8_t* scales,
                    float* global_scale, uint32_t* amax_word, int32_t* dev_status,
                    cudaStream_t stream) {
  const int sms = nvfp4::sm_count();
  const int64_t count = n * k;
  if (cudaMemsetAsync(amax_word, 0, sizeof(uint32_t), stream) != cudaSuccess) return NVFP4_ERR_CUDA;
  const int64_t nvec = count / 8;
  int64_t grid = nvfp4::cdiv(nvec, (int64_t)kAbsmaxThreads * kAbsmaxUnroll);
  grid = grid < (int64_t)sms * 8 ? grid : (int64_t)sms * 8;
  if (grid < 1) grid = 1;
  absmax_kernel<<<(unsigned)grid, kAbsmaxThreads, 0, stream>>>(
      reinterpret_cast<const uint4*>(w), nvec, amax_word, dev_status);
  if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
  const int64_t nblocks = count / 16;
  int64_t qgrid = nvfp4::cdiv(nblocks, kQuantThreads);
  qgrid = qgrid < (int64_t)sms * 16 ? qgrid : (int64_t)sms * 16;
  if (qgrid < 1) qgrid = 1;
  quantize_kernel<<<(unsigned)qgrid, kQuantThreads, 0, stream>>>(
      reinterpret_cast<const uint4*>(w), nblocks, amax_word, reinterpret_cast<uint2*>(packed),
      scales, global_scale);
  if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
  return NVFP4_OK;
}
