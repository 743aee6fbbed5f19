// fp8.cu -- per-row FP8 (E4M3) weight quantisation for the FP8 weight
// variant of the GEMV path (quantize_bf16_to_fp8 of "spark_model/layers/
// mtp_head/new.rs", MtpHead::new):
//     s_n = fl32(amax_n / 448),   c = E4M3_RNE_SATFINITE(fl32(x / s_n))
// with the sign of x and all codes +0 for an all-zero row.
//
// One warp per row, every resident CTA sweeping rows in one front: a max pass
// with eight 16-byte loads in flight per lane, then the code pass re-reads
// the row (it was read a moment ago and is in L2).  The correctly rounded
// quotient's code is decided by a rounding test (Ziv, "Fast evaluation of
// elementary mathematical functions with correctly rounded last bit", 1991)
// on two bounds of x / s_n (round-toward-zero products with the row's
// reciprocal bounds), with a division per element only where the bounds
// straddle an E4M3 rounding boundary.

#include <cuda_fp8.h>

#include "common.cuh"

namespace {

constexpr int kThreads = 256;  // 8 warps, one row each at a time
constexpr int kMaxUnroll = 8;
constexpr int kCodeUnroll = 4;

__device__ __forceinline__ uint4 ld_u4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t mag_max8(uint4 v) {
  return __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                  __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
}

// Eight codes by one correctly rounded division each; code byte j is
// element j (even elements in the low BF16 half of each word).
__device__ __forceinline__ uint2 codes_exact(uint4 v, float s) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
  uint32_t out[2] = {0u, 0u};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t b = (j & 1) ? (u[j >> 1] & 0xFFFF0000u) : (u[j >> 1] << 16);
    const float q = __fdiv_rn(__uint_as_float(b), s);
    const uint32_t c = (uint32_t)__nv_cvt_float_to_fp8(q, __NV_SATFINITE, __NV_E4M3);
    out[j >> 2] |= c << (8 * (j & 3));
  }
  return make_uint2(out[0], out[1]);
}

__device__ __forceinline__ uint32_t e4m3_pair(float a_even, float a_odd) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a_even, a_odd), __NV_SATFINITE,
                                            __NV_E4M3);
}

// Two BF16 pairs -> four code bytes.  With rlo <= 1/s and rhi >= (1 + 2^-22)/s,
// RZ(x rlo) and RZ(x rhi) carry the sign of x and bracket the magnitude of
// fl32(x/s); the monotone, sign-keeping RNE satfinite conversion of the two
// bounds then brackets its code.  Returns false when the bracket holds two
// codes.
__device__ __forceinline__ uint64_t f32x2_of_bf16x2(uint32_t u) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(u << 16), "r"(u & 0xFFFF0000u));
  return r;
}
__device__ __forceinline__ uint64_t f32x2_splat(float a) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(a));
  return r;
}
// packed binary32 product of two pairs, rounded toward zero (sm_100+ f32x2)
__device__ __forceinline__ uint64_t mul_rz_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rz.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint32_t e4m3_pair2(uint64_t q) {
  float e, o;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(e), "=f"(o) : "l"(q));
  return e4m3_pair(e, o);
}

__device__ __forceinline__ bool codes_fast_word(uint32_t u0, uint32_t u1, uint64_t rlo2,
                                                uint64_t rhi2, uint32_t& out) {
  const uint64_t x01 = f32x2_of_bf16x2(u0), x23 = f32x2_of_bf16x2(u1);
  const uint32_t lo = e4m3_pair2(mul_rz_f32x2(x01, rlo2)) |
                      e4m3_pair2(mul_rz_f32x2(x23, rlo2)) << 16;
  const uint32_t hi = e4m3_pair2(mul_rz_f32x2(x01, rhi2)) |
                      e4m3_pair2(mul_rz_f32x2(x23, rhi2)) << 16;
  out = lo;
  return lo == hi;
}

__device__ __forceinline__ uint2 codes_of(uint4 v, float s, bool fast, uint64_t rlo2,
                                          uint64_t rhi2) {
  if (s == 0.0f) return make_uint2(0u, 0u);
  if (fast) {
    uint2 r;
    const bool ok0 = codes_fast_word(v.x, v.y, rlo2, rhi2, r.x);
    const bool ok1 = codes_fast_word(v.z, v.w, rlo2, rhi2, r.y);
    if (ok0 && ok1) return r;
  }
  return codes_exact(v, s);
}

__global__ void __launch_bounds__(kThreads) fp8_quantize_kernel(const uint4* __restrict__ w,
                                                                int64_t n, int64_t k,
                                                                uint2* __restrict__ codes,
                                                                float* __restrict__ row_scale,
                                                                int32_t* dev_status) {
  const int lane = threadIdx.x & 31;
  const int64_t nvec = k / 8;  // 8 BF16 per 16-byte load; k % 32 == 0, so nvec % 4 == 0
  const int64_t warps = (int64_t)gridDim.x * (kThreads / 32);
  for (int64_t row = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); row < n;
       row += warps) {
    const uint4* src = w + row * nvec;
    uint32_t m2 = 0u;
    int64_t i = lane;
    for (; i + (kMaxUnroll - 1) * 32 < nvec; i += kMaxUnroll * 32) {
      uint4 v[kMaxUnroll];
#pragma unroll
      for (int u = 0; u < kMaxUnroll; ++u) v[u] = ld_u4(src + i + 32 * u);
#pragma unroll
      for (int u = 0; u < kMaxUnroll; ++u) m2 = __vmaxu2(m2, mag_max8(v[u]));
    }
    for (; i < nvec; i += 32) m2 = __vmaxu2(m2, mag_max8(ld_u4(src + i)));
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, max(m2 & 0xFFFFu, m2 >> 16));
    if (m >= 0x7F80u && lane == 0) nvfp4::report(dev_status, NVFP4_ERR_NONFINITE);
    const float amax = __uint_as_float(m << 16);
    const float s = __fdiv_rn(amax, 448.0f);
    if (lane == 0) row_scale[row] = s;
    // 1/s normal and finite: the bounds below are then a few ulps apart
    const bool fast = s >= 0x1p-126f && s <= 0x1p126f;
    const uint64_t rlo = f32x2_splat(fast ? __frcp_rd(s) : 0.0f);
    const uint64_t rhi = f32x2_splat(fast ? __fmul_ru(__frcp_ru(s), 1.0f + 0x1p-22f) : 0.0f);
    uint2* dst = codes + row * nvec;
    i = lane;
    for (; i + (kCodeUnroll - 1) * 32 < nvec; i += kCodeUnroll * 32) {
      uint4 v[kCodeUnroll];
#pragma unroll
      for (int u = 0; u < kCodeUnroll; ++u) v[u] = ld_u4(src + i + 32 * u);
#pragma unroll
      for (int u = 0; u < kCodeUnroll; ++u) dst[i + 32 * u] = codes_of(v[u], s, fast, rlo, rhi);
    }
    for (; i < nvec; i += 32) dst[i] = codes_of(ld_u4(src + i), s, fast, rlo, rhi);
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
  const int per_sm = nvfp4::occupancy((const void*)fp8_quantize_kernel, kThreads, 0);
  const int64_t cap = (int64_t)nvfp4::sm_count() * (per_sm > 0 ? per_sm : 1);
  int64_t grid = nvfp4::cdiv(n, (int64_t)(kThreads / 32));
  grid = grid < cap ? grid : cap;
  fp8_quantize_kernel<<<(unsigned)grid, kThreads, 0, stream>>>(
      reinterpret_cast<const uint4*>(w), n, k, reinterpret_cast<uint2*>(codes), row_scale,
      dev_status);
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}
