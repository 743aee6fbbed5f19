// quantize.cu -- load-time BF16 -> NVFP4 quantisation on sm_103a.
//
// The load path of "spark_model/layers/mtp_head/new.rs" (MtpHead::new) runs two
// kernels per projection: a global |w| maximum, then the block quantiser.  Both
// are HBM-bound streams over the BF16 weight; the design keeps them that way:
//   absmax_kernel   grid-stride, 4 x 16-byte loads in flight per thread, a
//                   packed 16x2 integer max on (bits & 0x7FFF) (magnitude order
//                   of finite BF16 values is integer order), warp + block
//                   reduction, one atomicMax per CTA on the float bits.
//   quantize_kernel persistent, every CTA resident: a producer warp streams
//                   16 KB chunks of the weight (512 blocks of 16 elements)
//                   into a ring of shared-memory stages with bulk async
//                   copies; each compute thread takes two adjacent blocks of
//                   a chunk: the block
//                   scale and the E2M1 codes are the hardware round-to-
//                   nearest-even conversions of correctly rounded binary32
//                   quotients, decided by a rounding test on two bounds of
//                   each quotient, with a division only where the bounds
//                   straddle a rounding boundary; 8 bytes of codes + 1 scale
//                   byte stored.
// Every arithmetic step is one IEEE binary32 operation in a fixed order, so
// codes, scales, absmax and g match a scalar CPU restatement bit for bit.
#include <cuda_bf16.h>
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
  // the quantise grid may be scheduled as this grid's CTAs retire; it waits
  // for this grid's completion (and memory flush) before it reads the maximum
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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

// Eight packed codes (4 BF16 pairs -> 4 bytes, even element in the low
// nibble) by one correctly rounded division per element.
__device__ __forceinline__ uint32_t e2m1_word_exact(const uint32_t* u, float d) {
  uint32_t r = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    r |= e2m1_code(bf16_lo(u[j]), d) << (8 * j);
    r |= e2m1_code(bf16_hi(u[j]), d) << (8 * j + 4);
  }
  return r;
}

__device__ __forceinline__ uint32_t e2m1_pair(float q_even, float q_odd) {
  return (uint32_t)__nv_cvt_float2_to_fp4x2(make_float2(q_even, q_odd), __NV_E2M1,
                                            cudaRoundNearest);
}

// Packed binary32 pairs (sm_100+ f32x2 arithmetic): one instruction for the
// two products of a BF16 pair.
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
__device__ __forceinline__ uint64_t mul_rz_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rz.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// E2M1 codes of a packed pair: even element (low word) in the low nibble
__device__ __forceinline__ uint32_t e2m1_pair2(uint64_t q) {
  float e, o;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(e), "=f"(o) : "l"(q));
  return e2m1_pair(e, o);
}

// Division-free codes (Ziv's rounding test, "Fast evaluation of elementary
// mathematical functions with correctly rounded last bit", 1991).  With
// rlo <= 1/d and rhi >= (1 + 2^-22)/d, the round-toward-zero products
// RZ(x rlo) and RZ(x rhi) carry the sign of x and bracket the magnitude of
// x/d (RZ loses less than 2^-23 of it) and so of its correctly rounded
// quotient fl32(x/d).  The RNE satfinite conversion is monotone in the
// magnitude and keeps the sign, so when the two bounds convert to the same
// code that is the code of fl32(x/d); otherwise (a rounding boundary within
// the bracket, a few ulps wide) the word is recomputed by division.
__device__ __forceinline__ uint32_t e2m1_word_fast(const uint32_t* u, float d, uint64_t rlo2,
                                                   uint64_t rhi2) {
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint64_t x = f32x2_of_bf16x2(u[j]);
    lo |= e2m1_pair2(mul_rz_f32x2(x, rlo2)) << (8 * j);
    hi |= e2m1_pair2(mul_rz_f32x2(x, rhi2)) << (8 * j);
  }
  return lo == hi ? lo : e2m1_word_exact(u, d);
}

// Per E4M3 scale code s (128 entries, 127 = NaN): d = fl32(dec(s) g) and the
// reciprocal bounds of the rounding test, or fast = 0 where d or 1/d is not
// a finite normal number (d = 0 included).
struct ScaleEntry {
  float d, rlo, rhi;
  uint32_t fast;
};

__device__ __forceinline__ ScaleEntry scale_entry(uint32_t s, float g) {
  const __half_raw sh = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)s, __NV_E4M3);
  ScaleEntry e;
  e.d = __fmul_rn(__half2float(__half(sh)), g);
  e.fast = (e.d >= 0x1p-126f && e.d <= 0x1p126f) ? 1u : 0u;
  e.rlo = e.fast ? __frcp_rd(e.d) : 0.0f;
  e.rhi = e.fast ? __fmul_ru(__frcp_ru(e.d), 1.0f + 0x1p-22f) : 0.0f;
  return e;
}

// max |x| over a block's 16 BF16 values (packed pairs; equal to the integer
// maximum of the magnitude bits for finite values)
__device__ __forceinline__ float block_absmax(const uint32_t* u) {
  __nv_bfloat162 m[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&u[j]);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&u[j + 4]);
    m[j] = __hmax2(__habs2(a), __habs2(b));
  }
  const __nv_bfloat162 r = __hmax2(__hmax2(m[0], m[1]), __hmax2(m[2], m[3]));
  return fmaxf(__low2float(r), __high2float(r));
}

// Codes + scale of one 16-element block held in v0 (elements 0..7), v1 (8..15).
// The scale code s = E4M3(fl32(amax_b / 6g)) by the same rounding test on
// the two bounds of the quotient (t6lo, t6hi as rlo, rhi above for the
// divisor 6g; fast6 = 0 where that divisor fails the range check).
struct BlockCodes {
  uint2 codes;
  uint32_t scale;
};

__device__ __forceinline__ BlockCodes quantize_block(uint4 v0, uint4 v1, float g, float six_g,
                                                     bool fast6, float t6lo, float t6hi,
                                                     const ScaleEntry* tab) {
  const uint32_t u[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  const float amax_b = block_absmax(u);
  uint32_t s = 0;
  if (g != 0.0f && amax_b != 0.0f) {
    uint32_t pair = 0x100u;  // forces the division unless fast6
    if (fast6)
      pair = (uint32_t)__nv_cvt_float2_to_fp8x2(
          make_float2(__fmul_rz(amax_b, t6lo), __fmul_rz(amax_b, t6hi)), __NV_SATFINITE,
          __NV_E4M3);
    s = pair & 0xFFu;
    if (s != (pair >> 8)) {
      const float t = __fdiv_rn(amax_b, six_g);
      s = (uint32_t)__nv_cvt_float_to_fp8(t, __NV_SATFINITE, __NV_E4M3);
    }
  }
  const ScaleEntry e = tab[s];
  if (e.fast) {
    const uint64_t rlo2 = f32x2_splat(e.rlo), rhi2 = f32x2_splat(e.rhi);
    return {make_uint2(e2m1_word_fast(u, e.d, rlo2, rhi2), e2m1_word_fast(u + 4, e.d, rlo2, rhi2)),
            s};
  }
  if (e.d == 0.0f) return {make_uint2(0u, 0u), s};
  return {make_uint2(e2m1_word_exact(u, e.d), e2m1_word_exact(u + 4, e.d)), s};
}

// ------------------------------------------------ the staged quantise pass
__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
// try_wait with a suspend-time hint: a waiting warp issues nothing meanwhile
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}
// Bounded wait; false (and NVFP4_ERR_TIMEOUT recorded) if it ran out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int32_t* dev_status) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > nvfp4::kWaitLimit) {
      nvfp4::report(dev_status, NVFP4_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");  // stays after the barrier wait that makes the stage valid
  return v;
}

constexpr int kQuantWarps = 8;                          // compute warps
constexpr int kQuantThreads = kQuantWarps * 32 + 32;    // + one producer warp
constexpr int kBlocksPerThread = 2;                     // blocks 2t and 2t + 1 of a chunk
constexpr int kChunkBlocks = kQuantWarps * 32 * kBlocksPerThread;
constexpr int kChunkBytes = kChunkBlocks * 32;          // 16 KB of BF16 per stage
constexpr int kQuantStages = 3;
constexpr size_t kQuantSmem = (size_t)kQuantStages * kChunkBytes;

// Persistent: CTA c takes chunks c, c + grid, ...; chunk j of a CTA goes to
// stage j % kQuantStages.  full[s] completes when a chunk's bytes have landed
// (producer's expect_tx + the copy), empty[s] when all compute warps have
// read it out of shared memory.  Every wait is bounded; after a timeout the
// roles leave their loops and the producer waits (bounded) for the copies it
// issued, so none is in flight when the CTA exits.
__global__ void __launch_bounds__(kQuantThreads)
quantize_kernel(const uint4* __restrict__ w, int64_t nblocks, const uint32_t* __restrict__ amax_word,
                uint2* __restrict__ packed, uint8_t* __restrict__ scales,
                float* __restrict__ global_scale, int32_t* dev_status) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(8) uint64_t full[kQuantStages], empty[kQuantStages];
  __shared__ ScaleEntry tab[128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ring_base = (uint32_t)__cvta_generic_to_shared(ring);
  const uint32_t full0 = (uint32_t)__cvta_generic_to_shared(full);
  const uint32_t empty0 = (uint32_t)__cvta_generic_to_shared(empty);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kQuantStages; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, kQuantWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int64_t nchunks = nvfp4::cdiv(nblocks, kChunkBlocks);
  if (warp == kQuantWarps) {
    // producer: the weight is not written by the absmax grid, so copies start
    // before the grid-dependency wait
    if (lane != 0) return;
    int64_t it = 0;
    int st = 0;          // stage of chunk it (it mod kQuantStages)
    uint32_t ph = 0u;    // parity of its round (it / kQuantStages)
    for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x, ++it) {
      if (it >= kQuantStages && !mbar_wait(empty0 + 8 * st, ph ^ 1u, dev_status)) break;
      const int64_t nb = nblocks - c * kChunkBlocks;
      const uint32_t bytes = (uint32_t)(nb < kChunkBlocks ? nb : kChunkBlocks) * 32u;
      mbar_arrive_expect_tx(full0 + 8 * st, bytes);
      bulk_copy_g2s(ring_base + st * kChunkBytes, w + c * (kChunkBlocks * 2), bytes, full0 + 8 * st);
      if (++st == kQuantStages) {
        st = 0;
        ph ^= 1u;
      }
    }
    // every issued copy has landed before this thread (and so the CTA) exits
    const int64_t first = it > kQuantStages ? it - kQuantStages : 0;
    for (int64_t j = first; j < it; ++j)
      if (!mbar_wait(full0 + 8 * (int)(j % kQuantStages), (uint32_t)((j / kQuantStages) & 1),
                     dev_status))
        break;
    return;
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the absmax grid has completed
  const float amax = __uint_as_float(*amax_word);
  const float g = __fdiv_rn(amax, 2688.0f);  // absmax / (6 * 448)
  if (blockIdx.x == 0 && threadIdx.x == 0) *global_scale = g;
  const float six_g = __fmul_rn(6.0f, g);
  if (threadIdx.x < 128) tab[threadIdx.x] = scale_entry(threadIdx.x, g);
  const bool fast6 = six_g >= 0x1p-126f && six_g <= 0x1p126f;
  const float t6lo = fast6 ? __frcp_rd(six_g) : 0.0f;
  const float t6hi = fast6 ? __fmul_ru(__frcp_ru(six_g), 1.0f + 0x1p-22f) : 0.0f;
  asm volatile("bar.sync 1, %0;" ::"n"(kQuantWarps * 32) : "memory");  // compute warps only
  const bool scales_even = (reinterpret_cast<uintptr_t>(scales) & 1u) == 0;
  int st = 0;        // stage of the current chunk (its index mod kQuantStages)
  uint32_t ph = 0u;  // parity of its round
  const int64_t bstep = (int64_t)gridDim.x * kChunkBlocks;
  int64_t b0 = (int64_t)blockIdx.x * kChunkBlocks + 2 * threadIdx.x;
  for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x, b0 += bstep) {
    if (!mbar_wait(full0 + 8 * st, ph, dev_status)) break;
    // blocks 2t, 2t + 1 of the chunk (b0, b0 + 1): 64 contiguous bytes in,
    // 16 bytes of codes and 2 scale bytes out
    const int nb = b0 + 1 < nblocks ? 2 : (b0 < nblocks ? 1 : 0);
    uint4 v[4];
    const uint32_t src = ring_base + st * kChunkBytes + threadIdx.x * 64u;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (q < 2 * nb) v[q] = lds128(src + 16u * q);  // vectors 2h, 2h + 1 hold block h
    // the stage is released once every lane has used the values it read
    // (a load's data is only certain to have left shared memory when an
    // instruction has consumed it), then the results are stored
    BlockCodes q0 = {make_uint2(0u, 0u), 0u}, q1 = {make_uint2(0u, 0u), 0u};
    if (nb >= 1) q0 = quantize_block(v[0], v[1], g, six_g, fast6, t6lo, t6hi, tab);
    if (nb == 2) q1 = quantize_block(v[2], v[3], g, six_g, fast6, t6lo, t6hi, tab);
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * st);
    if (nb == 2) {
      *reinterpret_cast<uint4*>(packed + b0) = make_uint4(q0.codes.x, q0.codes.y, q1.codes.x, q1.codes.y);
      if (scales_even) {
        *reinterpret_cast<uint16_t*>(scales + b0) = (uint16_t)(q0.scale | q1.scale << 8);
      } else {  // the scale array may start at any byte
        scales[b0] = (uint8_t)q0.scale;
        scales[b0 + 1] = (uint8_t)q1.scale;
      }
    } else if (nb == 1) {
      packed[b0] = q0.codes;
      scales[b0] = (uint8_t)q0.scale;
    }
    if (++st == kQuantStages) {
      st = 0;
      ph ^= 1u;
    }
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
  // persistent: every CTA resident at once
  const int per_sm = nvfp4::occupancy((const void*)quantize_kernel, kQuantThreads, kQuantSmem);
  const int64_t qcap = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
  int64_t qgrid = nvfp4::cdiv(nblocks, (int64_t)kChunkBlocks);
  qgrid = qgrid < qcap ? qgrid : qcap;
  if (qgrid < 1) qgrid = 1;
  // programmatic dependent launch: the grid is scheduled as the absmax CTAs
  // retire; its compute warps wait (griddepcontrol.wait) for that grid before
  // reading amax
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)qgrid);
  cfg.blockDim = dim3(kQuantThreads);
  cfg.dynamicSmemBytes = kQuantSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, quantize_kernel, reinterpret_cast<const uint4*>(w), nblocks,
                         (const uint32_t*)amax_word, reinterpret_cast<uint2*>(packed), scales,
                         global_scale, dev_status) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  return NVFP4_OK;
}
