// gemv.cu -- batched NVFP4 W4A16 GEMV (m <= 8) with RMSNorm + concat fused on
// the input and greedy argmax fused on the output, for sm_103a.
//
// What it computes (the NVFP4 GEMV of the draft head, "metrale_model_layers/
// layers/mtp_head.rs" MtpHead::gemv, batched; norm/concat/argmax of the draft
// step in the same module and in "spark_model/layers/deepseek_v4_mtp.rs"):
//     a[m, :]   = concat_j( bf16(x_j[m, :] * rsqrt(mean(x_j^2) + eps_j) * gamma_j) )
//     y[m, n]   = g * sum_i a[m, i] * e4m3(s[n, i/16]) * e2m1(c[n, i])      (FP32)
//     argmax[m] = lowest n with y[m, n] maximal (NaN never wins)
//
// Design.  The kernel is bound by streaming the packed weights (0.5625 byte per
// weight incl. scales) from HBM.  On CUDA cores an 8-row batch would need 8 FP32
// FMAs per weight on top of the dequantisation, more instruction issue than the
// SMs have at HBM speed; so the inner product runs on the tensor cores with the
// legacy warp-level mma.sync m16n8k16 (BF16 in, FP32 accumulate) fed straight
// from registers: the 16-row A side is a weight tile dequantised in registers,
// the 8-column B side holds the (up to 8) activation rows.  That costs the same
// instructions per weight for m = 1..8.
//
//   * weights: each lane streams 16-byte vectors (ld.global.nc, L1 no-allocate)
//     of two rows, PF chunks of 128 K-elements ahead in registers;
//   * dequantisation: E2M1 nibbles -> BF16 bit patterns with two integer ops per
//     pair (value * 2^-126, exact, subnormal for the 0.5 code), then one packed
//     BF16 multiply by the block scale pre-multiplied by 2^118 (exact); the
//     final 2^8 and the global scale g meet the FP32 sum in the epilogue;
//   * the K order inside each 128-element chunk is permuted so that a lane's
//     16-byte load feeds its A fragments directly; the activations are laid out
//     once per CTA in shared memory in the same permuted fragment order (one
//     conflict-free 8-byte load per MMA), normalised on the way in;
//   * split-K inside the CTA (ks warps per 16-row tile) for small n, reduced in
//     a fixed order through shared memory (deterministic, so equal rows give
//     bit-equal logits);
//   * argmax: a 64-bit key (order-preserving float bits, inverted index) per
//     row, max-reduced per lane, warp, CTA, then one atomicMax per CTA; the last
//     CTA to finish converts the keys and returns the workspace to zero.
#include <cuda_fp8.h>

#include "common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 128;  // K elements per lane-group iteration (64 bytes per row)
constexpr int kPF = 2;       // chunks in flight per lane

struct GemvParams {
  const __nv_bfloat16* x[2];
  const __nv_bfloat16* gamma[2];
  int64_t kseg[2];
  int64_t ld[2];
  float eps[2];
  int nseg;
  int m;
  const uint8_t* packed;
  const uint8_t* scales;
  const float* gscale;
  int64_t n, k;
  void* y;
  int y_dtype;
  int64_t ldy;
  unsigned long long* keys;  // argmax mode when non-null
  unsigned int* counter;
  int32_t* argmax;
  int32_t* dev_status;
  int ks;          // warps sharing one 16-row tile (split K)
  int64_t ntiles;  // ceil(n / 16)
  int nchunks;     // ceil(k / 128)
};

__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two E4M3 block scales (low byte first) -> BF16 patterns of scale * 2^118,
// each replicated into both halves of a bf16x2.
__device__ __forceinline__ void decode_scales(uint32_t s2, uint32_t& lo, uint32_t& hi) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)s2, __NV_E4M3);
  // F16 -> BF16 by a 3-bit right shift: the exponent field lands unbiased-by-112,
  // i.e. the BF16 pattern holds value * 2^-112 (normal; zero stays zero).  The
  // F16 images of E4M3 values have their low 7 mantissa bits clear, so the shift
  // moves nothing across the half boundary.
  uint32_t v = ((uint32_t)h.x | ((uint32_t)h.y << 16)) >> 3;
  v = bf16x2_mul(v, 0x79007900u);  // * 2^115
  v = bf16x2_mul(v, 0x79007900u);  // * 2^115  -> scale * 2^118
  lo = __byte_perm(v, 0, 0x1010);
  hi = __byte_perm(v, 0, 0x3232);
}

// E2M1 nibble pair -> bf16x2 pattern (value * 2^-126).  x holds one nibble in
// each 16-bit half at bit offset 0 (mul = 0x1040) or 4 (mul = 0x104): the
// multiply makes two non-overlapping shifted copies, one placing the sign at
// bit 15, one placing the 3 magnitude bits at bits 8..6 (exponent LSBs +
// mantissa MSB); the mask keeps exactly those.
__device__ __forceinline__ uint32_t e2m1_pair(uint32_t x, uint32_t mul) {
  return (x * mul) & 0x81C081C0u;
}

// One 128-element chunk of one lane: weights qg (row g) / qh (row g + 8),
// scale pairs sg / sh, B fragments from shared memory.
__device__ __forceinline__ void chunk_mma(float (&acc)[4], const uint4& qg, const uint4& qh,
                                          uint32_t sg, uint32_t sh, const uint2* bfrag,
                                          int bstride, bool bact, int64_t bleft,
                                          int32_t* dev_status) {
  (void)bleft;
  (void)dev_status;
  uint32_t Sg[2], Sh[2];
  decode_scales(sg, Sg[0], Sg[1]);
  decode_scales(sh, Sh[0], Sh[1]);
  const uint32_t wg[4] = {qg.x, qg.y, qg.z, qg.w};
  const uint32_t wh[4] = {qh.x, qh.y, qh.z, qh.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint32_t sG = Sg[w >> 1], sH = Sh[w >> 1];
    const uint32_t g0 = wg[w], g8 = wg[w] >> 8;
    const uint32_t h0 = wh[w], h8 = wh[w] >> 8;
    const uint32_t ag0 = bf16x2_mul(e2m1_pair(g0 & 0x000F000Fu, 0x1040u), sG);  // nibbles 0,4
    const uint32_t ag1 = bf16x2_mul(e2m1_pair(g0 & 0x00F000F0u, 0x0104u), sG);  // 1,5
    const uint32_t ag2 = bf16x2_mul(e2m1_pair(g8 & 0x000F000Fu, 0x1040u), sG);  // 2,6
    const uint32_t ag3 = bf16x2_mul(e2m1_pair(g8 & 0x00F000F0u, 0x0104u), sG);  // 3,7
    const uint32_t ah0 = bf16x2_mul(e2m1_pair(h0 & 0x000F000Fu, 0x1040u), sH);
    const uint32_t ah1 = bf16x2_mul(e2m1_pair(h0 & 0x00F000F0u, 0x0104u), sH);
    const uint32_t ah2 = bf16x2_mul(e2m1_pair(h8 & 0x000F000Fu, 0x1040u), sH);
    const uint32_t ah3 = bf16x2_mul(e2m1_pair(h8 & 0x00F000F0u, 0x0104u), sH);
    uint2 b = make_uint2(0u, 0u);
    if (bact && NVFP4_GUARD((2 * w) * bstride < bleft, 7, dev_status)) b = bfrag[(2 * w) * bstride];
    mma_bf16_16816(acc, ag0, ah0, ag1, ah1, b.x, b.y);
    b = make_uint2(0u, 0u);
    if (bact && NVFP4_GUARD((2 * w + 1) * bstride < bleft, 7, dev_status))
      b = bfrag[(2 * w + 1) * bstride];
    mma_bf16_16816(acc, ag2, ah2, ag3, ah3, b.x, b.y);
  }
}

__device__ __forceinline__ unsigned long long argmax_key(float v, uint32_t idx) {
  if (!(v > -INFINITY)) return 0ull;  // -inf and NaN never win
  uint32_t b = (v == 0.0f) ? 0u : __float_as_uint(v);
  uint32_t o = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((unsigned long long)o << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ---------------------------------------------------------------- prologue
// Normalise (optionally) and lay out the activations as B fragments.
// Fragment layout: MMA index q = 8 * chunk + j, lane L = 4 * m + t (m < M):
// uint2 at bfrag[q * 4M + L].  For the 8 activations at
// kk = 128 c + 32 t + 8 w (+0..7):  MMA 8c+2w gets {a0,a4},{a1,a5};
// MMA 8c+2w+1 gets {a2,a6},{a3,a7}.
__device__ void build_fragments(const GemvParams& p, uint2* bfrag, float* rms) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int M = p.m;
  // 1. inverse RMS per (row, segment)
  for (int job = warp; job < M * p.nseg; job += kWarps) {
    const int r = job / p.nseg, s = job % p.nseg;
    if (p.gamma[s] == nullptr) {
      if (lane == 0) rms[job] = 1.0f;
      continue;
    }
    const __nv_bfloat16* xr = p.x[s] + (int64_t)r * p.ld[s];
    float ss = 0.0f;
    for (int64_t i = (int64_t)lane * 8; i < p.kseg[s]; i += 32 * 8) {
      if (!NVFP4_GUARD(r < M && s < p.nseg && i + 8 <= p.kseg[s], 1, p.dev_status)) continue;
      const uint4 v = *reinterpret_cast<const uint4*>(xr + i);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float a = __uint_as_float(u[j] << 16), b = __uint_as_float(u[j] & 0xFFFF0000u);
        ss = fmaf(a, a, ss);
        ss = fmaf(b, b, ss);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    if (lane == 0) rms[job] = 1.0f / sqrtf(ss / (float)p.kseg[s] + p.eps[s]);
  }
  __syncthreads();
  // 2. fragments
  const int64_t kpad = (int64_t)p.nchunks * kChunk;
  const int64_t groups = (int64_t)M * (kpad / 8);
  const int bstride = 4 * M;
  for (int64_t gi = tid; gi < groups; gi += kThreads) {
    const int r = (int)(gi / (kpad / 8));
    const int64_t kk = (gi % (kpad / 8)) * 8;
    uint32_t a[4] = {0u, 0u, 0u, 0u};  // bf16 pairs (a0,a1),(a2,a3),(a4,a5),(a6,a7)
    const int s = (p.nseg == 2 && kk >= p.kseg[0]) ? 1 : 0;
    const int64_t ko = kk - (s ? p.kseg[0] : 0);
    if (kk < p.k && NVFP4_GUARD(r < M && ko >= 0 && ko + 8 <= p.kseg[s], 2, p.dev_status)) {
      const uint4 v = *reinterpret_cast<const uint4*>(p.x[s] + (int64_t)r * p.ld[s] + ko);
      a[0] = v.x; a[1] = v.y; a[2] = v.z; a[3] = v.w;
      if (p.gamma[s] != nullptr) {
        const uint4 gv = *reinterpret_cast<const uint4*>(p.gamma[s] + ko);
        const uint32_t gg[4] = {gv.x, gv.y, gv.z, gv.w};
        const float rr = rms[r * p.nseg + s];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float lo = __uint_as_float(a[j] << 16) * rr * __uint_as_float(gg[j] << 16);
          const float hi =
              __uint_as_float(a[j] & 0xFFFF0000u) * rr * __uint_as_float(gg[j] & 0xFFFF0000u);
          a[j] = pack_bf16x2(lo, hi);
        }
      }
    }
    const int c = (int)(kk / kChunk), t = (int)((kk % kChunk) / 32), w = (int)((kk % 32) / 8);
    const int L = 4 * r + t;
    if (!NVFP4_GUARD((int64_t)(8 * c + 2 * w + 1) * bstride + L < (int64_t)p.nchunks * 8 * bstride &&
                         L < bstride, 3, p.dev_status))
      continue;
    // element e of the group lives in half (e & 1) of a[e >> 1]
    const uint32_t e0 = a[0] & 0xFFFFu, e1 = a[0] >> 16, e2 = a[1] & 0xFFFFu, e3 = a[1] >> 16;
    const uint32_t e4 = a[2] & 0xFFFFu, e5 = a[2] >> 16, e6 = a[3] & 0xFFFFu, e7 = a[3] >> 16;
    bfrag[(int64_t)(8 * c + 2 * w) * bstride + L] = make_uint2(e0 | (e4 << 16), e1 | (e5 << 16));
    bfrag[(int64_t)(8 * c + 2 * w + 1) * bstride + L] = make_uint2(e2 | (e6 << 16), e3 | (e7 << 16));
  }
}

// ------------------------------------------------------------------ kernel
__global__ void __launch_bounds__(kThreads)
gemv_kernel(const __grid_constant__ GemvParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int M = p.m;
  const int bstride = 4 * M;
  uint2* bfrag = reinterpret_cast<uint2*>(smem);
  const size_t bbytes = (size_t)p.nchunks * 8 * bstride * sizeof(uint2);
  float* red = reinterpret_cast<float*>(smem + bbytes);                // [kWarps][32][4]
  float* rms = red + kWarps * 32 * 4;                                  // [16]
  unsigned long long* kred = reinterpret_cast<unsigned long long*>(rms + 16);  // [kWarps][8]

  build_fragments(p, bfrag, rms);
  __syncthreads();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int ks = p.ks;
  const int tpc = kWarps / ks;  // tiles per CTA iteration
  const int slot = warp / ks, kpart = warp % ks;
  const int cpp = (p.nchunks + ks - 1) / ks;
  const int c_begin = kpart * cpp;
  const int c_end = min(p.nchunks, c_begin + cpp);
  const bool bact = lane < bstride;
  const float gs = __ldg(p.gscale) * 256.0f;  // g * 2^8 (the dequant fold)
  const int64_t rowbytes = p.k / 2, rowscales = p.k / 16;
  unsigned long long best[2] = {0ull, 0ull};

  for (int64_t base = (int64_t)blockIdx.x * tpc; base < p.ntiles; base += (int64_t)gridDim.x * tpc) {
    const int64_t tile = base + slot;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (tile < p.ntiles && c_begin < c_end) {
      const int64_t r0 = tile * 16 + g, r1 = r0 + 8;
      const bool v0 = r0 < p.n, v1 = r1 < p.n;
      const uint8_t* w0 = p.packed + (v0 ? r0 : 0) * rowbytes + 16 * t;
      const uint8_t* w1 = p.packed + (v1 ? r1 : 0) * rowbytes + 16 * t;
      const uint16_t* s0 = reinterpret_cast<const uint16_t*>(p.scales + (v0 ? r0 : 0) * rowscales) + t;
      const uint16_t* s1 = reinterpret_cast<const uint16_t*>(p.scales + (v1 ? r1 : 0) * rowscales) + t;
      uint4 qa[kPF], qb[kPF];
      uint32_t sa[kPF], sb[kPF];
      auto load = [&](int i, int c) {
        bool kv = c < c_end && (int64_t)c * kChunk + 32 * t < p.k;
        kv = kv && NVFP4_GUARD(!v0 || (r0 * rowbytes + 16 * t + (int64_t)c * 64 + 16 <= p.n * rowbytes &&
                                       r0 * rowscales + 2 * t + 8 * (int64_t)c + 2 <= p.n * rowscales),
                               4, p.dev_status);
        kv = kv && NVFP4_GUARD(!v1 || (r1 * rowbytes + 16 * t + (int64_t)c * 64 + 16 <= p.n * rowbytes &&
                                       r1 * rowscales + 2 * t + 8 * (int64_t)c + 2 <= p.n * rowscales),
                               5, p.dev_status);
        qa[i] = (kv && v0) ? ld_stream_u4(w0 + (int64_t)c * 64) : make_uint4(0, 0, 0, 0);
        qb[i] = (kv && v1) ? ld_stream_u4(w1 + (int64_t)c * 64) : make_uint4(0, 0, 0, 0);
        sa[i] = (kv && v0) ? (uint32_t)__ldg(s0 + 4 * c) : 0u;
        sb[i] = (kv && v1) ? (uint32_t)__ldg(s1 + 4 * c) : 0u;
      };
#pragma unroll
      for (int i = 0; i < kPF; ++i) load(i, c_begin + i);
      for (int c = c_begin; c < c_end; c += kPF) {
#pragma unroll
        for (int i = 0; i < kPF; ++i) {
          if (c + i < c_end) {
            const int64_t boff = (int64_t)(8 * (c + i)) * bstride + lane;
            chunk_mma(acc, qa[i], qb[i], sa[i], sb[i], bfrag + boff, bstride, bact,
                      (int64_t)p.nchunks * 8 * bstride - boff, p.dev_status);
            load(i, c + i + kPF);
          }
        }
      }
    }
    if (ks > 1) {
      float* mine = red + (warp * 32 + lane) * 4;
      if (kpart != 0) {
        mine[0] = acc[0]; mine[1] = acc[1]; mine[2] = acc[2]; mine[3] = acc[3];
      }
      __syncthreads();
      if (kpart == 0) {
        for (int j = 1; j < ks; ++j) {
          const float* o = red + ((warp + j) * 32 + lane) * 4;
          acc[0] += o[0]; acc[1] += o[1]; acc[2] += o[2]; acc[3] += o[3];
        }
      }
      __syncthreads();
    }
    if (kpart == 0 && tile < p.ntiles) {
      const int64_t rows[2] = {tile * 16 + g, tile * 16 + g + 8};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (rows[h] >= p.n) continue;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int mm = 2 * t + e;
          if (mm >= M) continue;
          const float v = acc[2 * h + e] * gs;
          if (p.y != nullptr && NVFP4_GUARD(mm < M && rows[h] < p.n && rows[h] < p.ldy, 6, p.dev_status)) {
            if (p.y_dtype == NVFP4_DTYPE_F32)
              reinterpret_cast<float*>(p.y)[mm * p.ldy + rows[h]] = v;
            else
              reinterpret_cast<__nv_bfloat16*>(p.y)[mm * p.ldy + rows[h]] = __float2bfloat16_rn(v);
          }
          if (p.keys != nullptr) {
            const unsigned long long key = argmax_key(v, (uint32_t)rows[h]);
            best[e] = key > best[e] ? key : best[e];
          }
        }
      }
    }
  }

  if (p.keys == nullptr) return;
  // argmax: lanes sharing t hold the same two rows of the batch
#pragma unroll
  for (int e = 0; e < 2; ++e) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, best[e], o);
      best[e] = other > best[e] ? other : best[e];
    }
  }
  if (g == 0) {
    kred[warp * 8 + 2 * t] = best[0];
    kred[warp * 8 + 2 * t + 1] = best[1];
  }
  __syncthreads();
  if (threadIdx.x < (unsigned)M) {
    unsigned long long b = 0ull;
    for (int w = 0; w < kWarps; ++w) {
      const unsigned long long o = kred[w * 8 + threadIdx.x];
      b = o > b ? o : b;
    }
    if (b != 0ull) atomicMax(p.keys + threadIdx.x, b);
  }
  __threadfence();
  __syncthreads();
  __shared__ bool last;
  if (threadIdx.x == 0) last = atomicAdd(p.counter, 1u) == gridDim.x - 1;
  __syncthreads();
  if (last) {
    __threadfence();
    if (threadIdx.x < (unsigned)M) {
      const unsigned long long key = atomicExch(p.keys + threadIdx.x, 0ull);
      p.argmax[threadIdx.x] =
          key == 0ull ? 0 : (int32_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
    }
    if (threadIdx.x == 0) atomicExch(p.counter, 0u);
  }
}

}  // namespace

int launch_gemv(const w4a16_act_segment* seg, int nseg, int m, const nvfp4_weight* w, void* y,
                int y_dtype, int64_t ldy, bool want_argmax, int32_t* argmax, void* workspace,
                int32_t* dev_status, cudaStream_t stream) {
  GemvParams p{};
  for (int s = 0; s < 2; ++s) {
    p.x[s] = s < nseg ? reinterpret_cast<const __nv_bfloat16*>(seg[s].x) : nullptr;
    p.gamma[s] = s < nseg ? reinterpret_cast<const __nv_bfloat16*>(seg[s].gamma) : nullptr;
    p.kseg[s] = s < nseg ? seg[s].k_seg : 0;
    p.ld[s] = s < nseg ? seg[s].ld : 0;
    p.eps[s] = s < nseg ? seg[s].eps : 0.f;
  }
  p.nseg = nseg;
  p.m = m;
  p.packed = w->packed;
  p.scales = w->scales;
  p.gscale = w->global_scale;
  p.n = w->n;
  p.k = w->k;
  p.y = y;
  p.y_dtype = y_dtype;
  p.ldy = ldy;
  if (want_argmax) {
    p.keys = reinterpret_cast<unsigned long long*>(workspace);
    p.counter = reinterpret_cast<unsigned int*>(reinterpret_cast<char*>(workspace) + 64);
    p.argmax = argmax;
  }
  p.dev_status = dev_status;
  p.ntiles = nvfp4::cdiv(w->n, 16);
  p.nchunks = (int)nvfp4::cdiv(w->k, kChunk);

  const size_t bbytes = (size_t)p.nchunks * 8 * 4 * m * sizeof(uint2);
  const size_t smem = bbytes + kWarps * 32 * 4 * sizeof(float) + 16 * sizeof(float) +
                      kWarps * 8 * sizeof(unsigned long long);
  const int occ = nvfp4::occupancy(reinterpret_cast<const void*>(gemv_kernel), kThreads, smem);
  if (occ < 1) return NVFP4_ERR_CUDA;
  const int sms = nvfp4::sm_count();
  const int64_t slots = (int64_t)sms * occ * kWarps;  // resident warps
  // split K until every resident warp has work, keeping >= 2 chunks per part
  int ks = 1;
  while (ks < kWarps && p.ntiles * ks < slots && p.nchunks / (2 * ks) >= 2) ks *= 2;
  p.ks = ks;
  const int tpc = kWarps / ks;
  int64_t grid = nvfp4::cdiv(p.ntiles, tpc);
  if (grid > (int64_t)sms * occ) grid = (int64_t)sms * occ;
  gemv_kernel<<<(unsigned)grid, kThreads, smem, stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
  return NVFP4_OK;
}
