// gemv.cu -- batched NVFP4 W4A16 GEMV (m <= 16) with RMSNorm + concat fused on
// the input and greedy argmax fused on the output, for sm_103a.
//
// What it computes (the NVFP4 GEMV of the draft head, "metrale_model_layers/
// layers/mtp_head.rs" MtpHead::gemv, batched; norm/concat/argmax of the draft
// step in the same module and in "spark_model/layers/deepseek_v4_mtp.rs"):
//     a[m, :]   = concat_j( bf16(x_j[m, :] * rsqrt(mean(x_j^2) + eps_j) * gamma_j) )
//     y[m, n]   = g * sum_i a[m, i] * e4m3(s[n, i/16]) * e2m1(c[n, i])      (FP32)
//     argmax[m] = lowest n with y[m, n] maximal (NaN never wins)
//
// Design.  The kernel is bound by streaming the weights from HBM (NVFP4: 0.5625
// byte per weight incl. scales; the FP8 variant: 1 byte + 4 per row).
//   * Weight stream: every warp owns a 2-stage shared-memory ring; one lane
//     issues a 2-D TMA copy (cp.async.bulk.tensor) per stage -- 16 rows x 128
//     bytes (two 128-element K chunks of NVFP4 codes) or 16 rows x 256 bytes
//     (two chunks of FP8 codes) -- with an mbarrier completion.  Rows past n
//     and bytes past k arrive as zeros (TMA bounds fill), which removes every
//     predicate from the loop.  NVFP4 block scales (2 bytes per lane and row
//     and chunk) are prefetched into registers at issue time.
//   * Products on the tensor cores: warp-level mma.sync m16n8k16 (FP16 in,
//     FP32 accumulate).  A = the 16-row weight tile: each E2M1 pair becomes an
//     exact f16x2 by the hardware conversion, times the block scale (E4M3 ->
//     F16, exact; the product has at most 6 significant bits); FP8 codes
//     convert pairwise with no scale (the row scale multiplies the sum).
//     B = the activation rows (8 MMA columns per column group; 9..16 rows use
//     two groups that share each dequantised A fragment), FP16 after an exact
//     per-row power-of-two scale that the epilogue removes.  On CUDA cores an
//     8-row batch would need 8 FP32 FMAs per weight on top of the
//     dequantisation; here the instruction count per weight does not depend
//     on m up to 8.
//   * Lane (g, t) of a warp reads rows g and g+8, K elements 32t..32t+31 of a
//     chunk; MMA 2w+u takes elements 32t+8w+4u .. +3, so one B fragment is four
//     consecutive activations, laid out in shared memory in that order (one
//     conflict-free 8-byte load per MMA), normalised on the way in: by every
//     CTA's prologue, or once per call by act_prep_kernel (m >= 2 with the
//     workspace) and then copied by one bulk copy.
//   * Split K inside the CTA (ks warps per 16-row tile) while there are fewer
//     tile groups than resident CTAs; partials are combined in a fixed order
//     (deterministic: equal weight rows give bit-equal logits).
//   * Argmax: a 64-bit key (order-preserving float bits, inverted index) per
//     row, max-reduced per lane, warp, CTA, then one atomic max per CTA and
//     row; the last CTA to finish converts the keys and returns the workspace
//     to zero.  Optional grammar mask and top-1 log-probability (an online
//     log-sum-exp per lane, per-CTA partials combined in a fixed order).
//   * Every mbarrier wait is bounded; one that runs out records
//     NVFP4_ERR_TIMEOUT, the lane waits no more and issues no further copies,
//     and before the CTA exits its copies still in flight are waited for
//     (bounded again).
#include <cuda.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace {

constexpr int kChunk = 128;       // K elements per chunk (64 packed bytes per row)
constexpr int kItem = 2;          // chunks per stage (one TMA box of 16 rows x 128 bytes)
constexpr int kStageBytes = 16 * 64 * kItem;
// FP8 weights: one ring stage is 16 rows x 256 bytes (two 128-element chunks
// of codes), so each row segment a TMA box reads is 256 contiguous bytes.
constexpr int kStageBytesFp8 = 16 * 256;
__host__ __device__ constexpr int stage_bytes(bool fp8) { return fp8 ? kStageBytesFp8 : kStageBytes; }
// TMA stages per warp (two two-chunk boxes: 4 KB in flight per warp; deeper
// rings measured no faster).
__host__ __device__ constexpr int ring_stages(int, int) { return 2; }
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
constexpr int kL2Prefetch = 4;    // items per warp pulled into L2 while the previous call ends

struct GemvParams {
  const __nv_bfloat16* x[2];
  const int32_t* ridx[2];  // gather indices per segment, or null
  int64_t tab_rows[2];     // rows of a gathered segment's table
  const __nv_bfloat16* gamma[2];
  int64_t kseg[2];
  int64_t ld[2];
  float eps[2];
  int nseg;
  int m;
  const uint8_t* scales;     // NVFP4: E4M3 block scales [n, k/16]
  const float* gscale;       // NVFP4: global scale
  const float* row_scale;    // FP8: per-row scales [n]
  int64_t n, k;
  void* y;
  int y_dtype;
  int64_t ldy;
  unsigned long long* keys;  // argmax mode when non-null
  unsigned int* counter;
  int32_t* argmax;
  float* logprob;            // top-1 log-probability per batch row, or null
  float2* lse;               // per-CTA (max, sum) log-sum-exp partials [grid][16]
  const int32_t* mask;       // grammar bitmask [m][ld_mask] int32 words, or null
  int64_t ld_mask;
  int32_t* dev_status;
  int ks;          // warps sharing one 16-row tile (split K)
  const uint2* frag_src;          // fragments prepared by act_prep_kernel, or null
  const unsigned int* rowmax_src; // their per-row scale carriers [8]
  int64_t ntiles;  // ceil(n / 16)
  int nchunks;     // ceil(k / 128)
  // shared-memory carve-up (bytes from the 1 KB-aligned base)
  uint32_t off_red, off_small, off_kred, off_ring, off_bar;
};

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait; false (and NVFP4_ERR_TIMEOUT recorded) if it ran out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int32_t* dev_status) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) {
      nvfp4::report(dev_status, NVFP4_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ void mma_f16_16816(float (&c)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two E4M3 block scales (low byte first) -> F16 (exact: E4M3 values are F16
// normals), each replicated into both halves of an f16x2.
__device__ __forceinline__ void decode_scales(uint32_t s2, uint32_t& lo, uint32_t& hi) {
  // both halves of lo (hi) carry the first (second) scale: the broadcast is
  // written as half moves, which the multiply can take as operand selects
  asm("{\n .reg .b16 a, b;\n .reg .b32 v;\n cvt.rn.f16x2.e4m3x2 v, %2;\n mov.b32 {a, b}, v;\n"
      " mov.b32 %0, {a, a};\n mov.b32 %1, {b, b};\n}"
      : "=r"(lo), "=r"(hi)
      : "h"((uint16_t)s2));
}

// The 8 E2M1 codes of word q -> 4 f16x2 (nibbles 0|1, 2|3, 4|5, 6|7; the even
// nibble in the low half) by the hardware conversion, exact.
__device__ __forceinline__ void e2m1_word_to_f16(uint32_t q, uint32_t& h0, uint32_t& h1,
                                                 uint32_t& h2, uint32_t& h3) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
      : "r"(q));
}

// One 128-element chunk of one lane: weights qg (row g) / qh (row g + 8),
// scale pairs sg / sh, B fragments from shared memory at bfrag[j * BSTRIDE]
// for MMA j (lanes whose batch column is >= M read a duplicate of a valid
// column: MMA columns are independent and those outputs are discarded).
// Lane (g, t) holds K elements 32t .. 32t+31 of the chunk; word w of its
// 16-byte load covers 32t + 8w .. +7, and MMA 2w+u takes the pairs of
// elements 4u .. 4u+3 of that word, so the MMA's column c = 2t + e + 8h is
// element 32t + 8w + 4u + 2h + e: a B fragment is 4 consecutive activations.
template <int BSTRIDE, int NCG, int GSTRIDE>
__device__ __forceinline__ void chunk_mma(float (&acc)[NCG][4], const uint4& qg, const uint4& qh,
                                          uint32_t sg, uint32_t sh, const uint2* bfrag) {
  uint32_t Sg[2], Sh[2];
  decode_scales(sg, Sg[0], Sg[1]);
  decode_scales(sh, Sh[0], Sh[1]);
  const uint32_t wg[4] = {qg.x, qg.y, qg.z, qg.w};
  const uint32_t wh[4] = {qh.x, qh.y, qh.z, qh.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint32_t sG = Sg[w >> 1], sH = Sh[w >> 1];
    uint32_t g0, g1, g2, g3, h0, h1, h2, h3;
    e2m1_word_to_f16(wg[w], g0, g1, g2, g3);
    e2m1_word_to_f16(wh[w], h0, h1, h2, h3);
    // one dequantised A fragment feeds the MMA of every column group
    const uint32_t a0 = f16x2_mul(g0, sG), a1 = f16x2_mul(h0, sH), a2 = f16x2_mul(g1, sG),
                   a3 = f16x2_mul(h1, sH);
#pragma unroll
    for (int cg = 0; cg < NCG; ++cg) {
      const uint2 b0 = bfrag[(2 * w) * BSTRIDE + cg * GSTRIDE];
      mma_f16_16816(acc[cg], a0, a1, a2, a3, b0.x, b0.y);
    }
    const uint32_t c0 = f16x2_mul(g2, sG), c1 = f16x2_mul(h2, sH), c2 = f16x2_mul(g3, sG),
                   c3 = f16x2_mul(h3, sH);
#pragma unroll
    for (int cg = 0; cg < NCG; ++cg) {
      const uint2 b1 = bfrag[(2 * w + 1) * BSTRIDE + cg * GSTRIDE];
      mma_f16_16816(acc[cg], c0, c1, c2, c3, b1.x, b1.y);
    }
  }
}

// FP8 weights: the lane's 32 codes of row g (g + 8) for one 128-element
// chunk are words W0..W7 of qg0, qg1 (qh0, qh1); MMA q takes word Wq (k
// elements 4q .. 4q+3 of the lane's 32, the same order as the NVFP4 path, so
// the activation fragments are shared).  No block scales: the row scale
// multiplies the finished sum.
__device__ __forceinline__ void e4m3_word_to_f16(uint32_t q, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n cvt.rn.f16x2.e4m3x2 %0, a;\n"
      " cvt.rn.f16x2.e4m3x2 %1, b;\n}"
      : "=r"(lo), "=r"(hi)
      : "r"(q));
}

template <int BSTRIDE, int NCG, int GSTRIDE>
__device__ __forceinline__ void chunk_mma_fp8(float (&acc)[NCG][4], const uint4& qg0, const uint4& qg1,
                                              const uint4& qh0, const uint4& qh1,
                                              const uint2* bfrag) {
  const uint32_t wg[8] = {qg0.x, qg0.y, qg0.z, qg0.w, qg1.x, qg1.y, qg1.z, qg1.w};
  const uint32_t wh[8] = {qh0.x, qh0.y, qh0.z, qh0.w, qh1.x, qh1.y, qh1.z, qh1.w};
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    uint32_t g0, g1, h0, h1;
    e4m3_word_to_f16(wg[q], g0, g1);
    e4m3_word_to_f16(wh[q], h0, h1);
#pragma unroll
    for (int cg = 0; cg < NCG; ++cg) {
      const uint2 b = bfrag[q * BSTRIDE + cg * GSTRIDE];
      mma_f16_16816(acc[cg], g0, h0, g1, h1, b.x, b.y);
    }
  }
}

__device__ __forceinline__ unsigned long long argmax_key(float v, uint32_t idx) {
  if (!(v > -INFINITY)) return 0ull;  // -inf and NaN never win
  uint32_t b = (v == 0.0f) ? 0u : __float_as_uint(v);
  uint32_t o = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((unsigned long long)o << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
}

// (m, s) <- log-sum-exp merge of (m, s) and (om, os), s the sum of exp(x - m).
__device__ __forceinline__ void lse_merge(float& m, float& s, float om, float os) {
  const float nm = fmaxf(m, om);
  if (nm == -INFINITY) return;  // both empty
  s = s * __expf(m - nm) + os * __expf(om - nm);
  m = nm;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 2^e (or 2^-e when inverse) for a row whose largest BF16 magnitude has the
// bit pattern `maxbits`: e = 14 - exponent(max), clamped to [-120, 120]; 1 for
// an all-zero row.
__device__ __forceinline__ float row_scale_pow2(unsigned int maxbits, bool inverse) {
  const int ef = (int)(maxbits >> 7);  // biased BF16 exponent
  int e = maxbits == 0u ? 0 : 14 - (ef == 0 ? -126 : ef - 127);
  e = e < -120 ? -120 : (e > 120 ? 120 : e);
  return ldexpf(1.0f, inverse ? -e : e);
}

// ---------------------------------------------------------------- prologue
// Normalise (optionally) and lay out the activations as B fragments.
// Fragment layout: MMA index q = 8 * chunk + j; batch row m, lane quad t:
// uint2 at bfrag[q * BSTRIDE + (m / 8) * GSTRIDE + 4 * (m % 8) + t], with
// GSTRIDE = 4 * min(M, 8) slots per column group and BSTRIDE = GSTRIDE times
// the number of column groups (one, or two for 9..16 rows).  For the 8 activations at
// kk = 128 c + 32 t + 8 w (+0..7):  MMA 8c+2w gets {a0,a4},{a1,a5};
// MMA 8c+2w+1 gets {a2,a6},{a3,a7}.  Positions past k are zero.
// Row r of segment s: row r of x, or, for a gathered segment, table row
// ridx[r] (out-of-range indices read row 0 and are reported).
__device__ __forceinline__ const __nv_bfloat16* seg_row(const GemvParams& p, int s, int r) {
  int64_t row = r;
  if (p.ridx[s] != nullptr) {
    row = __ldg(p.ridx[s] + r);
    if (row < 0 || row >= p.tab_rows[s]) {
      nvfp4::report(p.dev_status, NVFP4_ERR_INDEX);
      row = 0;
    }
  }
  return p.x[s] + row * p.ld[s];
}

// Shared "small" area (floats): [0,32) inverse RMS per (row, segment);
// [32,48) per-row scale exponent carrier (BF16 magnitude bits, see
// row_scale_pow2); [48,50) max |gamma| per segment; [64,96) max |x| per
// (row, segment); then per-(job, warp) partial sums of squares and maxima.
constexpr int kSmallRowmax = 32, kSmallMaxg = 48, kSmallMaxx = 64, kSmallParts = 96;
constexpr int kMaxJobs = 40;  // 16 rows x 2 segments + 2 gamma jobs, rounded up
constexpr int kMaxRows = 16;  // batch rows of one call (W4A16_GEMV_MAX_M)
__host__ __device__ constexpr int small_floats(int warps) { return kSmallParts + 2 * kMaxJobs * warps; }

// Kept out of line: the prologue's registers then do not compete with the
// main loop's (which hold the first ring stages' scales across it).
// Rows r0 .. r0+nrows-1 of the batch; bfrag may be shared or global memory
// (generic addresses), rowmax_out receives the rows' scale carriers too.
template <int M, int WARPS>
__device__ __noinline__ void build_fragments(const GemvParams& p, uint2* bfrag, float* small, int r0,
                                             int nrows, unsigned int* rowmax_out) {
  // fragment slots per MMA k-step: column groups of (up to) 8 batch rows
  constexpr int MC = M > 8 ? 8 : M, NCG = (M + 7) / 8, GSTRIDE = 4 * MC, BSTRIDE = GSTRIDE * NCG;
  constexpr int kWarps = WARPS, kThreads = WARPS * 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float* rms = small;
  unsigned int* rowmax = reinterpret_cast<unsigned int*>(small + kSmallRowmax);
  float* maxg = small + kSmallMaxg;
  float* maxx = small + kSmallMaxx;
  float* part_ss = small + kSmallParts;                                          // [job][warp]
  unsigned int* part_mx = reinterpret_cast<unsigned int*>(part_ss + kMaxJobs * kWarps);
  // 1. statistics.  Jobs 0 .. nrows*nseg-1: row r0 + job / nseg, segment
  //    job % nseg: sum of squares (RMSNorm segments) and the largest |x| (BF16
  //    magnitude bits order like the values).  Jobs nrows*nseg + s: the
  //    largest |gamma_s|.  The
  //    CTA's warps split each job's k range; partials are combined in a fixed
  //    order, so the result does not depend on timing.
  const int JR = nrows * p.nseg, J = JR + p.nseg;
  const int wpj = J >= kWarps ? 1 : kWarps / J;  // warps per job
  const int jpp = kWarps / wpj;                  // jobs per pass
  for (int j0 = 0; j0 < J; j0 += jpp) {
    const int job = j0 + warp / wpj, wj = warp % wpj;
    if (job < J) {
      const int s = job < JR ? job % p.nseg : job - JR;
      const bool is_gamma = job >= JR;
      const __nv_bfloat16* src =
          is_gamma ? p.gamma[s] : seg_row(p, s, r0 + job / p.nseg);
      const bool want_ss = !is_gamma && p.gamma[s] != nullptr;
      float ss = 0.0f;
      uint32_t mx = 0u;
      if (src != nullptr) {
#pragma unroll 4
        for (int i = (wj * 32 + lane) * 8; i < (int)p.kseg[s]; i += wpj * 256) {
          if (!NVFP4_GUARD(s < p.nseg && i + 8 <= p.kseg[s], 1, p.dev_status)) continue;
          const uint4 v = *reinterpret_cast<const uint4*>(src + i);
          const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            mx = __vmaxu2(mx, u[j] & 0x7FFF7FFFu);
            if (want_ss) {
              const float a = __uint_as_float(u[j] << 16), b = __uint_as_float(u[j] & 0xFFFF0000u);
              ss = fmaf(a, a, ss);
              ss = fmaf(b, b, ss);
            }
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
      mx = __reduce_max_sync(0xFFFFFFFFu, max(mx & 0xFFFFu, mx >> 16));
      if (lane == 0) {
        part_ss[job * kWarps + wj] = ss;
        part_mx[job * kWarps + wj] = mx;
      }
    }
  }
  __syncthreads();
  if (tid < J) {
    const int s = tid < JR ? tid % p.nseg : tid - JR;
    float ss = 0.0f;
    unsigned int mx = 0u;
    for (int w = 0; w < wpj; ++w) {
      ss += part_ss[tid * kWarps + w];
      mx = max(mx, part_mx[tid * kWarps + w]);
    }
    if (tid < JR) {
      rms[tid] = p.gamma[s] == nullptr ? 1.0f : 1.0f / sqrtf(ss / (float)p.kseg[s] + p.eps[s]);
      maxx[tid] = __uint_as_float(mx << 16);
    } else {
      maxg[s] = __uint_as_float(mx << 16);
    }
  }
  __syncthreads();
  // Per-row power of two 2^e from an upper bound B of the row's normalised
  // magnitudes (|bf16(x r gamma)| <= max|x| r max|gamma| (1 + 2^-7)): B 2^e
  // lies in [2^14, 2^15), so every activation converts to FP16 without
  // overflow, and exactly unless it is below 2^-29 B.
  if (tid < nrows) {
    float bound = 0.0f;
    for (int s = 0; s < p.nseg; ++s) {
      const int j = tid * p.nseg + s;
      const float b = p.gamma[s] == nullptr ? maxx[j] : maxx[j] * rms[j] * maxg[s] * (1.0f + 0.0078125f);
      bound = fmaxf(bound, b);
    }
    const unsigned int carrier = __float_as_uint(bound) >> 16;  // carries the bound's exponent
    rowmax[r0 + tid] = carrier;
    if (rowmax_out != nullptr) rowmax_out[r0 + tid] = carrier;
  }
  __syncthreads();
  // 2. normalised, scaled FP16 activations into the fragment slots.  The 8
  //    activations at kk = 128c + 32t + 8w of row m fill MMA 8c+2w (elements
  //    0..3) and MMA 8c+2w+1 (elements 4..7) of slot L(m, t) above.  Positions
  //    past k are zero.
  const int gpr = p.nchunks * (kChunk / 8);  // 8-element groups per row
  for (int r = r0; r < r0 + nrows; ++r) {
    const float sc = row_scale_pow2(rowmax[r], false);
    // the row's base in each segment, resolved once (a gathered row reads its index here)
    const __nv_bfloat16* xr0 = seg_row(p, 0, r);
    const __nv_bfloat16* xr1 = p.nseg == 2 ? seg_row(p, 1, r) : xr0;
#pragma unroll 2
    for (int q = tid; q < gpr; q += kThreads) {
      const int kk = q * 8;
      uint32_t a[4] = {0u, 0u, 0u, 0u};  // bf16 pairs (a0,a1),(a2,a3),(a4,a5),(a6,a7)
      const int s = (p.nseg == 2 && kk >= p.kseg[0]) ? 1 : 0;
      const int ko = kk - (s ? (int)p.kseg[0] : 0);
      if (kk < p.k && NVFP4_GUARD(ko >= 0 && ko + 8 <= p.kseg[s], 2, p.dev_status)) {
        const uint4 v = *reinterpret_cast<const uint4*>((s ? xr1 : xr0) + ko);
        a[0] = v.x; a[1] = v.y; a[2] = v.z; a[3] = v.w;
        if (p.gamma[s] != nullptr) {
          const uint4 gv = *reinterpret_cast<const uint4*>(p.gamma[s] + ko);
          const uint32_t gg[4] = {gv.x, gv.y, gv.z, gv.w};
          const float rr = rms[(r - r0) * p.nseg + s];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float lo = __uint_as_float(a[j] << 16) * rr * __uint_as_float(gg[j] << 16);
            const float hi =
                __uint_as_float(a[j] & 0xFFFF0000u) * rr * __uint_as_float(gg[j] & 0xFFFF0000u);
            a[j] = pack_bf16x2(lo, hi);
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // BF16 -> FP16, times 2^e (exact)
          const __half2 h = __floats2half2_rn(__uint_as_float(a[j] << 16) * sc,
                                              __uint_as_float(a[j] & 0xFFFF0000u) * sc);
          a[j] = *reinterpret_cast<const uint32_t*>(&h);
        }
      }
      const int c = kk / kChunk, t = (kk % kChunk) / 32, w = (kk % 32) / 8;
      const int L = (r / 8) * GSTRIDE + 4 * (r % 8) + t;
      if (!NVFP4_GUARD((8 * c + 2 * w + 1) * BSTRIDE + L < p.nchunks * 8 * BSTRIDE && L < BSTRIDE, 3,
                       p.dev_status))
        continue;
      bfrag[(8 * c + 2 * w) * BSTRIDE + L] = make_uint2(a[0], a[1]);
      bfrag[(8 * c + 2 * w + 1) * BSTRIDE + L] = make_uint2(a[2], a[3]);
    }
  }
}

// One CTA per batch row: normalise, scale and convert the row's activations
// once into the fragment layout in global memory, for every GEMV CTA to copy.
// It waits for the previous grid before reading x and lets the GEMV start
// right after (the GEMV reads the fragments only after its own wait).
template <int M>
__global__ void __launch_bounds__(512) act_prep_kernel(const __grid_constant__ GemvParams p, uint2* frag,
                                                       unsigned int* rowmax) {
  __shared__ __align__(16) float small[small_floats(16)];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  build_fragments<M, 16>(p, frag, small, (int)blockIdx.x, 1, rowmax);
}

// Named barriers over the `count` threads of one tile group: the split-K
// partials go from the ks-1 producer warps to the tile's first warp through a
// "full" barrier (ids 1..4: producers arrive, the consumer waits); an "empty"
// barrier (ids 5..8: the consumer arrives after reading tile t, producers wait
// on it before publishing tile t+1) keeps every producer from arriving twice
// on a full barrier before it completes.  Split factors are 1, 4, 8 or 16, so
// at most 4 tile groups share a CTA.
__device__ __forceinline__ void bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ------------------------------------------------------------------ kernel
// Work split: WARPS warps per CTA; ks warps share one 16-row tile, each taking
// a contiguous range of its k chunks (split K); a CTA takes WARPS/ks tiles at a
// time and strides over the tiles persistently.  Each warp streams its
// (tile, chunk) items in order through its TMA ring, across tile boundaries.
template <int M, int WARPS, bool FP8>
__global__ void __launch_bounds__(WARPS * 32, (WARPS >= 16 && M <= 8) ? 2 : 1)
gemv_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ GemvParams p) {
  // M <= 8: one MMA column per batch row.  M = 16 (any 9..16 rows): two column
  // groups of 8 share every dequantised A fragment; MM is the call's row count.
  constexpr int MC = M > 8 ? 8 : M, NCG = (M + 7) / 8, GSTRIDE = 4 * MC, BSTRIDE = GSTRIDE * NCG;
  const int MM = M > 8 ? p.m : M;
  constexpr int kRing = ring_stages(M, WARPS);
  constexpr int kWarps = WARPS;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw));
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* const smem = smem_raw + (base - raw);
  uint2* bfrag = reinterpret_cast<uint2*>(smem);
  float* red = reinterpret_cast<float*>(smem + p.off_red);  // [kWarps][32][4]
  float* rms = reinterpret_cast<float*>(smem + p.off_small);
  unsigned long long* kred = reinterpret_cast<unsigned long long*>(smem + p.off_kred);

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int ks = p.ks;
  const int tpc = kWarps / ks;  // tiles per CTA iteration
  const int slot = warp / ks, kpart = warp % ks;
  // this warp's items (pairs of chunks) [ib, ib + L) of every tile
  constexpr int kIt = kItem;               // chunks per ring stage
  constexpr int kStage = stage_bytes(FP8);  // 16 rows x 128 (NVFP4) or 256 (FP8) bytes
  constexpr int kRowBytes = kStage / 16;
  const int nitems = (p.nchunks + kIt - 1) / kIt;
  const int ib = (int)((int64_t)kpart * nitems / ks);
  const int L = (int)((int64_t)(kpart + 1) * nitems / ks) - ib;
  const int64_t ngroups = (p.ntiles + tpc - 1) / tpc;
  const int n_iter = blockIdx.x < ngroups ? (int)((ngroups - 1 - blockIdx.x) / gridDim.x) + 1 : 0;
  const uint32_t ring = base + p.off_ring + (uint32_t)warp * (kRing * kStage);
  const uint32_t bars = base + p.off_bar + (uint32_t)warp * (kRing * 8);
  // chunks c with 128c + 32t < k hold this lane's data (scales past k read 0)
  const int cmax = (int)((p.k - 32 * t + kChunk - 1) / kChunk);
  // The item whose wait ran out in this lane (kAlive while none has): from
  // then on the lane waits no more and lane 0 issues no further copies.
  constexpr int kAlive = 0x7FFFFFFF;
  int failed_at = kAlive;

  const bool prepped = p.frag_src != nullptr;
  const uint32_t fbar = base + p.off_bar + (uint32_t)kWarps * (kRing * 8);  // fragment copy
  if (lane == 0) {
    for (int i = 0; i < kRing; ++i) mbar_init(bars + 8 * i, 1);
    if (threadIdx.x == 0) mbar_init(fbar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (prepped) __syncthreads();  // fbar initialised before any thread waits on it
  __syncwarp();

  // load cursor over (tile, item); scale row pointers change once per tile
  int lt = 0, lc = 0;
  int ltile16 = 0;
  const uint16_t* sp0 = nullptr;
  const uint16_t* sp1 = nullptr;
  auto set_tile = [&](int it) {
    const int64_t tile = ((int64_t)blockIdx.x + (int64_t)it * gridDim.x) * tpc + slot;
    ltile16 = (int)(tile * 16);
    int64_t r0 = tile * 16 + g, r1 = r0 + 8;
    r0 = r0 < p.n ? r0 : p.n - 1;  // rows past n: any valid scale (their codes read as 0)
    r1 = r1 < p.n ? r1 : p.n - 1;
    if constexpr (!FP8) {
      sp0 = reinterpret_cast<const uint16_t*>(p.scales + r0 * (p.k / 16)) + t;
      sp1 = reinterpret_cast<const uint16_t*>(p.scales + r1 * (p.k / 16)) + t;
    }
  };
  const int total = n_iter * L;
  uint32_t sreg[kRing][kItem];  // block-scale pairs of rows g, g+8 (low / high 16 bits)
  if (total > 0) set_tile(0);
  auto issue = [&](int i) {
    const int c0 = (ib + lc) * kIt;
    if (lane == 0 && failed_at == kAlive) {
      mbar_arrive_expect_tx(bars + 8 * i, kStage);
      tma_load_2d(ring + i * kStage, &tmap_w, (ib + lc) * kRowBytes, ltile16, bars + 8 * i);
    }
    if constexpr (!FP8) {
#pragma unroll
      for (int j = 0; j < kItem; ++j) {
        const int c = c0 + j;
        sreg[i][j] = c < cmax ? ((uint32_t)__ldg(sp0 + 4 * c) | ((uint32_t)__ldg(sp1 + 4 * c) << 16)) : 0u;
      }
    }
    if (++lc == L) {
      lc = 0;
      if (++lt < n_iter) set_tile(lt);
    }
  };
  // Back-to-back calls (programmatic dependent launch): let the next grid
  // start now, pull this warp's first weight boxes into L2 (a hint only: L2 is
  // the point of coherence, so this is correct even if the previous kernel on
  // the stream is still writing them), then wait for the previous grid to
  // finish before reading anything.  Without PDL both controls are no-ops.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (lane == 0) {
    int pt = 0, pc = 0;
    for (int q = 0; q < total && q < kL2Prefetch; ++q) {
      const int64_t tile = ((int64_t)blockIdx.x + (int64_t)pt * gridDim.x) * tpc + slot;
      asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global [%0, {%1, %2}];" ::"l"(
                       reinterpret_cast<uint64_t>(&tmap_w)),
                   "r"((ib + pc) * kRowBytes), "r"((int)(tile * 16))
                   : "memory");
      if (++pc == L) { pc = 0; ++pt; }
    }
  }
  // With prepared fragments the previous grid is act_prep_kernel, which let
  // this grid start only after its own predecessor had finished: the weights
  // are final, so the first ring stages may load before the wait.
  if (prepped) {
#pragma unroll
    for (int i = 0; i < kRing; ++i)
      if (i < total) issue(i);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (prepped) {
    // one bulk copy of the prepared fragments and row-scale carriers
    if (threadIdx.x == 0) {
      const uint32_t fbytes = (uint32_t)p.nchunks * 8u * BSTRIDE * 8u;
      mbar_arrive_expect_tx(fbar, fbytes + 4u * kMaxRows);
      const uint32_t dst = base;  // bfrag
      for (uint32_t off = 0; off < fbytes; off += 32768u) {
        const uint32_t n = fbytes - off < 32768u ? fbytes - off : 32768u;
        bulk_copy_g2s(dst + off, reinterpret_cast<const char*>(p.frag_src) + off, n, fbar);
      }
      bulk_copy_g2s(base + p.off_small + kSmallRowmax * 4u, p.rowmax_src, 4u * kMaxRows, fbar);
    }
    if (!mbar_wait(fbar, 0u, p.dev_status)) failed_at = 0;
  } else {
    // start streaming before the activation prologue
#pragma unroll
    for (int i = 0; i < kRing; ++i)
      if (i < total) issue(i);
    if (n_iter > 0 || blockIdx.x == 0) build_fragments<M, WARPS>(p, bfrag, rms, 0, MM, nullptr);
  }
  __syncthreads();

  const float gsc = FP8 ? 1.0f : __ldg(p.gscale);
  // inverse activation scales of this lane's two batch columns (2t, 2t+1)
  const unsigned int* rowmax = reinterpret_cast<const unsigned int*>(rms + kSmallRowmax);
  float inv[NCG][2];  // inverse activation scales of this lane's columns 8cg + 2t + e
#pragma unroll
  for (int cg = 0; cg < NCG; ++cg)
#pragma unroll
    for (int e = 0; e < 2; ++e) inv[cg][e] = row_scale_pow2(rowmax[min(8 * cg + 2 * t + e, MM - 1)], true);
  const uint2* bbase = bfrag + (lane % GSTRIDE);
  unsigned long long best[NCG][2];  // running argmax keys, columns 8cg + 2t + e
  float lm[NCG][2], ls[NCG][2];      // log-sum-exp (max, sum)
  float acc[NCG][4];
#pragma unroll
  for (int cg = 0; cg < NCG; ++cg) {
    best[cg][0] = best[cg][1] = 0ull;
    lm[cg][0] = lm[cg][1] = -INFINITY;
    ls[cg][0] = ls[cg][1] = 0.f;
    acc[cg][0] = acc[cg][1] = acc[cg][2] = acc[cg][3] = 0.f;
  }
  int ct = 0, cc = 0;  // compute cursor

  // Grammar mask: the 16 rows of a tile share one 32-bit mask word per batch
  // column; the consumer warp loads the next tile's words during this tile.
  // FP8: the row scales of the consumer's rows g, g + 8, loaded the same way.
  uint32_t mword[NCG][2];
#pragma unroll
  for (int cg = 0; cg < NCG; ++cg) mword[cg][0] = mword[cg][1] = 0xFFFFFFFFu;
  float rsc[2] = {0.f, 0.f};
  auto load_mask = [&](int it) {
    if (!FP8 && p.mask == nullptr) return;
    const int64_t tile = ((int64_t)blockIdx.x + (int64_t)it * gridDim.x) * tpc + slot;
    if (it >= n_iter || tile >= p.ntiles) return;
    if constexpr (FP8) {
#pragma unroll
      for (int h = 0; h < 2; ++h) rsc[h] = __ldg(p.row_scale + min(tile * 16 + g + 8 * h, p.n - 1));
    }
    if (p.mask == nullptr) return;
#pragma unroll
    for (int cg = 0; cg < NCG; ++cg)
#pragma unroll
      for (int e = 0; e < 2; ++e)
        mword[cg][e] = __ldg(reinterpret_cast<const uint32_t*>(p.mask) +
                             min(8 * cg + 2 * t + e, MM - 1) * p.ld_mask + (tile >> 1));
  };
  if (kpart == 0) load_mask(0);

  auto epilogue = [&](int it) {
    const int64_t tile = ((int64_t)blockIdx.x + (int64_t)it * gridDim.x) * tpc + slot;
    if (ks > 1) {
      const int full_id = 1 + slot, empty_id = 5 + slot;  // slot < 4 when ks >= 4
      float* mine = red + (warp * 32 + lane) * 4 * NCG;
      if (kpart != 0) {
        // the consumer has finished tile it-1 (so no producer can arrive on the
        // full barrier twice before it completes, and the buffer is free)
        if (it >= 1) bar_sync(empty_id, ks * 32);
#pragma unroll
        for (int cg = 0; cg < NCG; ++cg)
#pragma unroll
          for (int i = 0; i < 4; ++i) mine[4 * cg + i] = acc[cg][i];
        bar_arrive(full_id, ks * 32);
      } else {
        bar_sync(full_id, ks * 32);
        for (int j = 1; j < ks; ++j) {
          const float* o = red + ((warp + j) * 32 + lane) * 4 * NCG;
#pragma unroll
          for (int cg = 0; cg < NCG; ++cg)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[cg][i] += o[4 * cg + i];
        }
        bar_arrive(empty_id, ks * 32);
      }
    }
    if (kpart == 0 && tile < p.ntiles) {
      const int64_t rows[2] = {tile * 16 + g, tile * 16 + g + 8};
#pragma unroll
      for (int cg = 0; cg < NCG; ++cg) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (rows[h] >= p.n) continue;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int mm = 8 * cg + 2 * t + e;
            if (mm >= MM) continue;
            const float v = (acc[cg][2 * h + e] * inv[cg][e]) * (FP8 ? rsc[h] : gsc);
            if (p.y != nullptr &&
                NVFP4_GUARD(mm < MM && rows[h] < p.n && rows[h] < p.ldy, 6, p.dev_status)) {
              if (p.y_dtype == NVFP4_DTYPE_F32)
                reinterpret_cast<float*>(p.y)[mm * p.ldy + rows[h]] = v;
              else
                reinterpret_cast<__nv_bfloat16*>(p.y)[mm * p.ldy + rows[h]] = __float2bfloat16_rn(v);
            }
            if (p.keys != nullptr && ((mword[cg][e] >> (((int)(tile & 1) << 4) + g + 8 * h)) & 1u)) {
              const unsigned long long key = argmax_key(v, (uint32_t)rows[h]);
              best[cg][e] = key > best[cg][e] ? key : best[cg][e];
              if (p.logprob != nullptr) {  // online log-sum-exp over the allowed logits
                if (v > lm[cg][e]) {
                  ls[cg][e] = ls[cg][e] * __expf(lm[cg][e] - v) + 1.0f;
                  lm[cg][e] = v;
                } else {
                  ls[cg][e] += __expf(v - lm[cg][e]);
                }
              }
            }
          }
        }
      }
    }
    if (kpart == 0) load_mask(it + 1);
#pragma unroll
    for (int cg = 0; cg < NCG; ++cg) acc[cg][0] = acc[cg][1] = acc[cg][2] = acc[cg][3] = 0.f;
  };

  for (int q0 = 0; q0 < total; q0 += kRing) {
#pragma unroll
    for (int i = 0; i < kRing; ++i) {
      const int q = q0 + i;
      if (q < total) {
        if (failed_at == kAlive && !mbar_wait(bars + 8 * i, (uint32_t)(q / kRing) & 1u, p.dev_status))
          failed_at = q;
        const unsigned char* st = smem + (ring - base) + i * kStage;
        const uint2* bq = bbase + (int64_t)(8 * kIt * (ib + cc)) * BSTRIDE;
        if constexpr (FP8) {  // box rows are two 128-element chunks of codes
#pragma unroll
          for (int j = 0; j < kItem; ++j) {
            const unsigned char* rg = st + g * kRowBytes + j * 128 + t * 32;
            const unsigned char* rh = st + (g + 8) * kRowBytes + j * 128 + t * 32;
            const uint4 qg0 = *reinterpret_cast<const uint4*>(rg);
            const uint4 qg1 = *reinterpret_cast<const uint4*>(rg + 16);
            const uint4 qh0 = *reinterpret_cast<const uint4*>(rh);
            const uint4 qh1 = *reinterpret_cast<const uint4*>(rh + 16);
            chunk_mma_fp8<BSTRIDE, NCG, GSTRIDE>(acc, qg0, qg1, qh0, qh1, bq + 8 * j * BSTRIDE);
          }
        } else {
#pragma unroll
          for (int j = 0; j < kItem; ++j) {  // box rows are 64 * kItem bytes
            const uint4 qg = *reinterpret_cast<const uint4*>(st + g * (64 * kItem) + j * 64 + t * 16);
            const uint4 qh =
                *reinterpret_cast<const uint4*>(st + (g + 8) * (64 * kItem) + j * 64 + t * 16);
            const uint32_t s2 = sreg[i][j];
            chunk_mma<BSTRIDE, NCG, GSTRIDE>(acc, qg, qh, s2 & 0xFFFFu, s2 >> 16, bq + 8 * j * BSTRIDE);
          }
        }
        __syncwarp();  // every lane is done with stage i before it is refilled
        if (q + kRing < total) issue(i);
        if (++cc == L) {
          epilogue(ct);
          cc = 0;
          ++ct;
        }
      }
    }
  }
  if (L == 0)  // no chunk for this warp: still take part in every tile's epilogue
    for (int it = 0; it < n_iter; ++it) epilogue(it);

  if (ks > 1 && kpart != 0 && n_iter > 0)  // match the consumer's last "empty" arrival
    bar_sync(5 + slot, ks * 32);
  // After a wait ran out in lane 0, the copies of items failed_at ..
  // failed_at + kRing - 1 (the last one on each ring stage) may still be in
  // flight, and thread 0's fragment copy too: wait for them, again bounded,
  // before the CTA's shared memory can be released.
  if (lane == 0 && failed_at != kAlive) {
    for (int q = failed_at; q < total && q < failed_at + kRing; ++q)
      mbar_wait(bars + 8 * (q % kRing), (uint32_t)(q / kRing) & 1u, p.dev_status);
    if (threadIdx.x == 0 && prepped) mbar_wait(fbar, 0u, p.dev_status);
  }

  if (p.keys == nullptr) return;
  // lanes sharing t hold the same batch columns: reduce over g, then per warp
  float2* lred = reinterpret_cast<float2*>(kred + kWarps * kMaxRows);  // [kWarps][kMaxRows]
#pragma unroll
  for (int cg = 0; cg < NCG; ++cg) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, best[cg][e], o);
        best[cg][e] = other > best[cg][e] ? other : best[cg][e];
        if (p.logprob != nullptr) {
          const float om = __shfl_xor_sync(0xFFFFFFFFu, lm[cg][e], o);
          const float os = __shfl_xor_sync(0xFFFFFFFFu, ls[cg][e], o);
          lse_merge(lm[cg][e], ls[cg][e], om, os);
        }
      }
      if (g == 0) {
        kred[warp * kMaxRows + 8 * cg + 2 * t + e] = best[cg][e];
        if (p.logprob != nullptr) lred[warp * kMaxRows + 8 * cg + 2 * t + e] = make_float2(lm[cg][e], ls[cg][e]);
      }
    }
  }
  __syncthreads();
  if (threadIdx.x < (unsigned)MM) {
    const int m = threadIdx.x;
    unsigned long long b = 0ull;
    for (int w = 0; w < kWarps; ++w) {
      const unsigned long long o = kred[w * kMaxRows + m];
      b = o > b ? o : b;
    }
    if (b != 0ull)
      asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(p.keys + m), "l"(b) : "memory");
    if (p.logprob != nullptr) {  // this CTA's log-sum-exp partial, combined in CTA order below
      float cm = -INFINITY, cs = 0.f;
      for (int w = 0; w < kWarps; ++w)
        lse_merge(cm, cs, lred[w * kMaxRows + m].x, lred[w * kMaxRows + m].y);
      p.lse[(int64_t)blockIdx.x * kMaxRows + m] = make_float2(cm, cs);
    }
  }
  // Count the finished CTAs with an acquire-release add: the barrier orders this
  // CTA's key updates before thread 0's release, and the last CTA's acquire
  // makes every CTA's keys visible to it, without separate fences.
  __syncthreads();
  __shared__ unsigned int prev;
  if (threadIdx.x == 0) {
    unsigned int v;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(v) : "l"(p.counter) : "memory");
    prev = v;
  }
  __syncthreads();
  if (prev == gridDim.x - 1) {  // the last CTA: convert the keys and re-zero the workspace
    if (p.logprob != nullptr) {
      // combine the per-CTA log-sum-exp partials: CTA b goes to thread b mod
      // blockDim, then a fixed shuffle tree and a fixed pass over the warps,
      // so the result does not depend on which CTA finished last
      for (int m = 0; m < MM; ++m) {
        float cm = -INFINITY, cs = 0.f;
        for (unsigned int b = threadIdx.x; b < gridDim.x; b += blockDim.x) {
          float2 v;
          asm volatile("ld.relaxed.gpu.global.v2.f32 {%0, %1}, [%2];"
                       : "=f"(v.x), "=f"(v.y)
                       : "l"(p.lse + (int64_t)b * kMaxRows + m)
                       : "memory");
          lse_merge(cm, cs, v.x, v.y);
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float om = __shfl_xor_sync(0xFFFFFFFFu, cm, o);
          const float os = __shfl_xor_sync(0xFFFFFFFFu, cs, o);
          lse_merge(cm, cs, om, os);
        }
        if (lane == 0) lred[warp * kMaxRows + m] = make_float2(cm, cs);
      }
      __syncthreads();
    }
    if (threadIdx.x < (unsigned)MM) {
      unsigned long long key;
      asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(key) : "l"(p.keys + threadIdx.x) : "memory");
      asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p.keys + threadIdx.x), "l"(0ull) : "memory");
      p.argmax[threadIdx.x] =
          key == 0ull ? 0 : (int32_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
      if (p.logprob != nullptr) {
        float cm = -INFINITY, cs = 0.f;
        for (int w = 0; w < kWarps; ++w)
          lse_merge(cm, cs, lred[w * kMaxRows + threadIdx.x].x, lred[w * kMaxRows + threadIdx.x].y);
        // the winning logit back from its key (inverse of the order-preserving map)
        const uint32_t o = (uint32_t)(key >> 32);
        const float ymax = __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
        p.logprob[threadIdx.x] = key == 0ull ? __int_as_float(0x7FC00000) : ymax - (cm + logf(cs));
      }
    }
    if (threadIdx.x == 0)
      asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p.counter), "r"(0u) : "memory");
  }
}

using KernelFn = void (*)(CUtensorMap, GemvParams);
using PrepFn = void (*)(GemvParams, uint2*, unsigned int*);

PrepFn prep_for(int m) {
  switch (m) {
    case 1: return act_prep_kernel<1>;
    case 2: return act_prep_kernel<2>;
    case 3: return act_prep_kernel<3>;
    case 4: return act_prep_kernel<4>;
    case 5: return act_prep_kernel<5>;
    case 6: return act_prep_kernel<6>;
    case 7: return act_prep_kernel<7>;
    case 8: return act_prep_kernel<8>;
    default: return act_prep_kernel<16>;
  }
}

template <int WARPS, bool FP8>
KernelFn kernel_for(int m) {
  switch (m) {
    case 1: return gemv_kernel<1, WARPS, FP8>;
    case 2: return gemv_kernel<2, WARPS, FP8>;
    case 3: return gemv_kernel<3, WARPS, FP8>;
    case 4: return gemv_kernel<4, WARPS, FP8>;
    case 5: return gemv_kernel<5, WARPS, FP8>;
    case 6: return gemv_kernel<6, WARPS, FP8>;
    case 7: return gemv_kernel<7, WARPS, FP8>;
    case 8: return gemv_kernel<8, WARPS, FP8>;
    default: return gemv_kernel<16, WARPS, FP8>;  // 9..16 rows
  }
}

struct Layout {
  uint32_t off_red, off_small, off_kred, off_ring, off_bar;
  size_t bytes;  // dynamic shared memory to request (includes 1 KB alignment slack)
};

Layout layout_for(int warps, int m, int nchunks, bool fp8) {
  const int kRing = ring_stages(m, warps);
  Layout l;
  const int cols = m <= 8 ? m : 16, ncg = (m + 7) / 8;        // the kernel's M, column groups
  size_t off = (size_t)nchunks * 8 * 4 * cols * sizeof(uint2);  // B fragments
  l.off_red = (uint32_t)off;
  off += (size_t)warps * 32 * 4 * ncg * sizeof(float);
  l.off_small = (uint32_t)off;
  off += (size_t)small_floats(warps) * sizeof(float);
  off = (off + 15) & ~(size_t)15;
  l.off_kred = (uint32_t)off;
  off += (size_t)warps * kMaxRows * sizeof(unsigned long long) + (size_t)warps * kMaxRows * sizeof(float2);
  off = (off + 1023) & ~(size_t)1023;
  l.off_ring = (uint32_t)off;
  off += (size_t)warps * kRing * stage_bytes(fp8);
  l.off_bar = (uint32_t)off;
  off += (size_t)warps * kRing * 8 + 8;  // ring barriers + the fragment-copy barrier
  l.bytes = off + 1024;
  return l;
}

}  // namespace

int launch_gemv(const w4a16_act_segment* seg, int nseg, int m, const WeightRef& w, void* y,
                int y_dtype, int64_t ldy, bool want_argmax, int32_t* argmax, void* workspace,
                size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream, float* logprob,
                const int32_t* mask, int64_t ld_mask) {
  GemvParams p{};
  for (int s = 0; s < 2; ++s) {
    p.x[s] = s < nseg ? reinterpret_cast<const __nv_bfloat16*>(seg[s].x) : nullptr;
    p.ridx[s] = s < nseg ? seg[s].row_index : nullptr;
    p.tab_rows[s] = s < nseg ? seg[s].index_rows : 0;
    p.gamma[s] = s < nseg ? reinterpret_cast<const __nv_bfloat16*>(seg[s].gamma) : nullptr;
    p.kseg[s] = s < nseg ? seg[s].k_seg : 0;
    p.ld[s] = s < nseg ? seg[s].ld : 0;
    p.eps[s] = s < nseg ? seg[s].eps : 0.f;
  }
  p.nseg = nseg;
  p.m = m;
  p.scales = w.scales;
  p.gscale = w.gscale;
  p.row_scale = w.row_scale;
  p.n = w.n;
  p.k = w.k;
  p.y = y;
  p.y_dtype = y_dtype;
  p.ldy = ldy;
  if (want_argmax) {
    p.keys = reinterpret_cast<unsigned long long*>(workspace);
    p.counter = reinterpret_cast<unsigned int*>(reinterpret_cast<char*>(workspace) + 8 * kMaxRows);
    p.argmax = argmax;
    p.logprob = logprob;
    p.mask = mask;
    p.ld_mask = ld_mask;
    p.lse = reinterpret_cast<float2*>(reinterpret_cast<char*>(workspace) + W4A16_ARGMAX_WS_BYTES);
  }
  p.dev_status = dev_status;
  p.ntiles = nvfp4::cdiv(w.n, 16);
  // Round k's chunks up to whole items (two chunks per ring stage); the
  // padding chunk's activations are zero and its weights arrive as zeros (TMA
  // bounds fill).
  const int item_chunks = kItem;
  p.nchunks = (int)(nvfp4::cdiv(nvfp4::cdiv(w.k, kChunk), item_chunks) * item_chunks);
  const int nitems = p.nchunks / item_chunks;
  if (p.ntiles * 16 > 0x7FFFFFFFLL) return NVFP4_ERR_SHAPE;  // TMA row coordinate

  // 16-warp CTAs when their shared memory fits, else 8-warp CTAs.
  int warps = 16;
  Layout lay = layout_for(16, m, p.nchunks, w.fp8);
  KernelFn fn = w.fp8 ? kernel_for<16, true>(m) : kernel_for<16, false>(m);
  int occ = nvfp4::occupancy(reinterpret_cast<const void*>(fn), 16 * 32, lay.bytes);
  if (occ < 1) {
    warps = 8;
    lay = layout_for(8, m, p.nchunks, w.fp8);
    fn = w.fp8 ? kernel_for<8, true>(m) : kernel_for<8, false>(m);
    occ = nvfp4::occupancy(reinterpret_cast<const void*>(fn), 8 * 32, lay.bytes);
  }
  if (occ < 1) {
    // the activation fragments (2 m k bytes) plus the weight ring do not fit
    // one CTA's shared memory: a size limit of the call, not a launch failure
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess &&
        lay.bytes > (size_t)optin)
      return NVFP4_ERR_SHAPE;
    return NVFP4_ERR_CUDA;
  }
  p.off_red = lay.off_red;
  p.off_small = lay.off_small;
  p.off_kred = lay.off_kred;
  p.off_ring = lay.off_ring;
  p.off_bar = lay.off_bar;

  CUtensorMap tmap;
  const int64_t row_bytes = w.fp8 ? w.k : w.k / 2;
  const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)w.n};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)(stage_bytes(w.fp8) / 16), 16};  // one ring stage
  const cuuint32_t estr[2] = {1, 1};
  if (!nvfp4::encode_tiled(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(w.codes),
                           dims, strides, box, estr, CU_TENSOR_MAP_SWIZZLE_NONE))
    return NVFP4_ERR_CUDA;

  const int sms = nvfp4::sm_count();
  const int64_t slots = (int64_t)sms * occ;  // resident CTAs
  // Split K (ks warps per tile) only while there are fewer tile groups than
  // resident CTAs (the split-K hand-off costs more than the load imbalance it
  // removes beyond that), keeping at least 4 chunks per warp; split factors
  // are 1, 4, 8, 16 (at most 4 tile groups per CTA share its named barriers).
  int ks = 1;
  while (ks < warps && nvfp4::cdiv(p.ntiles, warps / ks) < slots &&
         nitems / (2 * ks) >= 2)
    ks = ks == 1 ? 4 : 2 * ks;
  if (ks > 1 && warps / ks > 4) ks = warps / 4;
  p.ks = ks;
  const int64_t ngroups = nvfp4::cdiv(p.ntiles, warps / ks);
  int64_t grid = ngroups < slots ? ngroups : slots;
  if (grid > W4A16_GEMV_MAX_CTAS) grid = W4A16_GEMV_MAX_CTAS;  // bound of the log-prob workspace
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  // With room in the workspace and more than one batch row, one small grid
  // normalises the activations once (one CTA per batch row) and every GEMV
  // CTA copies its result.  At m = 1 the per-CTA prologue is short and mostly
  // hidden behind the first weight loads; the extra launch costs more.
  const bool prep = m >= 2 && workspace != nullptr &&
                    workspace_bytes >= W4A16_GEMV_WS_BYTES(m, w.k) && nvfp4::aligned16(workspace);
  if (prep) {
    char* ws = reinterpret_cast<char*>(workspace);
    unsigned int* rowmax = reinterpret_cast<unsigned int*>(ws + W4A16_GEMV_PREP_OFFSET);
    uint2* frag = reinterpret_cast<uint2*>(ws + W4A16_GEMV_PREP_OFFSET + 256);
    p.frag_src = frag;
    p.rowmax_src = rowmax;
    cudaLaunchConfig_t pc = {};
    pc.gridDim = dim3((unsigned)m);
    pc.blockDim = dim3(512);
    pc.dynamicSmemBytes = 0;
    pc.stream = stream;
    pc.attrs = attr;
    pc.numAttrs = 1;
    if (cudaLaunchKernelEx(&pc, prep_for(m), p, frag, rowmax) != cudaSuccess) return NVFP4_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(warps * 32);
  cfg.dynamicSmemBytes = lay.bytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, fn, tmap, p) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
  return NVFP4_OK;
}
