// gemv.cu -- batched NVFP4 W4A16 GEMV (up to 16 rows per launch) with RMSNorm +
// concat fused on the input and greedy argmax (+ grammar mask, top-1
// log-probability) fused on the output, for sm_103a.  The FP8 weight variant
// shares the kernel.
//
// What it computes (the NVFP4 GEMV of the draft head, "metrale_model_layers/
// layers/mtp_head.rs" MtpHead::gemv, batched; norm/concat/argmax of the draft
// step in the same module and in "spark_model/layers/deepseek_v4_mtp.rs"):
//     a[m, :]   = concat_j( bf16(x_j[m, :] * rsqrt(mean(x_j^2) + eps_j) * gamma_j) )
//     y[m, n]   = g * sum_i a[m, i] * e4m3(s[n, i/16]) * e2m1(c[n, i])      (FP32)
//     argmax[m] = lowest n with y[m, n] maximal (NaN never wins)
//
// Design.  The kernel streams the weights from HBM once (NVFP4: 0.5625 byte
// per weight incl. scales; FP8: 1 byte + 4 per row); with NVFP4 weights the
// decode and the legacy MMAs keep the SM's issue slots about half busy, so the
// main loop runs somewhat below the copy rate.
//   * Work split: one CTA per SM (grid <= SM count), each owning a contiguous,
//     equal range of 16-row tiles, so every SM streams the same number of weight
//     bytes.  Inside the CTA each warp takes a contiguous run of the CTA's
//     work units: whole tiles, or, when the CTA has at most half as many tiles
//     as warps, K parts of tiles (split K, ks parts per tile).  A split tile's
//     part sums are added in K-part order once every warp has streamed its
//     units, so every tile's sum is formed the same way (equal weight rows
//     give bit-equal logits).
//   * Weight stream: every warp owns a 2-stage shared-memory ring; one lane
//     issues the TMA copy (cp.async.bulk.tensor) of a stage -- 256 K elements
//     of 16 rows: one box of 16 rows x 128 bytes (NVFP4) or 16 x 256 bytes
//     (FP8) -- with an mbarrier completion.  Rows past n and bytes past k
//     arrive as zeros (TMA bounds fill).  NVFP4 block scales arrive in the
//     same stage by a second TMA box (16 rows x 16 bytes) when k is a multiple
//     of 256, else are read from global memory as the stage is computed.  (Two
//     64-byte-wide boxes per stage avoid a 2-way bank conflict on the code
//     loads but measured slower: the TMA request count matters more.)
//   * Across calls: the weights, their scales and the norm weights are
//     load-time constants, so with two or more rows a CTA issues its first
//     ring stages (and reads the norm weights) before the grid-dependency
//     wait; at M = 1 it issues them right after its activation loads, so that
//     those are not queued behind the ring fills.  Activations are read
//     only after the wait: normalised by every CTA for one row, or, with a
//     large enough workspace and two or more rows, once per call by a small
//     grid (one CTA per row) whose result every GEMV CTA copies.
//   * Products on the tensor cores (warp-level mma.sync m16n8k16, FP16 in,
//     FP32 accumulate), A = a 16-row weight tile, exact in FP16:
//       - M = 1, NVFP4 ("block columns"): MMA column j holds the activations of
//         the chunk's K block j (zeros elsewhere), so column j sums block j's
//         unscaled products e2m1(c) * a; the E4M3 block scale then multiplies
//         that FP32 partial once (one FMA per block instead of one packed
//         multiply per weight pair).
//       - otherwise: each E2M1 pair times its block scale (FP16, exact: at most
//         6 significant bits) or an FP8 pair as is; B = the activation rows (8
//         MMA columns per column group, two groups for 9..16 rows sharing each
//         dequantised A fragment); the FP8 row scale multiplies the finished sum.
//     Activations are FP16 after an exact per-row power-of-two scale that the
//     epilogue removes.
//   * Argmax: a 64-bit key (order-preserving float bits, inverted index) per
//     row, max-reduced per lane, warp, CTA, then one atomic max per CTA and row;
//     the last CTA converts the keys and returns the workspace to zero.
//     Optional grammar mask and top-1 log-probability (an online log-sum-exp,
//     per-CTA partials combined in a fixed order).
//   * Every mbarrier wait is bounded; one that runs out records
//     NVFP4_ERR_TIMEOUT, the lane waits no more and issues no further copies,
//     and before the CTA exits its copies still in flight are waited for
//     (bounded again).
#include <cuda.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "common.cuh"

namespace {

constexpr int kChunk = 128;          // K elements per chunk (8 MMA k-steps)
constexpr int kItem = 2;             // chunks per ring stage
constexpr int kItemK = kChunk * kItem;
constexpr int kStageNv = 16 * 128 + 256;  // NVFP4 stage: 16 rows x 256 codes, then their 16 x 16 scales
constexpr int kScaleOff = 16 * 128;        // the scales' offset in an NVFP4 stage
constexpr int kStageF8 = 16 * 256;   // FP8 stage: 16 rows x 256 codes
__host__ __device__ constexpr int stage_bytes(bool fp8) { return fp8 ? kStageF8 : kStageNv; }
// ring stages per warp (NVFP4: 4 KB in flight per warp; FP8: 8 KB); deeper
// rings measured slower (fewer warps fit)
__host__ __device__ constexpr int ring_depth(bool) { return 2; }
constexpr unsigned long long kWaitLimitNs = nvfp4::kWaitLimit;
constexpr int kMaxRows = 16;         // batch rows of one launch
// Block-column activations (M = 1), per 128-element chunk: block j (16
// values, 8 FP16 pairs) at byte 64 j as 8-byte (b0, b1) MMA operand pairs --
// (pair q, 0) for even j, (0, pair q) for odd j, the register pair lane
// (g = j, t = j / 2) feeds MMA q -- then a zero block for every other lane at
// byte kBcZero (16 bytes off the banks of each quarter-warp's active lanes).
// One 16-byte load gives the operands of two MMAs; every lane walks the
// chunks with one stride.
constexpr int kBcChunkBytes = 640;
constexpr int kBcZero = 528;
constexpr int kMaxKs = 16;           // warps sharing one tile

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
  int64_t ntiles;  // ceil(n / 16)
  int nitems;      // ceil(k / 256): ring stages per tile
  int tpc;         // tiles per CTA (the last CTA may have fewer)
  int ks;          // warps sharing one tile (split K), 1..16, <= nitems
  int kbeg[kMaxKs + 1];  // first stage of K part kp: kp * nitems / ks (no division on the device)
  const uint2* frag_src;          // fragments prepared by act_prep_kernel, or null
  const unsigned int* rowmax_src; // their per-row scale carriers [16]
  int scale_tma;      // NVFP4 block scales arrive by TMA with the codes (k % 256 == 0)
  // shared-memory carve-up (bytes from the 1 KB-aligned base)
  uint32_t off_frag, off_zero, off_part, off_small, off_kred, off_bar;
};

// Block-column path: lanes (g, t = 0) emit rows g and g + 8 of every tile; their
// running argmax key and log-sum-exp live in shared memory (off_zero area),
// [warp][g], which keeps them out of the main loop's registers.
struct BcRun {
  unsigned long long key;
  float lm, ls;
};

// (local tile, K part) of a work unit; next() steps to the following unit.
struct UnitCursor {
  int tl, kp;
  __device__ __forceinline__ void next(int ks) {
    if (++kp == ks) {
      kp = 0;
      ++tl;
    }
  }
};

// ------------------------------------------------------------ PTX helpers
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
// The same, letting the hardware suspend the warp for up to `hint_ns` while
// the phase is incomplete (a waiting warp then issues nothing, leaving the
// issue slots to the warps that have data).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
// Bounded wait; false (and NVFP4_ERR_TIMEOUT recorded) if it ran out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int32_t* dev_status) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait_sleep(bar, parity, 1000000u)) {
    if (globaltimer() - t0 > kWaitLimitNs) {
      nvfp4::report(dev_status, NVFP4_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
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
// The same with a zero accumulator input (a fresh sum).
__device__ __forceinline__ void mma_f16_16816_z(float (&c)[4], uint32_t a0, uint32_t a1,
                                                uint32_t a2, uint32_t a3, uint32_t b0,
                                                uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

// Two E4M3 block scales (low byte first) -> F16 (exact: E4M3 values are F16
// normals), each replicated into both halves of an f16x2.
__device__ __forceinline__ void decode_scales(uint32_t s2, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 a, b;\n .reg .b32 v;\n cvt.rn.f16x2.e4m3x2 v, %2;\n mov.b32 {a, b}, v;\n"
      " mov.b32 %0, {a, a};\n mov.b32 %1, {b, b};\n}"
      : "=r"(lo), "=r"(hi)
      : "h"((uint16_t)s2));
}
// Two E4M3 block scales (low byte first) -> two FP32 values (exact).
__device__ __forceinline__ void decode_scales_f32(uint32_t s2, float& lo, float& hi) {
  uint32_t v;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(v) : "h"((uint16_t)s2));
  const __half2 h = *reinterpret_cast<const __half2*>(&v);
  const float2 f = __half22float2(h);
  lo = f.x;
  hi = f.y;
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

// One 128-element chunk, scaled weights (every M except the block-column path).
// Lane (g, t) holds rows g, g+8 and K elements 32t .. 32t+31 of the chunk
// (qg, qh); word w of its 16-byte load covers 32t + 8w .. +7, and MMA 2w+u
// takes the pairs of elements 4u .. 4u+3 of that word, so the MMA's column
// c = 2t + e + 8h is element 32t + 8w + 4u + 2h + e: a B fragment is 4
// consecutive activations, at bfrag[j * BSTRIDE] for MMA j (lanes whose batch
// column is >= M read a duplicate of a valid column: MMA columns are
// independent and those outputs are discarded).
// The MMAs alternate between two accumulator sets (acc[.][0..3] and
// acc[.][4..7], added at the end of a unit) so consecutive MMAs do not wait on
// each other.
template <int BSTRIDE, int NCG, int GSTRIDE>
__device__ __forceinline__ void chunk_mma(float (&acc)[NCG][8], const uint4& qg, const uint4& qh,
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
      mma_f16_16816(*reinterpret_cast<float(*)[4]>(&acc[cg][0]), a0, a1, a2, a3, b0.x, b0.y);
    }
    const uint32_t c0 = f16x2_mul(g2, sG), c1 = f16x2_mul(h2, sH), c2 = f16x2_mul(g3, sG),
                   c3 = f16x2_mul(h3, sH);
#pragma unroll
    for (int cg = 0; cg < NCG; ++cg) {
      const uint2 b1 = bfrag[(2 * w + 1) * BSTRIDE + cg * GSTRIDE];
      mma_f16_16816(*reinterpret_cast<float(*)[4]>(&acc[cg][4]), c0, c1, c2, c3, b1.x, b1.y);
    }
  }
}

// One E2M1 code pair (byte `by` of word q) -> f16x2 (exact).
__device__ __forceinline__ uint32_t e2m1_byte_to_f16(uint32_t q, int by) {
  uint32_t h;
  if (by == 0)
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b0;\n}" : "=r"(h) : "r"(q));
  else if (by == 1)
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b1;\n}" : "=r"(h) : "r"(q));
  else if (by == 2)
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b2;\n}" : "=r"(h) : "r"(q));
  else
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b3;\n}" : "=r"(h) : "r"(q));
  return h;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");  // not hoisted above the barrier that publishes the fragments
  return v;
}

// One 128-element chunk at M = 1 with block columns.  Lane (g, t) holds rows
// g, g+8 and the chunk's K blocks 2t (words x, y of qg / qh: element pairs
// 0..3, 4..7) and 2t+1 (words z, w).  MMA q takes element pair q of every
// block: its K index 2t' + e + 8h is element 2q + e of block 2t' + h, so A is
// a0 = (row g, block 2t, pair q), a1 = (row g+8, block 2t), a2 = (row g,
// block 2t+1), a3 = (row g+8, block 2t+1), and B column c holds block c's
// pair q: b0 of lane (g, t) is non-zero only when g == 2t, b1 only when
// g == 2t+1; the lane's (b0, b1) pairs of MMAs q, q+1 are one 16-byte load at
// bq + 8 q (see kBcChunkBytes).  The MMAs leave in d the unscaled block sums
// of rows g, g+8 and blocks 2t, 2t+1; sg / sh hold their scale pairs.
__device__ __forceinline__ void chunk_bc(float (&acc)[8], const uint4& qg, const uint4& qh, uint32_t sg,
                                         uint32_t sh, uint32_t bq) {
  float d[2][4];  // even / odd MMAs: two independent chains
#pragma unroll
  for (int hw = 0; hw < 2; ++hw) {
    const uint32_t wg0 = hw ? qg.y : qg.x, wh0 = hw ? qh.y : qh.x;  // block 2t
    const uint32_t wg1 = hw ? qg.w : qg.z, wh1 = hw ? qh.w : qh.z;  // block 2t+1
#pragma unroll
    for (int hq = 0; hq < 2; ++hq) {
      const uint4 b = lds128(bq + 32 * hw + 16 * hq);  // MMAs 4hw + 2hq, +1
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int by = 2 * hq + e;
        const uint32_t x0 = e2m1_byte_to_f16(wg0, by), x1 = e2m1_byte_to_f16(wh0, by);
        const uint32_t x2 = e2m1_byte_to_f16(wg1, by), x3 = e2m1_byte_to_f16(wh1, by);
        const uint32_t bb0 = e ? b.z : b.x, bb1 = e ? b.w : b.y;
        if (hw == 0 && hq == 0)
          mma_f16_16816_z(d[e], x0, x1, x2, x3, bb0, bb1);
        else
          mma_f16_16816(d[e], x0, x1, x2, x3, bb0, bb1);
      }
    }
  }
  float sg0, sg1, sh0, sh1;
  decode_scales_f32(sg, sg0, sg1);
  decode_scales_f32(sh, sh0, sh1);
  acc[0] = fmaf(d[0][0] + d[1][0], sg0, acc[0]);  // (row g,   block 2t)
  acc[1] = fmaf(d[0][1] + d[1][1], sg1, acc[1]);  // (row g,   block 2t+1)
  acc[2] = fmaf(d[0][2] + d[1][2], sh0, acc[2]);  // (row g+8, block 2t)
  acc[3] = fmaf(d[0][3] + d[1][3], sh1, acc[3]);  // (row g+8, block 2t+1)
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
__device__ __forceinline__ void chunk_mma_fp8(float (&acc)[NCG][8], const uint4& qg0, const uint4& qg1,
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
      mma_f16_16816(*reinterpret_cast<float(*)[4]>(&acc[cg][4 * (q & 1)]), g0, h0, g1, h1, b.x, b.y);
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
// Row r of segment s: row r of x, or, for a gathered segment, table row
// ridx[r] (out-of-range indices read row 0 and are reported).  Read only after
// the grid-dependency wait (the index may come from the previous call).
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
constexpr int kMaxJobs = 2 * kMaxRows;  // (row, segment) pairs
__host__ __device__ constexpr int small_floats(int warps) { return kSmallParts + 2 * kMaxJobs * warps + 2 * 2 * warps; }

// Largest |gamma_s| per segment (the norm weights are load-time constants, so
// this runs before the grid-dependency wait).  Partials per (segment, warp) in
// small[kSmallParts + 2 kMaxJobs warps ...], combined by gamma_max_finish.
template <int WARPS>
__device__ __forceinline__ void gamma_max_partials(const GemvParams& p, float* small) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned int* part = reinterpret_cast<unsigned int*>(small + kSmallParts + 2 * kMaxJobs * WARPS);
  for (int s = 0; s < p.nseg; ++s) {
    uint32_t mx = 0u;
    if (p.gamma[s] != nullptr) {
      for (int i = threadIdx.x * 8; i < (int)p.kseg[s]; i += WARPS * 256) {
        if (!NVFP4_GUARD(i + 8 <= p.kseg[s], 7, p.dev_status)) continue;
        const uint4 v = *reinterpret_cast<const uint4*>(p.gamma[s] + i);
        mx = __vmaxu2(mx, v.x & 0x7FFF7FFFu);
        mx = __vmaxu2(mx, v.y & 0x7FFF7FFFu);
        mx = __vmaxu2(mx, v.z & 0x7FFF7FFFu);
        mx = __vmaxu2(mx, v.w & 0x7FFF7FFFu);
      }
    }
    mx = __reduce_max_sync(0xFFFFFFFFu, max(mx & 0xFFFFu, mx >> 16));
    if (lane == 0) part[s * WARPS + warp] = mx;
  }
}

// Normalise (optionally) and lay out the activations of rows 0 .. MM-1.
// Statistics: jobs (row, segment) split over the warps (fixed combination
// order, so the result does not depend on timing); then every 8-element group
// is read again (an L1 hit), normalised, rounded to BF16, scaled by the row's
// power of two and stored as FP16:
//   in the MMA fragment order: MMA index q = 8 * chunk + j; batch row m,
//        lane quad t: uint2 at bfrag[q * BSTRIDE + (m / 8) * GSTRIDE + 4 * (m % 8) + t],
//        GSTRIDE = 4 * min(M, 8), BSTRIDE = GSTRIDE times the column groups.
//        For the 8 activations at kk = 128 c + 32 t + 8 w (+0..7): MMA 8c+2w
//        gets {a0,a4},{a1,a5}; MMA 8c+2w+1 gets {a2,a6},{a3,a7}.  Zeros past k.
// Rows r0 .. r0 + nrows - 1 of the batch; `frag` may be shared or global
// memory (generic addresses); rowmax_out (nullable) receives the rows' scale
// carriers too.
template <int M, int WARPS, bool BC>
__device__ __forceinline__ void build_fragments(const GemvParams& p, unsigned char* frag, float* small,
                                                int r0, int nrows, int nchunks, unsigned int* rowmax_out) {
  constexpr int MC = M > 8 ? 8 : M, NCG = (M + 7) / 8, GSTRIDE = 4 * MC, BSTRIDE = GSTRIDE * NCG;
  constexpr int kThreads = WARPS * 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float* rms = small;
  unsigned int* rowmax = reinterpret_cast<unsigned int*>(small + kSmallRowmax);
  float* maxg = small + kSmallMaxg;
  float* maxx = small + kSmallMaxx;
  float* part_ss = small + kSmallParts;                                          // [job][warp]
  unsigned int* part_mx = reinterpret_cast<unsigned int*>(part_ss + kMaxJobs * WARPS);
  const unsigned int* part_g = reinterpret_cast<const unsigned int*>(small + kSmallParts + 2 * kMaxJobs * WARPS);
  // 1. statistics: sum of squares (normalised segments) and the largest |x|
  //    (BF16 magnitude bits order like the values) per (row, segment)
  const int J = nrows * p.nseg;
  const int wpj = J >= WARPS ? 1 : WARPS / J;  // warps per job
  const int jpp = WARPS / wpj;                  // jobs per pass
  for (int j0 = 0; j0 < J; j0 += jpp) {
    const int job = j0 + warp / wpj, wj = warp % wpj;
    if (job < J) {
      const int s = job % p.nseg;
      const __nv_bfloat16* src = seg_row(p, s, r0 + job / p.nseg);
      const bool want_ss = p.gamma[s] != nullptr;
      float ss = 0.0f;
      uint32_t mx = 0u;
#pragma unroll 4
      for (int i = (wj * 32 + lane) * 8; i < (int)p.kseg[s]; i += wpj * 256) {
        if (!NVFP4_GUARD(i + 8 <= p.kseg[s], 1, p.dev_status)) continue;
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
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
      mx = __reduce_max_sync(0xFFFFFFFFu, max(mx & 0xFFFFu, mx >> 16));
      if (lane == 0) {
        part_ss[job * WARPS + wj] = ss;
        part_mx[job * WARPS + wj] = mx;
      }
    }
  }
  __syncthreads();
  if (tid < J) {
    const int s = tid % p.nseg;
    float ss = 0.0f;
    unsigned int mx = 0u;
    for (int w = 0; w < wpj; ++w) {
      ss += part_ss[tid * WARPS + w];
      mx = max(mx, part_mx[tid * WARPS + w]);
    }
    rms[tid] = p.gamma[s] == nullptr ? 1.0f : 1.0f / sqrtf(ss / (float)p.kseg[s] + p.eps[s]);
    maxx[tid] = __uint_as_float(mx << 16);
  } else if (tid >= 32 && tid < 32 + p.nseg) {
    const int s = tid - 32;
    unsigned int mx = 0u;
    for (int w = 0; w < WARPS; ++w) mx = max(mx, part_g[s * WARPS + w]);
    maxg[s] = __uint_as_float(mx << 16);
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
  // 2. normalised, scaled FP16 activations
  const int gpr = nchunks * (kChunk / 8);  // 8-element groups per row
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
      {
        uint2* bfrag = reinterpret_cast<uint2*>(frag);
        const int c = kk / kChunk, t = (kk % kChunk) / 32, w = (kk % 32) / 8;
        const int L = (r / 8) * GSTRIDE + 4 * (r % 8) + t;
        if (!NVFP4_GUARD((8 * c + 2 * w + 1) * BSTRIDE + L < nchunks * 8 * BSTRIDE && L < BSTRIDE, 3,
                         p.dev_status))
          continue;
        bfrag[(8 * c + 2 * w) * BSTRIDE + L] = make_uint2(a[0], a[1]);
        bfrag[(8 * c + 2 * w + 1) * BSTRIDE + L] = make_uint2(a[2], a[3]);
      }
    }
  }
}

// M = 1 with block columns: normalise the row into the block-column operand
// layout (see kBcChunkBytes).  Each thread reads its 8-element groups of x and
// gamma once, in one round trip (held in registers across the statistics);
// the statistics are reduced per warp, then by warp 0 over the warps in a
// fixed order.
// Registers of the M = 1 prologue: this thread's 8-element groups of x and
// gamma (at most kBcG of them).
template <int WARPS>
struct BcRegs {
  static constexpr int kG = (W4A16_GEMV_MAX_K / 8 + WARPS * 32 - 1) / (WARPS * 32);
  uint4 xv[kG], gv[kG];
};

// First half of the M = 1 prologue: issue this thread's loads of x and gamma
// (one round trip; nothing here waits for them).
template <int WARPS>
__device__ __forceinline__ void build_bc_load(const GemvParams& p, BcRegs<WARPS>& r) {
  constexpr int kThreads = WARPS * 32, kG = BcRegs<WARPS>::kG;
  const int tid = threadIdx.x;
  const __nv_bfloat16* xr0 = seg_row(p, 0, 0);
  const __nv_bfloat16* xr1 = p.nseg == 2 ? seg_row(p, 1, 0) : xr0;
#pragma unroll
  for (int i = 0; i < kG; ++i) {
    const int kk = 8 * (tid + i * kThreads);
    r.xv[i] = make_uint4(0u, 0u, 0u, 0u);
    r.gv[i] = make_uint4(0u, 0u, 0u, 0u);
    if (kk < p.k) {
      const int s = (p.nseg == 2 && kk >= p.kseg[0]) ? 1 : 0;
      const int ko = kk - (s ? (int)p.kseg[0] : 0);
      if (!NVFP4_GUARD(ko + 8 <= p.kseg[s], 2, p.dev_status)) continue;
      r.xv[i] = *reinterpret_cast<const uint4*>((s ? xr1 : xr0) + ko);
      if (p.gamma[s] != nullptr) r.gv[i] = *reinterpret_cast<const uint4*>(p.gamma[s] + ko);
    }
  }
}

// Second half: statistics, normalisation and the block-column layout.
template <int WARPS>
__device__ __forceinline__ void build_bc(const GemvParams& p, unsigned char* frag, float* small, int nchunks,
                                         const BcRegs<WARPS>& r) {
  constexpr int kThreads = WARPS * 32, kG = BcRegs<WARPS>::kG;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float* rms = small;
  unsigned int* rowmax = reinterpret_cast<unsigned int*>(small + kSmallRowmax);
  float* part = small + kSmallParts;  // [warp][6]: sum of squares, max |x|, max |gamma| per segment
  const uint4* xv = r.xv;
  const uint4* gv = r.gv;
  float ss[2] = {0.f, 0.f};
  uint32_t mx[2] = {0u, 0u}, mg[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < kG; ++i) {
    const int kk = 8 * (tid + i * kThreads);
    if (kk >= p.k) continue;
    const int s = (p.nseg == 2 && kk >= p.kseg[0]) ? 1 : 0;
    const uint32_t u[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
    const uint32_t gw[4] = {gv[i].x, gv[i].y, gv[i].z, gv[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      mx[s] = __vmaxu2(mx[s], u[j] & 0x7FFF7FFFu);
      mg[s] = __vmaxu2(mg[s], gw[j] & 0x7FFF7FFFu);
      const float a = __uint_as_float(u[j] << 16), b = __uint_as_float(u[j] & 0xFFFF0000u);
      ss[s] = fmaf(a, a, ss[s]);
      ss[s] = fmaf(b, b, ss[s]);
    }
  }
#pragma unroll
  for (int s = 0; s < 2; ++s) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss[s] += __shfl_xor_sync(0xFFFFFFFFu, ss[s], o);
    mx[s] = __reduce_max_sync(0xFFFFFFFFu, max(mx[s] & 0xFFFFu, mx[s] >> 16));
    mg[s] = __reduce_max_sync(0xFFFFFFFFu, max(mg[s] & 0xFFFFu, mg[s] >> 16));
  }
  if (lane == 0) {
    part[6 * warp + 0] = ss[0];
    part[6 * warp + 1] = ss[1];
    part[6 * warp + 2] = __uint_as_float(mx[0]);
    part[6 * warp + 3] = __uint_as_float(mx[1]);
    part[6 * warp + 4] = __uint_as_float(mg[0]);
    part[6 * warp + 5] = __uint_as_float(mg[1]);
  }
  __syncthreads();
  if (warp == 0) {
    float t0 = 0.f, t1 = 0.f;
    uint32_t m0 = 0u, m1 = 0u, g0 = 0u, g1 = 0u;
    if (lane < WARPS) {
      t0 = part[6 * lane + 0];
      t1 = part[6 * lane + 1];
      m0 = __float_as_uint(part[6 * lane + 2]);
      m1 = __float_as_uint(part[6 * lane + 3]);
      g0 = __float_as_uint(part[6 * lane + 4]);
      g1 = __float_as_uint(part[6 * lane + 5]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      t0 += __shfl_xor_sync(0xFFFFFFFFu, t0, o);
      t1 += __shfl_xor_sync(0xFFFFFFFFu, t1, o);
    }
    m0 = __reduce_max_sync(0xFFFFFFFFu, m0);
    m1 = __reduce_max_sync(0xFFFFFFFFu, m1);
    g0 = __reduce_max_sync(0xFFFFFFFFu, g0);
    g1 = __reduce_max_sync(0xFFFFFFFFu, g1);
    if (lane == 0) {
      float bound = 0.0f;
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        if (s >= p.nseg) break;
        const float tt = s ? t1 : t0;
        const uint32_t mm = s ? m1 : m0, gg = s ? g1 : g0;
        const float r = p.gamma[s] == nullptr ? 1.0f : 1.0f / sqrtf(tt / (float)p.kseg[s] + p.eps[s]);
        rms[s] = r;
        const float mxs = __uint_as_float(mm << 16), mgs = __uint_as_float(gg << 16);
        bound = fmaxf(bound, p.gamma[s] == nullptr ? mxs : mxs * r * mgs * (1.0f + 0.0078125f));
      }
      rowmax[0] = __float_as_uint(bound) >> 16;  // carries the bound's exponent
    }
  }
  __syncthreads();
  const float sc = row_scale_pow2(rowmax[0], false);
#pragma unroll
  for (int i = 0; i < kG; ++i) {
    const int q = tid + i * kThreads, kk = 8 * q;
    if (kk >= nchunks * kChunk) continue;
    uint32_t a[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
    if (kk < p.k) {
      const int s = (p.nseg == 2 && kk >= p.kseg[0]) ? 1 : 0;
      if (p.gamma[s] != nullptr) {
        const uint32_t gw[4] = {gv[i].x, gv[i].y, gv[i].z, gv[i].w};
        const float rr = rms[s];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float lo = __uint_as_float(a[j] << 16) * rr * __uint_as_float(gw[j] << 16);
          const float hi = __uint_as_float(a[j] & 0xFFFF0000u) * rr * __uint_as_float(gw[j] & 0xFFFF0000u);
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
    // element pairs p0 .. p0+3 of block jb of chunk c: slots 64 jb + 8 p
    const int c = kk / kChunk, jb = (kk % kChunk) / 16, p0 = (kk % 16) / 2;
    unsigned char* slot = frag + (size_t)c * kBcChunkBytes + 64 * jb + 8 * p0;
    if (jb & 1) {
      *reinterpret_cast<uint4*>(slot) = make_uint4(0u, a[0], 0u, a[1]);
      *reinterpret_cast<uint4*>(slot + 16) = make_uint4(0u, a[2], 0u, a[3]);
    } else {
      *reinterpret_cast<uint4*>(slot) = make_uint4(a[0], 0u, a[1], 0u);
      *reinterpret_cast<uint4*>(slot + 16) = make_uint4(a[2], 0u, a[3], 0u);
    }
  }
  // each chunk's zero block (64 bytes)
  for (int i = tid; i < nchunks * 4; i += kThreads)
    *reinterpret_cast<uint4*>(frag + (size_t)(i / 4) * kBcChunkBytes + kBcZero + 16 * (i % 4)) =
        make_uint4(0u, 0u, 0u, 0u);
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
  gamma_max_partials<16>(p, small);
  build_fragments<M, 16, false>(p, reinterpret_cast<unsigned char*>(frag), small, (int)blockIdx.x, 1,
                                p.nitems * kItem, rowmax);
}

// ------------------------------------------------------------------ kernel
// Template: M batch rows (1..8 exact; 16 = any 9..16), WARPS per CTA, weight
// format, and the block-column path (M = 1, NVFP4).
template <int M, int WARPS, bool FP8, bool BC>
__global__ void __launch_bounds__(WARPS * 32, 1)
gemv_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_s,
            const __grid_constant__ GemvParams p) {
  constexpr int MC = M > 8 ? 8 : M, NCG = (M + 7) / 8, GSTRIDE = 4 * MC, BSTRIDE = GSTRIDE * NCG;
  constexpr int S = ring_depth(FP8);
  constexpr int kStage = stage_bytes(FP8);
  constexpr int NACC = BC ? 1 : NCG;  // accumulator sets (4 floats each)
  constexpr int NE = M == 1 ? 1 : 2;  // batch columns 2t + e a lane emits (M = 1: column 0 only)
  static_assert(!BC || (M == 1 && !FP8), "block columns are the M = 1 NVFP4 path");
  const int MM = M > 8 ? p.m : M;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw));
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* const smem = smem_raw + (base - raw);
  unsigned char* frag = smem + p.off_frag;
  float* small = reinterpret_cast<float*>(smem + p.off_small);
  float* part = reinterpret_cast<float*>(smem + p.off_part);
  unsigned long long* kred = reinterpret_cast<unsigned long long*>(smem + p.off_kred);

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;

  // This CTA's tiles [tile0, tile0 + nt), as units u = (local tile u / ks, K
  // part u % ks); warp w takes the contiguous units [ceil(w U / WARPS),
  // ceil((w + 1) U / WARPS)) (warp 0 always starts at unit 0; with fewer units
  // than warps the last warps idle).  Tile indices fit 27 bits (checked on the
  // host).
  const int tile0 = (int)blockIdx.x * p.tpc;
  const int nt = min(p.tpc, (int)p.ntiles - tile0);
  const int ks = p.ks;
  const int64_t U = nt > 0 ? (int64_t)nt * ks : 0;
  const int ubeg = (int)(((int64_t)warp * U + WARPS - 1) / WARPS);
  const int nunits = (int)(((int64_t)(warp + 1) * U + WARPS - 1) / WARPS) - ubeg;
  auto kp_begin = [&](int kp) { return p.kbeg[kp]; };
  const UnitCursor first{ubeg / ks, ubeg % ks};
  int total = 0;  // ring stages this warp streams
  {
    UnitCursor c = first;
    for (int j = 0; j < nunits; ++j, c.next(ks)) total += kp_begin(c.kp + 1) - kp_begin(c.kp);
  }
  const uint32_t ring = base;  // the ring sits at the start of the carve-up (1 KB aligned)
  const uint32_t wring = ring + (uint32_t)warp * (S * kStage);
  const uint32_t bars = base + p.off_bar + (uint32_t)warp * (S * 8);
  // chunks c with 128c + 32t < k hold this lane's data (scales past k read 0)
  const int cmax = (int)((p.k - 32 * t + kChunk - 1) / kChunk);
  // The stage whose wait ran out in this lane (kAlive while none has): from
  // then on the lane waits no more and lane 0 issues no further copies.
  constexpr int kAlive = 0x7FFFFFFF;
  int failed_at = kAlive;

  const bool prepped = !BC && p.frag_src != nullptr;
  const uint32_t fbar = base + p.off_bar + (uint32_t)WARPS * (S * 8);  // fragment copy
  if (lane == 0) {
    for (int i = 0; i < S; ++i) mbar_init(bars + 8 * i, 1);
    if (threadIdx.x == 0) mbar_init(fbar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();

  // ---- load cursor over (unit, item); scale rows change once per unit
  int lj = 0, li = 0, l_ib = 0, l_len = 0, l_tile = 0;
  UnitCursor lc = first;
  auto set_unit = [&]() {
    l_ib = kp_begin(lc.kp);
    l_len = kp_begin(lc.kp + 1) - l_ib;
    l_tile = tile0 + lc.tl;
  };
  if (nunits > 0) set_unit();
  // NVFP4 block scales: with scale_tma a 16 x 16-byte box of the stage's rows
  // lands behind its codes (row r's 16 bytes: the 8 blocks of each of the two
  // chunks); otherwise a lane reads its scale pairs from global memory when it
  // computes the stage (k not a multiple of 256: small shapes only).
  const uint32_t stage_tx = FP8 ? (uint32_t)kStage : (p.scale_tma ? (uint32_t)kStage : (uint32_t)kScaleOff);
  bool skip_next = nvfp4::kWithhold && blockIdx.x == 0 && warp == 0;  // test build: one copy never issued
  auto issue = [&](int i) {
    const int item = l_ib + li;
    const bool send = !skip_next;
    skip_next = false;
    if (lane == 0 && failed_at == kAlive && send) {
      mbar_arrive_expect_tx(bars + 8 * i, stage_tx);
      if constexpr (FP8) {
        tma_load_2d(wring + i * kStage, &tmap_w, item * 256, l_tile * 16, bars + 8 * i);
      } else {
        tma_load_2d(wring + i * kStage, &tmap_w, item * 128, l_tile * 16, bars + 8 * i);
        if (p.scale_tma) tma_load_2d(wring + i * kStage + kScaleOff, &tmap_s, item * 16, l_tile * 16, bars + 8 * i);
      }
    }
    if (++li == l_len) {
      li = 0;
      lc.next(ks);
      if (++lj < nunits) set_unit();
    }
  };
  __syncthreads();  // barriers initialised

  // ---- before the grid-dependency wait: the weights, their scales and the
  // norm weights are load-time constants.  Start this warp's weight stream and
  // take the norm weights' maxima.  M = 1 issues its ring stages right after
  // the activation loads instead (so those loads are not queued behind them).
#pragma unroll
  for (int i = 0; i < S; ++i)
    if (i < total && !BC) issue(i);
  if (!prepped && !BC) gamma_max_partials<WARPS>(p, small);
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- activations (may be the previous call's output): read now
  const int nchunks_frag = p.nitems * kItem;
  if (prepped) {
    // one bulk copy of the prepared fragments and row-scale carriers
    if (threadIdx.x == 0) {
      constexpr uint32_t kFragPerChunk = 8u * BSTRIDE * 8u;
      const uint32_t fbytes = (uint32_t)nchunks_frag * kFragPerChunk;
      mbar_arrive_expect_tx(fbar, fbytes + 4u * kMaxRows);
      for (uint32_t off = 0; off < fbytes; off += 32768u) {
        const uint32_t nb = fbytes - off < 32768u ? fbytes - off : 32768u;
        bulk_copy_g2s(base + p.off_frag + off, reinterpret_cast<const char*>(p.frag_src) + off, nb, fbar);
      }
      bulk_copy_g2s(base + p.off_small + kSmallRowmax * 4u, p.rowmax_src, 4u * kMaxRows, fbar);
    }
    if (!mbar_wait(fbar, 0u, p.dev_status)) failed_at = 0;
  } else if constexpr (BC) {
    BcRegs<WARPS> br;
    build_bc_load<WARPS>(p, br);
#pragma unroll
    for (int i = 0; i < S; ++i)
      if (i < total) issue(i);
    build_bc<WARPS>(p, frag, small, nchunks_frag, br);
  } else {
    build_fragments<M, WARPS, BC>(p, frag, small, 0, MM, nchunks_frag, nullptr);
  }
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const float gsc = FP8 ? 1.0f : __ldg(p.gscale);
  const unsigned int* rowmax = reinterpret_cast<const unsigned int*>(small + kSmallRowmax);
  // inverse activation scales of this lane's batch columns 8 cg + 2t + e
  float inv[NCG][NE];
#pragma unroll
  for (int cg = 0; cg < NCG; ++cg)
#pragma unroll
    for (int e = 0; e < NE; ++e) inv[cg][e] = row_scale_pow2(rowmax[min(8 * cg + 2 * t + e, MM - 1)], true);
  if constexpr (BC) inv[0][0] *= gsc;
  unsigned long long best[NCG][NE];  // running argmax keys, columns 8cg + 2t + e
  float lm[NCG][NE], ls[NCG][NE];     // log-sum-exp (max, sum)
  float acc[NACC][8];  // two accumulator chains per set (BC uses [0..3])
#pragma unroll
  for (int cg = 0; cg < NCG; ++cg)
#pragma unroll
    for (int e = 0; e < NE; ++e) {
      best[cg][e] = 0ull;
      lm[cg][e] = -INFINITY;
      ls[cg][e] = 0.f;
    }
#pragma unroll
  for (int a = 0; a < NACC; ++a)
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[a][i] = 0.f;

  // Block-column B operand: lane (g, t) with g >> 1 == t reads block g of each
  // chunk (32 bytes of natural-order activations) into b0 (g even) or b1 (g
  // odd); every other read comes from a zero area.
  uint32_t pb = 0;
  if constexpr (BC) pb = base + p.off_frag + ((g >> 1) == t ? 64u * g : (uint32_t)kBcZero);
  const uint2* bbase = reinterpret_cast<const uint2*>(frag) + (lane % GSTRIDE);

  // Grammar mask words and FP8 row scales of the unit being computed: the 16
  // rows of a tile share one 32-bit mask word per batch column.
  uint32_t mword[NCG][NE];
  float rsc[2] = {0.f, 0.f};
  auto load_unit_extras = [&](int tile) {
    if constexpr (FP8) {
#pragma unroll
      for (int h = 0; h < 2; ++h) rsc[h] = __ldg(p.row_scale + min((int64_t)tile * 16 + g + 8 * h, p.n - 1));
    }
#pragma unroll
    for (int cg = 0; cg < NCG; ++cg)
#pragma unroll
      for (int e = 0; e < NE; ++e)
        mword[cg][e] = p.mask == nullptr
                           ? 0xFFFFFFFFu
                           : __ldg(reinterpret_cast<const uint32_t*>(p.mask) +
                                   min(8 * cg + 2 * t + e, MM - 1) * p.ld_mask + (tile >> 1));
  };

  BcRun* bc_run = reinterpret_cast<BcRun*>(smem + p.off_zero) + warp * 8 + g;
  if (BC && t == 0) *bc_run = BcRun{0ull, -INFINITY, 0.f};

  // One output value of row `row`, batch column mm: store, argmax key,
  // log-sum-exp.  `bit` is the row's bit in the tile's mask word.
  auto emit = [&](int cg, int e, int64_t row, int mm, float v, int bit) {
    if (p.y != nullptr && NVFP4_GUARD(mm < MM && row < p.n && row < p.ldy, 6, p.dev_status)) {
      if (p.y_dtype == NVFP4_DTYPE_F32)
        reinterpret_cast<float*>(p.y)[mm * p.ldy + row] = v;
      else
        reinterpret_cast<__nv_bfloat16*>(p.y)[mm * p.ldy + row] = __float2bfloat16_rn(v);
    }
    if (p.keys != nullptr && ((mword[cg][e] >> bit) & 1u)) {
      const unsigned long long key = argmax_key(v, (uint32_t)row);
      unsigned long long& bk = BC ? bc_run->key : best[cg][e];
      float& bm = BC ? bc_run->lm : lm[cg][e];
      float& bs = BC ? bc_run->ls : ls[cg][e];
      bk = key > bk ? key : bk;
      if (p.logprob != nullptr) {  // online log-sum-exp over the allowed logits
        if (v > bm) {
          bs = bs * __expf(bm - v) + 1.0f;
          bm = v;
        } else {
          bs += __expf(v - bm);
        }
      }
    }
  };

  // Emit a finished tile.  Block columns: rg, rh are the sums of rows g, g + 8
  // (lanes t == 0 emit them); otherwise acc[cg][0..3] hold the lane's outputs.
  auto emit_bc = [&](int64_t tile, float rg, float rh) {
    const int64_t rows[2] = {tile * 16 + g, tile * 16 + g + 8};
    const float vals[2] = {rg, rh};
#pragma unroll
    for (int h = 0; h < 2; ++h)
      if (rows[h] < p.n)  // inv is a power of two: (v inv) g == v (inv g) exactly
        emit(0, 0, rows[h], 0, vals[h] * inv[0][0], ((int)(tile & 1) << 4) + g + 8 * h);
  };
  auto emit_tile = [&](int64_t tile) {
    const int64_t rows[2] = {tile * 16 + g, tile * 16 + g + 8};
#pragma unroll
    for (int cg = 0; cg < NCG; ++cg)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (rows[h] >= p.n) continue;
#pragma unroll
        for (int e = 0; e < NE; ++e) {
          const int mm = 8 * cg + 2 * t + e;
          if (mm >= MM) continue;
          const float v = (acc[cg][2 * h + e] * inv[cg][e]) * (FP8 ? rsc[h] : gsc);
          emit(cg, e, rows[h], mm, v, ((int)(tile & 1) << 4) + g + 8 * h);
        }
      }
  };

  // A unit's K range is done.  A whole tile (ks = 1) is emitted now; a K
  // part's sums go to its slot, and the tile is combined once every warp has
  // streamed its units (after the main loop).
  auto finish_unit = [&](const UnitCursor& c) {
    const int64_t tile = (int64_t)tile0 + c.tl;
    if constexpr (BC) {
      float rg = acc[0][0] + acc[0][1], rh = acc[0][2] + acc[0][3];
      rg += __shfl_xor_sync(0xFFFFFFFFu, rg, 1);
      rh += __shfl_xor_sync(0xFFFFFFFFu, rh, 1);
      rg += __shfl_xor_sync(0xFFFFFFFFu, rg, 2);
      rh += __shfl_xor_sync(0xFFFFFFFFu, rh, 2);
      if (t == 0) {
        if (ks > 1) {
          float* slot = part + (size_t)(c.tl * ks + c.kp) * 16;
          slot[g] = rg;
          slot[g + 8] = rh;
        } else {
          emit_bc(tile, rg, rh);
        }
      }
    } else {
#pragma unroll
      for (int cg = 0; cg < NCG; ++cg)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[cg][i] += acc[cg][4 + i];
      if (ks > 1) {
        float* mine = part + ((size_t)(c.tl * ks + c.kp) * 32 + lane) * (4 * NCG);
#pragma unroll
        for (int cg = 0; cg < NCG; ++cg)
#pragma unroll
          for (int i = 0; i < 4; ++i) mine[4 * cg + i] = acc[cg][i];
      } else {
        emit_tile(tile);
      }
    }
#pragma unroll
    for (int a = 0; a < NACC; ++a)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[a][i] = 0.f;
  };

  // ---- main loop over this warp's stages
  int cj = 0, ci = 0, c_ib = 0, c_len = 0;
  uint32_t so0 = 0, so1 = 0;  // without scale_tma: 16-bit scale-pair offsets of rows g, g+8 (n k / 32 < 2^31)
  UnitCursor cc = first;
  auto set_cunit = [&]() {
    c_ib = kp_begin(cc.kp);
    c_len = kp_begin(cc.kp + 1) - c_ib;
    const int tile = tile0 + cc.tl;
    load_unit_extras(tile);
    if constexpr (!FP8) {
      int r0 = tile * 16 + g, r1 = r0 + 8;
      r0 = r0 < p.n ? r0 : (int)p.n - 1;  // rows past n: any valid scale (their codes read as 0)
      r1 = r1 < p.n ? r1 : (int)p.n - 1;
      so0 = (uint32_t)r0 * (uint32_t)(p.k / 32) + t;
      so1 = (uint32_t)r1 * (uint32_t)(p.k / 32) + t;
    }
  };
  if (nunits > 0) set_cunit();
  for (int q0 = 0; q0 < total; q0 += S) {
#pragma unroll
    for (int i = 0; i < S; ++i) {
      const int q = q0 + i;
      if (q < total) {
        if (failed_at == kAlive && !mbar_wait(bars + 8 * i, (uint32_t)(q / S) & 1u, p.dev_status))
          failed_at = q;
        const unsigned char* st = smem + (wring - base) + i * kStage;
        const int item = c_ib + ci;
        if constexpr (FP8) {  // box rows are two 128-element chunks of codes
          const uint2* bq = bbase + (int64_t)(8 * kItem * item) * BSTRIDE;
#pragma unroll
          for (int j = 0; j < kItem; ++j) {
            const unsigned char* rg = st + g * 256 + j * 128 + t * 32;
            const unsigned char* rh = st + (g + 8) * 256 + j * 128 + t * 32;
            const uint4 qg0 = *reinterpret_cast<const uint4*>(rg);
            const uint4 qg1 = *reinterpret_cast<const uint4*>(rg + 16);
            const uint4 qh0 = *reinterpret_cast<const uint4*>(rh);
            const uint4 qh1 = *reinterpret_cast<const uint4*>(rh + 16);
            chunk_mma_fp8<BSTRIDE, NCG, GSTRIDE>(acc, qg0, qg1, qh0, qh1, bq + 8 * j * BSTRIDE);
          }
        } else {
#pragma unroll
          for (int j = 0; j < kItem; ++j) {  // box rows are 128 bytes: chunk j at byte 64 j
            const uint4 qg = *reinterpret_cast<const uint4*>(st + g * 128 + j * 64 + t * 16);
            const uint4 qh = *reinterpret_cast<const uint4*>(st + (g + 8) * 128 + j * 64 + t * 16);
            uint32_t sg, sh;  // scale pairs (blocks 2t, 2t+1 of chunk j) of rows g, g+8
            if (p.scale_tma) {
              sg = *reinterpret_cast<const uint16_t*>(st + kScaleOff + g * 16 + 8 * j + 2 * t);
              sh = *reinterpret_cast<const uint16_t*>(st + kScaleOff + (g + 8) * 16 + 8 * j + 2 * t);
            } else {
              const int c = item * kItem + j;
              const uint16_t* sp = reinterpret_cast<const uint16_t*>(p.scales);
              sg = c < cmax ? __ldg(sp + so0 + 4 * c) : 0u;
              sh = c < cmax ? __ldg(sp + so1 + 4 * c) : 0u;
            }
            if constexpr (BC) {
              chunk_bc(acc[0], qg, qh, sg, sh, pb + (uint32_t)(item * kItem + j) * kBcChunkBytes);
            } else {
              const uint2* bq = bbase + (int64_t)(8 * (item * kItem + j)) * BSTRIDE;
              chunk_mma<BSTRIDE, NCG, GSTRIDE>(acc, qg, qh, sg, sh, bq);
            }
          }
        }
        __syncwarp();  // every lane is done with stage i before it is refilled
        if (q + S < total) issue(i);
        if (++ci == c_len) {
          finish_unit(cc);
          ci = 0;
          cc.next(ks);
          if (++cj < nunits) set_cunit();
        }
      }
    }
  }

  // After a wait ran out in lane 0, the copies of stages failed_at ..
  // failed_at + S - 1 (the last one on each ring stage) may still be in
  // flight: wait for them, again bounded, before the CTA's shared memory can
  // be released.
  if (lane == 0 && failed_at != kAlive) {
    for (int q = failed_at; q < total && q < failed_at + S; ++q)
      mbar_wait(bars + 8 * (q % S), (uint32_t)(q / S) & 1u, p.dev_status);
    if (threadIdx.x == 0 && prepped) mbar_wait(fbar, 0u, p.dev_status);  // thread 0's fragment copy
  }

  // Tiles split over K parts: once every warp has streamed its units, each
  // tile's part sums are added in K-part order (the same for every tile, so
  // equal weight rows give equal logits) and the tile is emitted.
  if (ks > 1) {
    __syncthreads();
    for (int tl = warp; tl < nt; tl += WARPS) {
      const int64_t tile = (int64_t)tile0 + tl;
      load_unit_extras((int)tile);
      if constexpr (BC) {
        if (t == 0) {
          const float* slot = part + (size_t)tl * ks * 16;
          float rg = 0.f, rh = 0.f;
          for (int q = 0; q < ks; ++q) {
            rg += slot[q * 16 + g];
            rh += slot[q * 16 + g + 8];
          }
          emit_bc(tile, rg, rh);
        }
      } else {
        const float* slot = part + ((size_t)tl * ks * 32 + lane) * (4 * NCG);
#pragma unroll
        for (int cg = 0; cg < NCG; ++cg) acc[cg][0] = acc[cg][1] = acc[cg][2] = acc[cg][3] = 0.f;
        for (int q = 0; q < ks; ++q) {
          const float* o = slot + (size_t)q * 32 * 4 * NCG;
#pragma unroll
          for (int cg = 0; cg < NCG; ++cg)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[cg][i] += o[4 * cg + i];
        }
        emit_tile(tile);
      }
    }
  }

  if (p.keys == nullptr) return;
  if constexpr (BC) {
    __syncwarp();
    if (t == 0) {
      best[0][0] = bc_run->key;
      lm[0][0] = bc_run->lm;
      ls[0][0] = bc_run->ls;
    }
  }
  // lanes sharing t hold the same batch columns: reduce over g, then per warp
  float2* lred = reinterpret_cast<float2*>(kred + WARPS * kMaxRows);  // [WARPS][kMaxRows]
#pragma unroll
  for (int cg = 0; cg < NCG; ++cg) {
#pragma unroll
    for (int e = 0; e < NE; ++e) {
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
  // one warp per batch row: lane w takes warp w's partials, then a fixed
  // shuffle tree (the log-sum-exp partial is combined in CTA order below)
  for (int m = warp; m < MM; m += WARPS) {
    unsigned long long b = lane < WARPS ? kred[lane * kMaxRows + m] : 0ull;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, b, o);
      b = other > b ? other : b;
    }
    if (lane == 0 && b != 0ull)
      asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(p.keys + m), "l"(b) : "memory");
    if (p.logprob != nullptr) {
      float cm = -INFINITY, cs = 0.f;
      if (lane < WARPS) {
        cm = lred[lane * kMaxRows + m].x;
        cs = lred[lane * kMaxRows + m].y;
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float om = __shfl_xor_sync(0xFFFFFFFFu, cm, o);
        const float os = __shfl_xor_sync(0xFFFFFFFFu, cs, o);
        lse_merge(cm, cs, om, os);
      }
      if (lane == 0) p.lse[(int64_t)blockIdx.x * kMaxRows + m] = make_float2(cm, cs);
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
        for (int w = 0; w < WARPS; ++w)
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

using KernelFn = void (*)(CUtensorMap, CUtensorMap, GemvParams);
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

// The block-column kernel (m = 1, NVFP4).
KernelFn bc_kernel() { return gemv_kernel<1, 16, false, true>; }

template <int WARPS, bool FP8>
KernelFn kernel_for(int m) {
  switch (m) {
    case 1: return gemv_kernel<1, WARPS, FP8, false>;
    case 2: return gemv_kernel<2, WARPS, FP8, false>;
    case 3: return gemv_kernel<3, WARPS, FP8, false>;
    case 4: return gemv_kernel<4, WARPS, FP8, false>;
    case 5: return gemv_kernel<5, WARPS, FP8, false>;
    case 6: return gemv_kernel<6, WARPS, FP8, false>;
    case 7: return gemv_kernel<7, WARPS, FP8, false>;
    case 8: return gemv_kernel<8, WARPS, FP8, false>;
    default: return gemv_kernel<16, WARPS, FP8, false>;  // 9..16 rows
  }
}

// 12 warps: the 8- and 16-row kernels whose activations (160 KB at 16 rows x
// 5120 or 8 rows x 10240) leave room for 12 rings but not 16
template <bool FP8>
KernelFn kernel_for12(int m) {
  switch (m) {
    case 8: return gemv_kernel<8, 12, FP8, false>;
    case 16: return gemv_kernel<16, 12, FP8, false>;
    default: return nullptr;
  }
}

// 13 warps: the 16-row kernel, whose 63-tile CTAs then give every warp at
// most 5 tiles instead of 6 (the rings of 13 warps still fit beside 16 rows of
// 5120 activations)
template <bool FP8>
KernelFn kernel_for13(int m) {
  return m == 16 ? gemv_kernel<16, 13, FP8, false> : nullptr;
}

struct Layout {
  uint32_t off_frag, off_zero, off_part, off_small, off_kred, off_bar;
  size_t bytes;  // dynamic shared memory to request (includes 1 KB alignment slack)
};

// Shared-memory carve-up: ring | activations (+ zero area) | split-K partials |
// prologue scratch | argmax reduction | ring barriers.
Layout layout_for(int warps, int m, int nchunks, bool fp8, bool bc, int part_slots, bool argmax) {
  const int S = ring_depth(fp8);
  const int cols = m <= 8 ? m : 16, ncg = (m + 7) / 8;  // the kernel's M, column groups
  Layout l;
  size_t off = (size_t)warps * S * stage_bytes(fp8);
  l.off_frag = (uint32_t)off;
  off += bc ? (size_t)nchunks * kBcChunkBytes : (size_t)nchunks * 8 * 4 * cols * sizeof(uint2);
  off = (off + 127) & ~(size_t)127;
  l.off_zero = (uint32_t)off;  // block-column path: running argmax state per (warp, g)
  off += bc ? (size_t)warps * 8 * sizeof(BcRun) : 0;
  l.off_part = (uint32_t)off;
  off += (size_t)part_slots * (bc ? 16 : 32 * 4 * ncg) * sizeof(float);
  off = (off + 15) & ~(size_t)15;
  l.off_small = (uint32_t)off;
  off += (size_t)small_floats(warps) * sizeof(float);
  off = (off + 15) & ~(size_t)15;
  l.off_kred = (uint32_t)off;  // argmax reduction: only read when the call wants the argmax
  if (argmax) off += (size_t)warps * kMaxRows * (sizeof(unsigned long long) + sizeof(float2));
  l.off_bar = (uint32_t)off;
  off += (size_t)warps * S * 8 + 8;  // ring barriers + the fragment-copy barrier
  l.bytes = off + 1024;
  return l;
}

// One launch for rows 0 .. m-1 (m <= 16) of the call; NVFP4_ERR_SHAPE when its
// activations do not fit one CTA's shared memory.  With a workspace of
// W4A16_GEMV_WS_BYTES(m, k) and m >= 2, a small grid (one CTA per row)
// prepares the activations once and every GEMV CTA copies them.
int launch_rows(const GemvParams& base, const WeightRef& w, cudaStream_t stream, void* workspace,
                size_t workspace_bytes) {
  GemvParams p = base;
  const int m = p.m;
  p.ntiles = nvfp4::cdiv(w.n, 16);
  p.nitems = (int)nvfp4::cdiv(w.k, kItemK);
  if (p.ntiles * 16 > 0x7FFFFFFFLL) return NVFP4_ERR_SHAPE;  // TMA row coordinate
  const int nchunks = p.nitems * kItem;
  const bool bc = (m == 1 && !w.fp8);
  const int sms = nvfp4::sm_count();
  // one CTA per SM, each with an equal share of the tiles
  p.tpc = (int)nvfp4::cdiv(p.ntiles, sms);
  const int64_t grid = nvfp4::cdiv(p.ntiles, p.tpc);
  if (grid > W4A16_GEMV_MAX_CTAS) return NVFP4_ERR_SHAPE;  // bound of the log-prob workspace

  KernelFn fn = nullptr;
  Layout lay{};
  int warps = 0;
  // 16 warps of up to 128 registers (one CTA per SM; 32 warps at 64
  // registers and 2 CTAs of 16 warps both measured slower), or 13 (16 rows),
  // 12 (8 and 16 rows) or 8 warps when the activations leave too little
  // shared memory for 16 rings
  for (int wv : {16, 13, 12, 8}) {
    if (bc && wv != 16) break;
    const int mk = m <= 8 ? m : 16;  // the kernel's M
    if (wv == 12 && mk != 8 && mk != 16) continue;
    if (wv == 13 && mk != 16) continue;
    KernelFn f = bc ? bc_kernel()
               : wv == 16 ? (w.fp8 ? kernel_for<16, true>(m) : kernel_for<16, false>(m))
               : wv == 13 ? (w.fp8 ? kernel_for13<true>(mk) : kernel_for13<false>(mk))
               : wv == 12 ? (w.fp8 ? kernel_for12<true>(mk) : kernel_for12<false>(mk))
                          : (w.fp8 ? kernel_for<8, true>(m) : kernel_for<8, false>(m));
    // split K only where a CTA has at most half as many tiles as warps: with
    // more, every warp already streams whole tiles, and splitting them so that
    // the last idle warps join in measured slower (14 tiles of 4096 on 16
    // warps: 18.9 us split 8 ways against 17.9 us whole)
    const int ks = std::max(1, std::min({wv / p.tpc, p.nitems, kMaxKs}));
    const Layout l = layout_for(wv, m, nchunks, w.fp8, bc, ks > 1 ? p.tpc * ks : 0, p.keys != nullptr);
    if (nvfp4::occupancy(reinterpret_cast<const void*>(f), wv * 32, l.bytes) >= 1) {
      fn = f;
      lay = l;
      warps = wv;
      p.ks = ks;
      for (int i = 0; i <= ks; ++i) p.kbeg[i] = (int)((int64_t)i * p.nitems / ks);
      break;
    }
  }
  if (fn == nullptr) return NVFP4_ERR_SHAPE;
  // The work split gives every SM one CTA's share: make sure no SM can take
  // two CTAs of this grid (the block scheduler may pack two onto the SMs that
  // free up first when the previous kernel ends unevenly), by asking for more
  // than half of an SM's shared memory.
  {
    int dev = 0, per_sm = 0, optin = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess) {
      const size_t half = (size_t)per_sm / 2 + 1;
      if (lay.bytes < half && half <= (size_t)optin) lay.bytes = half;
    }
  }
  p.off_frag = lay.off_frag;
  p.off_zero = lay.off_zero;
  p.off_part = lay.off_part;
  p.off_small = lay.off_small;
  p.off_kred = lay.off_kred;
  p.off_bar = lay.off_bar;

  CUtensorMap tmap;
  const int64_t row_bytes = w.fp8 ? w.k : w.k / 2;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)w.n};
    const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)(w.fp8 ? 256 : 128), 16};
    const cuuint32_t estr[2] = {1, 1};
    if (!nvfp4::encode_tiled(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(w.codes),
                             dims, strides, box, estr, CU_TENSOR_MAP_SWIZZLE_NONE))
      return NVFP4_ERR_CUDA;
  }
  // block scales [n, k/16] bytes: 16 rows x 16 bytes (two chunks) per stage,
  // when a row's k/16 bytes are a multiple of 16 (the TMA stride rule)
  CUtensorMap tmap_s = tmap;
  p.scale_tma = 0;
  if (!w.fp8 && w.k % 256 == 0) {
    const cuuint64_t dims[2] = {(cuuint64_t)(w.k / 16), (cuuint64_t)w.n};
    const cuuint64_t strides[1] = {(cuuint64_t)(w.k / 16)};
    const cuuint32_t box[2] = {16, 16};
    const cuuint32_t estr[2] = {1, 1};
    if (!nvfp4::encode_tiled(&tmap_s, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(w.scales), dims,
                             strides, box, estr, CU_TENSOR_MAP_SWIZZLE_NONE))
      return NVFP4_ERR_CUDA;
    p.scale_tma = 1;
  }

  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  const bool prep = !bc && m >= 2 && workspace != nullptr &&
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
  } else {
    p.frag_src = nullptr;
    p.rowmax_src = nullptr;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(warps * 32);
  cfg.dynamicSmemBytes = lay.bytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, fn, tmap, tmap_s, p) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
  return NVFP4_OK;
}

}  // namespace

// Batches wider than one launch's activation storage (up to 16 rows, fewer at
// large k) run as consecutive launches of row blocks on the same stream; each
// block streams the weights and produces its rows' outputs, argmax and
// log-probability.  The argmax workspace is reused in stream order.
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
  p.scales = w.scales;
  p.gscale = w.gscale;
  p.row_scale = w.row_scale;
  p.n = w.n;
  p.k = w.k;
  p.y_dtype = y_dtype;
  p.ldy = ldy;
  p.dev_status = dev_status;
  if (want_argmax) {
    p.keys = reinterpret_cast<unsigned long long*>(workspace);
    p.counter = reinterpret_cast<unsigned int*>(reinterpret_cast<char*>(workspace) + 8 * kMaxRows);
    p.lse = reinterpret_cast<float2*>(reinterpret_cast<char*>(workspace) + W4A16_ARGMAX_WS_BYTES);
  }
  const int esize = y_dtype == NVFP4_DTYPE_F32 ? 4 : 2;
  int r0 = 0;
  while (r0 < m) {
    // rows of this launch: up to 16, halved while their activations do not fit
    int rc = NVFP4_ERR_SHAPE;
    for (int mb = std::min(m - r0, kMaxRows); mb >= 1; mb = mb > 8 ? 8 : mb / 2) {
      GemvParams q = p;
      q.m = mb;
      for (int s = 0; s < nseg; ++s) {
        if (q.ridx[s] != nullptr)
          q.ridx[s] += r0;
        else
          q.x[s] += (int64_t)r0 * q.ld[s];
      }
      q.y = y == nullptr ? nullptr : reinterpret_cast<char*>(y) + (int64_t)r0 * ldy * esize;
      if (want_argmax) {
        q.argmax = argmax + r0;
        q.logprob = logprob == nullptr ? nullptr : logprob + r0;
        q.mask = mask == nullptr ? nullptr : mask + (int64_t)r0 * ld_mask;
        q.ld_mask = ld_mask;
      }
      rc = launch_rows(q, w, stream, workspace, workspace_bytes);
      if (rc != NVFP4_ERR_SHAPE) {
        r0 += mb;
        break;
      }
      if (mb == 1) break;
    }
    if (rc != NVFP4_OK) return rc;
  }
  return NVFP4_OK;
}
