// gemm.cu -- prefill W4A16 GEMM on the 5th-generation tensor cores (sm_103a).
//
//   C[m, n] = bf16( g * sum_k A[m, k] * w~[n, k] ),   w~ = e4m3(s[n, k/16]) * e2m1(c[n, k])
//
// Numerics of the lossless prefill path of "spark_model/layers/qwen3_attention/
// prefill_weights.rs" (w4a16_gemm_m128_dispatch, BF16 tensor-core variant): the
// FP4 weight is dequantised exactly to BF16 and multiplied with BF16 MMAs
// accumulating in FP32, one 128-row tile of A at a time.
//
// One persistent CTA per SM computes 256 x BN output tiles (256 activation
// rows, BN = 256 or 240 weight rows, chosen per call to fill whole waves) as
// two 128 x BN tcgen05.mma tiles (cta_group::1, kind::f16, BF16 x BF16 ->
// FP32) that share every dequantised weight tile, their accumulators side by
// side in tensor memory (2 x 256 columns).  K runs in steps of 64 through
// shared-memory rings (3 stages of A, 3 of B, released together):
//   warp 0       TMA producer: the two 128 x 64 BF16 A boxes of a step by
//                cp.async.bulk.tensor (128-byte swizzle; rows past m read as 0);
//   warp 1       allocates TMEM; one thread issues the 8 MMAs of a step (K = 16,
//                two halves), commits each stage's completion to its "empty"
//                barrier and a tile's last one to the accumulator barrier;
//   warps 2..    dequantise the BN x 64 weight tile (two threads per row,
//                32 K-elements each, four steps of loads in flight) into the
//                same 128-byte-swizzled K-major layout, fence the async proxy
//                and arrive on the stage's "full" barrier;
//   last 4 warps epilogue: tcgen05.ld of their TMEM lane quadrant for both
//                halves, 32 columns at a time, times g, round to BF16; each
//                64-column piece is transposed in 16-byte units across 8
//                lanes (shuffles), so one store instruction writes 4 rows x
//                128 contiguous bytes rather than 32 rows x 16 bytes; stores
//                up to n and m; TMEM goes back to the next tile right after
//                its last load.
// Dequantisation: E2M1 nibble pairs become BF16 bit patterns of value * 2^-126
// (integer ops), then one packed BF16 multiply by the block scale * 2^118
// (exact); the 2^8 left over is folded into g in the epilogue.
// Every wait is bounded (2 s of globaltimer): a wait that runs out records
// NVFP4_ERR_TIMEOUT in the caller's status word and the CTA unwinds: every
// role leaves its loop, the A loads and MMAs still in flight are waited for
// (bounded again), and TMEM is freed.
#include <cuda.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace {

constexpr int BM = 128, BK = 64;  // one MMA: 128 x BN, K steps of 64
// Output tiles are 256 x BN with BN = 256 or 240, chosen per call so that the
// tiles fill whole waves of the persistent grid (2048 x 17408: 544 tiles of
// 256 columns make 3.58 waves on 152 SMs, 584 tiles of 240 make 3.84).
// An output tile is kMHalves MMA tiles high: both halves share each dequantised
// B tile, so the dequantisation per FLOP halves with two.  Their accumulators
// then fill TMEM (2 x 256 columns) and the epilogue no longer overlaps the
// next tile's MMAs; with one half, the two accumulators double-buffer tiles.
constexpr int kMHalves = 2;
constexpr int BMT = BM * kMHalves;  // output tile rows
constexpr bool kSingleBuf = true;  // TMEM holds one tile's accumulators only (2 x up to 256 columns)
constexpr int kAccStride = 256;    // TMEM columns between the two halves' accumulators
// Ring depths (A tiles by TMA, B tiles by the dequantising warps); measured
// best: 3 + 3 with two halves (2+4, 4+2, 2+3 slower), 4 + 4 with one.  Also
// measured: 128-column tiles with four halves (N = 128 MMAs) are slower.
constexpr int kStagesA = kMHalves == 2 ? 3 : 4;
constexpr int kStagesB = kMHalves == 2 ? 3 : 4;
static_assert(kStagesA == kStagesB, "A and B stages advance together: one commit releases both");
constexpr int kAHalfBytes = BM * BK * 2;          // 16 KB
constexpr int kABytes = kMHalves * kAHalfBytes;
constexpr int kRingABytes = kStagesA * kABytes;
constexpr int kEpilogueWarps = 4;
// The tile-width dependent sizes.
template <int BN>
struct Tile {
  static constexpr int kBBytes = BN * BK * 2;  // 32 KB or 30 KB
  static constexpr int kRingBytes = kRingABytes + kStagesB * kBBytes;
  static constexpr int kDequantWarps = BN / 16;  // two threads per weight row, 32 K-elements each
  static constexpr int kThreads = (2 + kDequantWarps + kEpilogueWarps) * 32;
  static constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + (size_t)kRingBytes + 256;
  static_assert(BN % 16 == 0 && BN <= kAccStride, "tile width");
};
// TMEM columns: one tile's kMHalves accumulators, kAccStride apart
constexpr int kTmemCols = kMHalves * kAccStride;  // alloc unit: 512 columns
constexpr int kPrefetch = 4;       // k steps of weight rows in flight per dequant thread
constexpr unsigned long long kWaitLimitNs = nvfp4::kWaitLimit;

// ------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
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
// Bounded wait: false if it gave up (timeout here, or another role aborted).
// The same, letting the hardware suspend the warp for up to `hint_ns` while the
// phase is incomplete (a waiting warp then issues nothing).
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
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort,
                                          int32_t* dev_status) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, 100000u)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > kWaitLimitNs) {
      *abort = 1u;
      nvfp4::report(dev_status, NVFP4_ERR_TIMEOUT);
      return false;
    }
  }
}
// Bounded by time only: after an abort, lets work already in flight land.
__device__ __forceinline__ bool mbar_drain(uint32_t bar, uint32_t parity, int32_t* dev_status) {
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
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (SBO), version 1 (bits 46..47), start address >> 4.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f16: D = F32 (bits 4..5 = 1), A = B = BF16
// (bits 7..9 = 1, 10..12 = 1), both K-major, N >> 3 at bits 17..22, M >> 4 at
// bits 24..28.
// With A = B = F16 the formats are 0 (bits 7..9 and 10..12).
__host__ __device__ constexpr uint32_t idesc_f16kind(bool bf16, int n) {
  return (1u << 4) | (bf16 ? (1u << 7) | (1u << 10) : 0u) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(BM >> 4) << 24);
}

__device__ __forceinline__ void mma_f16kind(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Transpose of 16-byte pieces within each group of G lanes (G = 4 or 8): on
// entry lane gG + a holds pieces b = 0..G-1 (8 consecutive BF16 each) of its
// own row a; on exit lane gG + b holds piece b of rows a = 0..G-1 in slot a.
// Rounds m = 1, 2 (, 4) swap, between lanes l and l ^ m, the pieces whose
// (lane ^ slot) bit m is set.
template <int G>
__device__ __forceinline__ void transpose_pieces(uint4 (&P)[G], int lane) {
#pragma unroll
  for (int m = 1; m < G; m <<= 1) {
    const bool hi = (lane & m) != 0;
#pragma unroll
    for (int s0 = 0; s0 < G; ++s0) {
      if (s0 & m) continue;
      const int s1 = s0 | m;
      const uint4 snd = hi ? P[s0] : P[s1];
      uint4 rcv;
      rcv.x = __shfl_xor_sync(0xFFFFFFFFu, snd.x, m);
      rcv.y = __shfl_xor_sync(0xFFFFFFFFu, snd.y, m);
      rcv.z = __shfl_xor_sync(0xFFFFFFFFu, snd.z, m);
      rcv.w = __shfl_xor_sync(0xFFFFFFFFu, snd.w, m);
      if (hi)
        P[s0] = rcv;
      else
        P[s1] = rcv;
    }
  }
}

__device__ __forceinline__ uint4 ld_nc_u4(const void* p) {
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
// Two E4M3 scales (low byte first) -> bf16x2 patterns of scale * 2^118, each
// replicated into both halves (see the GEMV for the construction).
__device__ __forceinline__ void decode_scales(uint32_t s2, uint32_t& lo, uint32_t& hi) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)s2, __NV_E4M3);
  uint32_t v = ((uint32_t)h.x | ((uint32_t)h.y << 16)) >> 3;
  v = bf16x2_mul(v, 0x79007900u);
  v = bf16x2_mul(v, 0x79007900u);
  lo = __byte_perm(v, 0, 0x1010);
  hi = __byte_perm(v, 0, 0x3232);
}
// prmt.b32 in its generic mode: a selector nibble with bit 3 set replicates
// the sign bit of the selected byte (CUDA's __byte_perm masks that bit off).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
// The 8 E2M1 codes of word q (k = 8w..8w+7, natural order) -> 4 bf16x2 patterns
// (value * 2^-126) times scale pattern s.  Pair p = (nibble 2p, nibble 2p+1):
// one byte_perm places nibble 2p in bits 0..3 and nibble 2p+1 in bits 16..19
// (zero bytes come from the sign-replicate mode on bytes whose top bit is 0);
// the multiply by 0x1040 makes the two shifted copies whose masked bits are
// the sign (bit 15) and the 3 magnitude bits (8..6) of each half.
__device__ __forceinline__ uint4 dequant_word(uint32_t q, uint32_t s) {
  const uint32_t ev = q & 0x0F0F0F0Fu, od = (q >> 4) & 0x0F0F0F0Fu;
  const uint32_t p0 = prmt(ev, od, 0xC480u);
  const uint32_t p1 = prmt(ev, od, 0xD591u);
  const uint32_t p2 = prmt(ev, od, 0xE6A2u);
  const uint32_t p3 = prmt(ev, od, 0xF7B3u);
  uint4 r;
  r.x = bf16x2_mul((p0 * 0x1040u) & 0x81C081C0u, s);
  r.y = bf16x2_mul((p1 * 0x1040u) & 0x81C081C0u, s);
  r.z = bf16x2_mul((p2 * 0x1040u) & 0x81C081C0u, s);
  r.w = bf16x2_mul((p3 * 0x1040u) & 0x81C081C0u, s);
  return r;
}

__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// Two E4M3 scales (low byte first) -> F16 (exact), each replicated into both
// halves of an f16x2.
__device__ __forceinline__ void decode_scales_f16(uint32_t s2, uint32_t& lo, uint32_t& hi) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)s2, __NV_E4M3);
  const uint32_t v = (uint32_t)h.x | ((uint32_t)h.y << 16);
  lo = __byte_perm(v, 0, 0x1010);
  hi = __byte_perm(v, 0, 0x3232);
}
// The 8 E2M1 codes of word q (natural order) -> 4 f16x2 by the hardware
// conversion (byte j = elements 2j, 2j+1), times the block-scale pattern s:
// every product is an exact F16 (at most 6 significant bits).
__device__ __forceinline__ uint4 dequant_word_f16(uint32_t q, uint32_t s) {
  uint32_t h0, h1, h2, h3;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
      : "r"(q));
  return make_uint4(f16x2_mul(h0, s), f16x2_mul(h1, s), f16x2_mul(h2, s), f16x2_mul(h3, s));
}

struct GemmParams {
  const uint8_t* packed;
  const uint8_t* scales;
  const float* gscale;
  __nv_bfloat16* c;
  int64_t m, n, k, ldc;
  int mtiles, ntiles;
  const float* row_inv;  // FP16 path: 2^-e of each activation row's staging scale
  int32_t* dev_status;
};

// Tile t of the persistent schedule: consecutive t share one 256-row weight
// slice (n tile), so the CTAs working on it at the same time find it in L2.
template <int BN>
__device__ __forceinline__ void tile_coords(const GemmParams& p, int t, int64_t& m0, int64_t& n0) {
  m0 = (int64_t)(t % p.mtiles) * BMT;
  n0 = (int64_t)(t / p.mtiles) * BN;
}

// F16 = false: A is the caller's BF16 activations, B is dequantised to BF16.
// F16 = true:  A is an FP16 copy of the activations, each row scaled by an
//              exact power of two (staged by stage_a_f16 in the workspace), B is
//              dequantised to FP16 with the hardware E2M1 conversion (fewer
//              instructions per weight); the epilogue removes the row scale.
template <bool F16, int BN>
__global__ void __launch_bounds__(Tile<BN>::kThreads, 1)
gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ GemmParams p) {
  constexpr uint32_t kIdesc = idesc_f16kind(!F16, BN);
  constexpr int kBBytes = Tile<BN>::kBBytes, kRingBytes = Tile<BN>::kRingBytes;
  constexpr int kDequantWarps = Tile<BN>::kDequantWarps;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle wants 1 KB alignment
  unsigned char* const smem = smem_raw + (base - raw);
  // ring layout: kStagesA A tiles, then kStagesB B tiles (all 1 KB aligned)
  auto a_tile = [&](int s) { return base + (uint32_t)(s * kABytes); };
  auto b_tile = [&](int s) { return (uint32_t)(kRingABytes + s * kBBytes); };  // offset from base
  const uint32_t bars = base + kRingBytes;
  auto full_a = [&](int s) { return bars + 8u * s; };
  auto empty_a = [&](int s) { return bars + 8u * (kStagesA + s); };
  auto full_b = [&](int s) { return bars + 8u * (2 * kStagesA + s); };
  constexpr int kNbar = 2 * kStagesA + 2 * kStagesB;
  auto tmem_full = [&](int b) { return bars + 8u * (kNbar + b); };
  auto tmem_empty = [&](int b) { return bars + 8u * (kNbar + 2 + b); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kRingBytes + 8 * (kNbar + 4));
  volatile uint32_t* abort = tmem_slot + 1;
  const uint32_t drain_bar = bars + 8u * (kNbar + 5);  // the MMAs in flight after an abort
  static_assert(8 * (kNbar + 6) <= 256, "barriers, TMEM slot and abort flag exceed their 256 bytes");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = (int)(p.k / BK);
  const int ntiles_all = p.mtiles * p.ntiles;
  // tiles of this CTA: blockIdx.x, blockIdx.x + gridDim.x, ...
  const int my_tiles =
      (int)blockIdx.x < ntiles_all ? (ntiles_all - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int total = my_tiles * nk;  // k steps streamed through the ring

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesA; ++s) {
      mbar_init(full_a(s), 1);
      mbar_init(empty_a(s), 1);
    }
    for (int s = 0; s < kStagesB; ++s) {
      mbar_init(full_b(s), kDequantWarps);  // (stage s of B is released by empty_a(s))
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tmem_full(b), 1);
      mbar_init(tmem_empty(b), kEpilogueWarps);
    }
    mbar_init(drain_bar, 1);
    *abort = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  int a_issued = 0;  // A-tile loads issued (TMA producer)

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      for (int g = 0; g < total; ++g) {
        const int s = g % kStagesA, r = g / kStagesA;
        const int kb = g % nk;
        int64_t m0, n0;
        tile_coords<BN>(p, (int)blockIdx.x + (g / nk) * (int)gridDim.x, m0, n0);
        if (r > 0 && !mbar_wait(empty_a(s), (r - 1) & 1, abort, p.dev_status)) break;
        a_issued = g + 1;
        if (nvfp4::kWithhold && blockIdx.x == 0 && g == 0) continue;  // test build: never issued
        mbar_arrive_expect_tx(full_a(s), kABytes);
#pragma unroll
        for (int h = 0; h < kMHalves; ++h)
          tma_load_2d(a_tile(s) + (uint32_t)(h * kAHalfBytes), &tmap_a, kb * BK, (int)m0 + h * BM,
                      full_a(s));
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      for (int it = 0; it < my_tiles && ok; ++it) {
        // accumulator buffer: the tile's halves fill TMEM, or tiles alternate
        const int ab = kSingleBuf ? 0 : (it & 1);
        const int nb = kSingleBuf ? 1 : 2;  // tiles per buffer reuse cycle
        if (it >= nb && !mbar_wait(tmem_empty(ab), ((it / nb) - 1) & 1, abort, p.dev_status)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(ab * kMHalves * kAccStride);
        for (int kb = 0; kb < nk; ++kb) {
          const int g = it * nk + kb;
          const int sa = g % kStagesA, ra = g / kStagesA;
          const int sb = g % kStagesB, rb = g / kStagesB;
          ok = mbar_wait(full_a(sa), ra & 1, abort, p.dev_status) &&
               mbar_wait(full_b(sb), rb & 1, abort, p.dev_status);
          if (!ok) break;
          tc_fence_after();
          const uint64_t ad = smem_desc(a_tile(sa));
          const uint64_t bd = smem_desc(base + b_tile(sb));
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {  // advance 32 bytes (16 BF16) along K
#pragma unroll
            for (int h = 0; h < kMHalves; ++h)
              mma_f16kind(d + (uint32_t)(h * kAccStride), ad + (uint64_t)(h * (kAHalfBytes >> 4)) + 2 * kk,
                          bd + 2 * kk, kIdesc, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(empty_a(sa));  // releases stage sa of both rings (sa == sb)
        }
        mma_commit(tmem_full(ab));  // fires once the tile's MMAs have completed
      }
    }
  } else if (warp < 2 + kDequantWarps) {
    // --------------------------------------------------------------- dequant
    const int d = threadIdx.x - 64;
    const int r = d >> 1, h = d & 1;  // B-tile row 0..255, K half (32 elements) 0..1
    const uint32_t swz = (uint32_t)(r & 7);
    uint4 qa[kPrefetch];
    uint32_t qs[kPrefetch];
    // load cursor over (tile, k step): row pointers change once per tile
    int lt = 0, lkb = 0;
    const uint8_t* wp = nullptr;
    const uint16_t* sp = nullptr;
    bool lvalid = false;
    auto set_tile = [&](int it) {
      int64_t m0, n0;
      tile_coords<BN>(p, (int)blockIdx.x + it * (int)gridDim.x, m0, n0);
      const int64_t nrow = n0 + r;
      lvalid = nrow < p.n;
      wp = p.packed + (lvalid ? nrow : 0) * (p.k / 2) + 16 * h;
      sp = reinterpret_cast<const uint16_t*>(p.scales + (lvalid ? nrow : 0) * (p.k / 16)) + h;
    };
    set_tile(0);
    auto issue = [&](int i) {
      if (lvalid) {  // rows past n: zero weights (their outputs are not stored)
        qa[i] = ld_nc_u4(wp + (int64_t)lkb * 32);
        qs[i] = __ldg(sp + 2 * lkb);
      } else {
        qa[i] = make_uint4(0, 0, 0, 0);
        qs[i] = 0u;
      }
      if (++lkb == nk) {
        lkb = 0;
        if (++lt < my_tiles) set_tile(lt);
      }
    };
#pragma unroll
    for (int i = 0; i < kPrefetch; ++i)
      if (i < total) issue(i);
    bool ok = true;
    for (int g0 = 0; g0 < total && ok; g0 += kPrefetch) {
#pragma unroll
      for (int i = 0; i < kPrefetch; ++i) {
        const int g = g0 + i;
        if (g < total && ok) {
          const int s = g % kStagesB, rr = g / kStagesB;
          const uint4 c0 = qa[i];
          const uint32_t cs = qs[i];
          if (g + kPrefetch < total) issue(i);
          if (rr > 0 && !mbar_wait(empty_a(s), (rr - 1) & 1, abort, p.dev_status)) {
            ok = false;
          } else {
            uint32_t S0, S1;
            if constexpr (F16)
              decode_scales_f16(cs, S0, S1);
            else
              decode_scales(cs, S0, S1);
            const uint32_t words[4] = {c0.x, c0.y, c0.z, c0.w};
            unsigned char* brow = smem + b_tile(s) + r * 128;
#pragma unroll
            for (int j = 0; j < 4; ++j) {  // chunk 4h+j holds k = 32h + 8j .. +7
              uint4 v;
              if constexpr (F16)
                v = dequant_word_f16(words[j], j < 2 ? S0 : S1);
              else
                v = dequant_word(words[j], j < 2 ? S0 : S1);
              *reinterpret_cast<uint4*>(brow + (((uint32_t)(4 * h + j) ^ swz) << 4)) = v;
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(full_b(s));
          }
        }
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue
    // warp quadrant q owns TMEM lanes 32q..32q+31 = rows 32q.. of the tile
    const int q = warp & 3;
    // BF16 path: g * 2^8 (the dequant fold); FP16 path: g, and 2^-e per row
    const float gs = F16 ? __ldg(p.gscale) : __ldg(p.gscale) * 256.0f;
    for (int it = 0; it < my_tiles; ++it) {
      const int ab = kSingleBuf ? 0 : (it & 1);
      const int nb = kSingleBuf ? 1 : 2;
      __syncwarp();
      if (!mbar_wait(tmem_full(ab), (it / nb) & 1, abort, p.dev_status)) break;
      __syncwarp();
      tc_fence_after();
      int64_t m0, n0;
      tile_coords<BN>(p, (int)blockIdx.x + it * (int)gridDim.x, m0, n0);
      // Each half's rows in 64-column pieces (two 32-column TMEM loads, an 8 x 8
      // transpose of 16-byte pieces within each group of 8 lanes, then 8 stores
      // that each write 4 rows x 128 contiguous bytes), and at BN = 240 the last
      // 48 columns as 32 + 16 (4-lane groups: 8 rows x 64 bytes per store).
      // Columns are stored up to n; rows up to m.
      constexpr int kWide = BN / 64, kRest = BN - 64 * kWide;
      const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
#pragma unroll 1
      for (int h = 0; h < kMHalves; ++h) {
        const int64_t rbase = m0 + h * BM + 32 * q;  // the warp's first row
        const int64_t row = rbase + lane;
        const float rs = (F16 && row < p.m) ? __ldg(p.row_inv + row) : 1.0f;
        const uint32_t tacc = tq + (uint32_t)((ab * kMHalves + h) * kAccStride);
        const bool last_half = h == kMHalves - 1;
        auto convert = [&](const uint32_t (&v)[32], uint4* P, int npieces) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (i >= npieces) {
              P[i] = make_uint4(0u, 0u, 0u, 0u);
              continue;
            }
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              __nv_bfloat162 b2 = __floats2bfloat162_rn((__uint_as_float(v[8 * i + 2 * e]) * rs) * gs,
                                                        (__uint_as_float(v[8 * i + 2 * e + 1]) * rs) * gs);
              w4[e] = *reinterpret_cast<uint32_t*>(&b2);
            }
            P[i] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        };
        auto release_if_done = [&](bool done) {  // TMEM fully read: the next tile may start
          if (done) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tmem_empty(ab));
          }
        };
#pragma unroll 1
        for (int c = 0; c < kWide; ++c) {
          uint4 P[8];
          uint32_t v[32];
          tmem_ld32(tacc + (uint32_t)(64 * c), v);
          convert(v, P, 4);
          tmem_ld32(tacc + (uint32_t)(64 * c + 32), v);
          release_if_done(last_half && kRest == 0 && c == kWide - 1);
          convert(v, P + 4, 4);
          transpose_pieces<8>(P, lane);
          const int j = lane & 7;
          const int64_t cc = n0 + 64 * c + 8 * j;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int64_t r = rbase + (lane & ~7) + k;
            if (r < p.m && cc < p.n) *reinterpret_cast<uint4*>(p.c + r * p.ldc + cc) = P[k];
          }
        }
        if constexpr (kRest > 0) {
          static_assert(kRest == 48, "the last columns are one 32-column and one 16-column load");
#pragma unroll 1
          for (int u = 0; u < 2; ++u) {
            const int col = 64 * kWide + 32 * u;
            uint4 P[4];
            uint32_t v[32];
            if (u == 0) {
              tmem_ld32(tacc + (uint32_t)col, v);
            } else {
              uint32_t v16[16];
              tmem_ld16(tacc + (uint32_t)col, v16);
#pragma unroll
              for (int i = 0; i < 16; ++i) v[i] = v16[i];
#pragma unroll
              for (int i = 16; i < 32; ++i) v[i] = 0u;
            }
            release_if_done(last_half && u == 1);
            convert(v, P, u == 0 ? 4 : 2);
            transpose_pieces<4>(P, lane);
            const int j = lane & 3;
            const int64_t cc = n0 + col + 8 * j;
            if (u == 0 || j < 2) {
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const int64_t r = rbase + (lane & ~3) + k;
                if (r < p.m && cc < p.n) *reinterpret_cast<uint4*>(p.c + r * p.ldc + cc) = P[k];
              }
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (*abort) {
    // A wait ran out somewhere in the CTA: the last A load on each stage and
    // the MMAs already issued may still be in flight.  Wait for them (bounded)
    // before TMEM is freed and the CTA's shared memory released.
    if (warp == 0 && lane == 0)
      for (int g = a_issued > kStagesA ? a_issued - kStagesA : 0; g < a_issued; ++g)
        mbar_drain(full_a(g % kStagesA), (uint32_t)(g / kStagesA) & 1u, p.dev_status);
    if (warp == 1 && lane == 0) {
      mma_commit(drain_bar);  // arrives once every MMA this thread issued has completed
      mbar_drain(drain_bar, 0u, p.dev_status);
    }
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                 : "memory");
  }
}

// One CTA per activation row: FP16 copy of the row times 2^e, where e puts the
// row's largest BF16 magnitude in [2^14, 2^15) (every activation within 2^-31
// of it converts exactly: 8 significant bits, FP16 normal range); 2^-e kept for
// the epilogue.  e is clamped to [-120, 120]; an all-zero row uses e = 0.
constexpr int kStageThreads = 256;
__global__ void __launch_bounds__(kStageThreads)
stage_a_f16(const __nv_bfloat16* __restrict__ a, int64_t lda, int64_t k, __half* __restrict__ out,
            float* __restrict__ row_inv) {
  const int64_t row = blockIdx.x;
  const uint4* src = reinterpret_cast<const uint4*>(a + row * lda);
  uint4* dst = reinterpret_cast<uint4*>(out + row * k);
  const int64_t nvec = k / 8;
  uint32_t m2 = 0;
  for (int64_t i = threadIdx.x; i < nvec; i += kStageThreads) {
    const uint4 v = src[i];
    m2 = __vmaxu2(m2, __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                               __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu)));
  }
  uint32_t mx = max(m2 & 0xFFFFu, m2 >> 16);
  mx = __reduce_max_sync(0xFFFFFFFFu, mx);
  __shared__ uint32_t red[kStageThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = 0;
  for (int w = 0; w < kStageThreads / 32; ++w) mx = max(mx, red[w]);
  const int ef = (int)(mx >> 7);
  int e = mx == 0u ? 0 : 14 - (ef == 0 ? -126 : ef - 127);
  e = e < -120 ? -120 : (e > 120 ? 120 : e);
  const float sc = ldexpf(1.0f, e);
  if (threadIdx.x == 0) row_inv[row] = ldexpf(1.0f, -e);
  for (int64_t i = threadIdx.x; i < nvec; i += kStageThreads) {
    const uint4 v = src[i];
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __half2 h = __floats2half2_rn(__uint_as_float(u[j] << 16) * sc,
                                          __uint_as_float(u[j] & 0xFFFF0000u) * sc);
      o[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
    dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace

size_t gemm_f16_workspace_bytes(int64_t m, int64_t k) {
  return (size_t)m * (size_t)k * 2 + (size_t)m * 4 + 256;
}

int launch_gemm(const void* a, int64_t m, int64_t lda, const nvfp4_weight* w, void* c,
                int64_t ldc, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                cudaStream_t stream) {
  // FP16 path when the workspace can hold the staged activations
  const bool f16 = workspace != nullptr && workspace_bytes >= gemm_f16_workspace_bytes(m, w->k) &&
                   nvfp4::aligned16(workspace) && m <= 0x7FFFFFFF;
  __half* a16 = reinterpret_cast<__half*>(workspace);
  float* row_inv = f16 ? reinterpret_cast<float*>(
                             reinterpret_cast<char*>(workspace) + (((size_t)m * w->k * 2 + 15) & ~(size_t)15))
                       : nullptr;
  if (f16) {
    stage_a_f16<<<(unsigned)m, kStageThreads, 0, stream>>>(
        reinterpret_cast<const __nv_bfloat16*>(a), lda, w->k, a16, row_inv);
    if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
  }
  CUtensorMap tmap;
  const cuuint64_t dims[2] = {(cuuint64_t)w->k, (cuuint64_t)m};
  const cuuint64_t strides[1] = {(cuuint64_t)(f16 ? w->k : lda) * 2};
  const cuuint32_t box[2] = {BK, BM};
  const cuuint32_t estr[2] = {1, 1};
  if (!nvfp4::encode_tiled(&tmap, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                           2, f16 ? static_cast<void*>(a16) : const_cast<void*>(a), dims, strides, box,
                           estr, CU_TENSOR_MAP_SWIZZLE_128B))
    return NVFP4_ERR_CUDA;
  GemmParams p;
  p.packed = w->packed;
  p.scales = w->scales;
  p.gscale = w->global_scale;
  p.c = reinterpret_cast<__nv_bfloat16*>(c);
  p.m = m;
  p.n = w->n;
  p.k = w->k;
  p.ldc = ldc;
  p.mtiles = (int)nvfp4::cdiv(m, BMT);
  p.row_inv = row_inv;
  p.dev_status = dev_status;
  // tile width: the one whose tiles, in whole waves of one CTA per SM, take
  // the least time (a tile's time taken as its width plus a fixed 16)
  const int sms = nvfp4::sm_count();
  auto cost = [&](int bn) {
    return nvfp4::cdiv((int64_t)p.mtiles * nvfp4::cdiv(w->n, bn), sms) * (bn + 16);
  };
  const bool narrow = cost(240) < cost(256);
  const int bn = narrow ? 240 : 256;
  p.ntiles = (int)nvfp4::cdiv(w->n, bn);
  const void* kern =
      narrow ? (f16 ? (const void*)gemm_tcgen05_kernel<true, 240> : (const void*)gemm_tcgen05_kernel<false, 240>)
             : (f16 ? (const void*)gemm_tcgen05_kernel<true, 256> : (const void*)gemm_tcgen05_kernel<false, 256>);
  const int threads = narrow ? Tile<240>::kThreads : Tile<256>::kThreads;
  const size_t smem = narrow ? Tile<240>::kSmemBytes : Tile<256>::kSmemBytes;
  if (nvfp4::occupancy(kern, threads, smem) < 1) return NVFP4_ERR_CUDA;
  const int64_t tiles = (int64_t)p.mtiles * p.ntiles;
  if (tiles > 0x7FFFFFFF) return NVFP4_ERR_SHAPE;
  const unsigned grid = (unsigned)(tiles < sms ? tiles : sms);  // persistent: one CTA per SM
  void* args[] = {&tmap, &p};
  if (cudaLaunchKernel(kern, dim3(grid), dim3(threads), args, smem, stream) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  return NVFP4_OK;
}
