// gemm.cu -- prefill W4A16 GEMM on the 5th-generation tensor cores (sm_103a).
//
//   C[m, n] = bf16( g * sum_k A[m, k] * w~[n, k] ),   w~ = e4m3(s[n, k/16]) * e2m1(c[n, k])
//
// Numerics of the lossless prefill path of "spark_model/layers/qwen3_attention/
// prefill_weights.rs" (w4a16_gemm_m128_dispatch, BF16 tensor-core variant): the
// FP4 weight is dequantised exactly to BF16 and multiplied with BF16 MMAs
// accumulating in FP32, one 128-row tile of A at a time.
//
// One persistent CTA per SM computes 256 x 256 output tiles (256 activation
// rows, 256 weight rows) as two 128 x 256 tcgen05.mma tiles (cta_group::1,
// kind::f16, BF16 x BF16 -> FP32) that share every dequantised weight tile,
// their accumulators side by side in tensor memory (2 x 256 columns).  K runs
// in steps of 64 through shared-memory rings (3 stages of A, 3 of B):
//   warp 0       TMA producer: the two 128 x 64 BF16 A boxes of a step by
//                cp.async.bulk.tensor (128-byte swizzle; rows past m read as 0);
//   warp 1       allocates TMEM; one thread issues the 8 MMAs of a step (K = 16,
//                two halves), commits each stage's completion to its "empty"
//                barriers and a tile's last one to the accumulator barrier;
//   warps 2..17  dequantise the 256 x 64 weight tile (two threads per row,
//                32 K-elements each, four steps of loads in flight) into the
//                same 128-byte-swizzled K-major layout, fence the async proxy
//                and arrive on the stage's "full" barrier;
//   warps 18..21 epilogue: tcgen05.ld of their TMEM lane quadrant for both
//                halves, times g, round to BF16, store; then release TMEM to
//                the next tile.
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

// A CTA pair (cluster of 2) computes 256 x BN output tiles with one
// tcgen05.mma.cta_group::2 (M = 256) per K = 16 step: CTA r of the pair holds
// activation rows 128r..128r+127 of the tile and weight rows (BN/2)r ..
// (BN/2)(r+1)-1 in its shared memory, and its 128 x BN accumulator in its
// tensor memory.  BN (a multiple of 16, at most 256) is chosen per call so
// that the tiles fill the pairs' waves.
constexpr int BM = 128, BK = 64;     // A rows per CTA, K step
constexpr int kMaxBN = 256;          // MMA N (the pair's tile width)
constexpr int kMaxHalfN = kMaxBN / 2;  // weight rows per CTA
constexpr int kStages = 6;           // ring depth (A and B stages advance together)
constexpr int kABytes = BM * BK * 2;          // 16 KB
constexpr int kBBytes = kMaxHalfN * BK * 2;   // 16 KB
constexpr int kRingABytes = kStages * kABytes;
constexpr int kRingBytes = kRingABytes + kStages * kBBytes;
constexpr int kDequantWarps = kMaxHalfN / 8;  // four threads per weight row, 16 K-elements each
constexpr int kEpilogueWarps = 4;
constexpr int kThreads = (2 + kDequantWarps + kEpilogueWarps) * 32;
constexpr int kAccCols = 256;        // TMEM columns per accumulator buffer
constexpr int kTmemCols = 2 * kAccCols;  // two buffers: a tile's epilogue overlaps the next's MMAs
constexpr int kPrefetch = 6;         // k steps of weight rows in flight per dequant thread
constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + (size_t)kRingBytes + 512;
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
// try_wait on a barrier of this CTA.  CLUSTER: acquire at cluster scope, for
// barriers the peer CTA arrives on (its arrivals release at cluster scope).
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  if (CLUSTER)
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
  else
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
  return ok != 0;
}
// The same, letting the hardware suspend the warp for up to `hint_ns` while the
// phase is incomplete (a waiting warp then issues nothing).
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  if (CLUSTER)
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
  else
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
  return ok != 0;
}
// Bounded wait: false if it gave up (timeout here, or another role of this CTA
// aborted).
// SPIN: poll without the suspend hint (the MMA issuer and the stage relay,
// whose waits sit on the critical path).
template <bool CLUSTER = false, bool SPIN = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort,
                                          int32_t* dev_status) {
  if (mbar_try_wait<CLUSTER>(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    if (SPIN ? mbar_try_wait<CLUSTER>(bar, parity)
             : mbar_try_wait_sleep<CLUSTER>(bar, parity, 100000u))
      return true;
    if (*abort) return false;
    if (globaltimer() - t0 > kWaitLimitNs) {
      *abort = 1u;
      nvfp4::report(dev_status, NVFP4_ERR_TIMEOUT);
      return false;
    }
  }
}
// Arrive on the barrier at the same shared-memory offset in CTA `rank` of the
// cluster (this CTA included), releasing this thread's prior writes at
// cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(bar), "r"(rank));
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote)
               : "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// All threads of both CTAs of the pair.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
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
// The same load into this CTA's shared memory with the completion (complete_tx)
// signalled on a barrier of CTA 0 of the pair (bar: a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_to_rank0(uint32_t dst, const CUtensorMap* map, int c0,
                                                     int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
// 16 bytes from this CTA's shared memory to CTA 0's (both shared::cluster
// addresses there: dst, bar) with complete_tx on CTA 0's barrier: a signal
// that needs no fence in the issuing thread.
__device__ __forceinline__ void bulk_token_to_rank0(uint32_t dst, uint32_t src, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], 16, [%2];" ::"r"(
          dst),
      "r"(src), "r"(bar)
      : "memory");
}
__device__ __forceinline__ uint32_t mapa_rank0(uint32_t addr) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(0));
  return r;
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
// (bits 7..9 = 1, 10..12 = 1) or F16 (format 0), both K-major, N >> 3 at bits
// 17..22, M >> 4 at bits 24..28 (M = 256: the pair's two 128-row halves).
__host__ __device__ constexpr uint32_t idesc_f16kind(bool bf16, int n) {
  return (1u << 4) | (bf16 ? (1u << 7) | (1u << 10) : 0u) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(2 * BM >> 4) << 24);
}

// One M = 256 MMA of the pair, issued by one thread of the even CTA: A rows
// 0..127 from this CTA's shared memory at adesc, rows 128..255 from the peer's
// at the same offset; B columns split the same way (N/2 per CTA); D in each
// CTA's tensor memory at tmem_d.
__device__ __forceinline__ void mma_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive (once) on the barrier at this offset in both CTAs when every MMA this
// thread issued so far has completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"((uint16_t)3)
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
  int bn;      // pair tile width (MMA N): a multiple of 16, at most kMaxBN
  int npairs;  // CTA pairs of the persistent grid
  const float* row_inv;  // FP16 path: 2^-e of each activation row's staging scale
  int32_t* dev_status;
};

// Tile t of the persistent schedule: consecutive t share one weight slice (n
// tile), so the pairs working on it at the same time find it in L2.
__device__ __forceinline__ void tile_coords(const GemmParams& p, int t, int64_t& m0, int64_t& n0) {
  m0 = (int64_t)(t % p.mtiles) * (2 * BM);
  n0 = (int64_t)(t / p.mtiles) * p.bn;
}

// F16 = false: A is the caller's BF16 activations, B is dequantised to BF16.
// F16 = true:  A is an FP16 copy of the activations, each row scaled by an
//              exact power of two (staged by stage_a_f16 in the workspace), B is
//              dequantised to FP16 with the hardware E2M1 conversion (fewer
//              instructions per weight); the epilogue removes the row scale.
// Launched as clusters of two CTAs (one per SM); rank 0 issues the MMAs.
template <bool F16>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ GemmParams p) {
  const uint32_t idesc = idesc_f16kind(!F16, p.bn);
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle wants 1 KB alignment
  unsigned char* const smem = smem_raw + (base - raw);
  // ring layout: kStages A tiles, then kStages B tiles (all 1 KB aligned); the
  // same offsets in both CTAs of the pair
  auto a_tile = [&](int s) { return base + (uint32_t)(s * kABytes); };
  auto b_tile = [&](int s) { return (uint32_t)(kRingABytes + s * kBBytes); };  // offset from base
  const uint32_t bars = base + kRingBytes;
  auto full_a = [&](int s) { return bars + 8u * s; };
  auto empty_a = [&](int s) { return bars + 8u * (kStages + s); };
  auto full_b = [&](int s) { return bars + 8u * (2 * kStages + s); };
  auto empty_b = [&](int s) { return bars + 8u * (3 * kStages + s); };
  constexpr int kNbar = 4 * kStages;
  auto tmem_full = [&](int b) { return bars + 8u * (kNbar + b); };
  auto tmem_empty = [&](int b) { return bars + 8u * (kNbar + 2 + b); };  // rank 0 only
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kRingBytes + 8 * (kNbar + 5));
  volatile uint32_t* abort = tmem_slot + 1;
  const uint32_t drain_bar = bars + 8u * (kNbar + 4);  // the MMAs in flight after an abort
  // 16 bytes that the stage tokens copy from rank 1 to the same place in rank 0
  const uint32_t token = bars + (uint32_t)((8 * (kNbar + 6) + 15) & ~15);
  static_assert(((8 * (kNbar + 6) + 15) & ~15) + 16 <= 512,
                "barriers, TMEM slot, abort flag and token exceed their 512 bytes");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int pair = (int)(blockIdx.x >> 1);
  const int half_n = p.bn / 2;  // weight rows of this CTA
  const int nk = (int)(p.k / BK);
  const int ntiles_all = p.mtiles * p.ntiles;
  // tiles of this pair: pair, pair + npairs, ...
  const int my_tiles = pair < ntiles_all ? (ntiles_all - 1 - pair) / p.npairs + 1 : 0;
  const int total = my_tiles * nk;  // k steps streamed through the ring

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_a(s), 1);
      mbar_init(empty_a(s), 1);
      mbar_init(full_b(s), kDequantWarps);
      mbar_init(empty_b(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tmem_full(b), 1);
      mbar_init(tmem_empty(b), 2 * kEpilogueWarps);  // both CTAs' epilogue warps
    }
    mbar_init(drain_bar, 1);
    *abort = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    // both CTAs of the pair allocate together (the same columns in each)
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  int a_issued = 0;  // A-tile loads issued (TMA producer)

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      for (int g = 0; g < total; ++g) {
        const int s = g % kStages, r = g / kStages;
        const int kb = g % nk;
        int64_t m0, n0;
        tile_coords(p, pair + (g / nk) * p.npairs, m0, n0);
        if (r > 0 && !mbar_wait(empty_a(s), (r - 1) & 1, abort, p.dev_status)) break;
        a_issued = g + 1;
        if (nvfp4::kWithhold && blockIdx.x == 0 && g == 0) continue;  // test build: never issued
        if (rank == 0) {
          // rank 0's full_a(s) completes with both CTAs' A halves and rank 1's
          // token for its B half
          mbar_arrive_expect_tx(full_a(s), 2 * kABytes + 16);
          tma_load_2d(a_tile(s), &tmap_a, kb * BK, (int)m0, full_a(s));
        } else {
          tma_load_2d_to_rank0(a_tile(s), &tmap_a, kb * BK, (int)m0 + BM, mapa_rank0(full_a(s)));
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------------------------------------------------- MMA issuer
      bool ok = true;
      for (int it = 0; it < my_tiles && ok; ++it) {
        const int ab = it & 1;  // accumulator buffer; tiles alternate
        if (it >= 2 && !mbar_wait<true, true>(tmem_empty(ab), ((it >> 1) - 1) & 1, abort, p.dev_status))
          break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(ab * kAccCols);
        for (int kb = 0; kb < nk; ++kb) {
          const int g = it * nk + kb;
          const int s = g % kStages, r = g / kStages;
          ok = mbar_wait<false, true>(full_a(s), r & 1, abort, p.dev_status) &&
               mbar_wait<false, true>(full_b(s), r & 1, abort, p.dev_status);
          if (!ok) break;
          tc_fence_after();
          const uint64_t ad = smem_desc(a_tile(s));
          const uint64_t bd = smem_desc(base + b_tile(s));
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)  // advance 32 bytes (16 elements) along K
            mma_pair(d, ad + 2 * kk, bd + 2 * kk, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          mma_commit_pair(empty_a(s));  // both commits track the same MMAs, in both CTAs
          mma_commit_pair(empty_b(s));
        }
        if (ok) mma_commit_pair(tmem_full(ab));  // fires once the tile's MMAs have completed
      }
    } else if (lane == 0) {
      // ------------------------------------------- stage relay (rank 1): once
      // this CTA's B half of a stage is written, a 16-byte token copy tells
      // rank 0's full_a(s) (its A half goes there by its own TMA)
      const uint32_t token0 = mapa_rank0(token);
      for (int g = 0; g < total; ++g) {
        const int s = g % kStages, r = g / kStages;
        if (!mbar_wait<false, true>(full_b(s), r & 1, abort, p.dev_status)) break;
        bulk_token_to_rank0(token0, token, mapa_rank0(full_a(s)));
      }
    }
  } else if (warp < 2 + kDequantWarps) {
    // --------------------------------------------------------------- dequant
    const int d = threadIdx.x - 64;
    const int r = d >> 2, h = d & 3;  // B-tile row 0..127, K quarter (16 elements = one scale block)
    const bool row_used = r < half_n;
    const uint32_t swz = (uint32_t)(r & 7);
    uint2 qa[kPrefetch];
    uint32_t qs[kPrefetch];
    // load cursor over (tile, k step): row pointers change once per tile
    int lt = 0, lkb = 0;
    const uint8_t* wp = nullptr;
    const uint8_t* sp = nullptr;
    bool lvalid = false;
    auto set_tile = [&](int it) {
      int64_t m0, n0;
      tile_coords(p, pair + it * p.npairs, m0, n0);
      const int64_t nrow = n0 + (int64_t)rank * half_n + r;
      lvalid = row_used && nrow < p.n;
      wp = p.packed + (lvalid ? nrow : 0) * (p.k / 2) + 8 * h;
      sp = p.scales + (lvalid ? nrow : 0) * (p.k / 16) + h;
    };
    set_tile(0);
    auto issue = [&](int i) {
      if (lvalid) {  // rows past n: zero weights (their outputs are not stored)
        qa[i] = __ldg(reinterpret_cast<const uint2*>(wp + (int64_t)lkb * 32));
        qs[i] = __ldg(sp + 4 * lkb);
      } else {
        qa[i] = make_uint2(0, 0);
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
          const int s = g % kStages, rr = g / kStages;
          const uint2 c0 = qa[i];
          const uint32_t cs = qs[i];
          if (g + kPrefetch < total) issue(i);
          if (rr > 0 && !mbar_wait(empty_b(s), (rr - 1) & 1, abort, p.dev_status)) {
            ok = false;
          } else {
            if (row_used) {
              uint32_t S0, S1;
              if constexpr (F16)
                decode_scales_f16(cs, S0, S1);
              else
                decode_scales(cs, S0, S1);
              unsigned char* brow = smem + b_tile(s) + r * 128;
              uint4 v0, v1;  // chunks 2h, 2h+1: k = 16h .. 16h + 15
              if constexpr (F16) {
                v0 = dequant_word_f16(c0.x, S0);
                v1 = dequant_word_f16(c0.y, S0);
              } else {
                v0 = dequant_word(c0.x, S0);
                v1 = dequant_word(c0.y, S0);
              }
              *reinterpret_cast<uint4*>(brow + (((uint32_t)(2 * h) ^ swz) << 4)) = v0;
              *reinterpret_cast<uint4*>(brow + (((uint32_t)(2 * h + 1) ^ swz) << 4)) = v1;
              fence_proxy_async();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(full_b(s));
          }
        }
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue
    // warp quadrant q owns TMEM lanes 32q..32q+31 = rows 32q.. of this CTA's half
    const int q = warp & 3;
    // BF16 path: g * 2^8 (the dequant fold); FP16 path: g, and 2^-e per row
    const float gs = F16 ? __ldg(p.gscale) : __ldg(p.gscale) * 256.0f;
    for (int it = 0; it < my_tiles; ++it) {
      const int ab = it & 1;
      __syncwarp();
      if (!mbar_wait(tmem_full(ab), (it >> 1) & 1, abort, p.dev_status)) break;
      __syncwarp();
      tc_fence_after();
      int64_t m0, n0;
      tile_coords(p, pair + it * p.npairs, m0, n0);
      const int64_t row = m0 + (int64_t)rank * BM + 32 * q + lane;
      const float rs = (F16 && row < p.m) ? __ldg(p.row_inv + row) : 1.0f;
      const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(ab * kAccCols);
#pragma unroll 1
      for (int col = 0; col < p.bn; col += 32) {
        // columns [col, col + w) of the tile, w = 32 or a last 16; the stored
        // part stops at n (a multiple of 16)
        const int w = p.bn - col >= 32 ? 32 : 16;
        const int64_t nvalid = p.n - (n0 + col);
        const int ws = nvalid >= w ? w : (nvalid > 0 ? (int)nvalid : 0);
        uint32_t v[32];
        if (w == 32) {
          tmem_ld32(tbase + (uint32_t)col, v);
        } else {
          uint32_t v16[16];
          tmem_ld16(tbase + (uint32_t)col, v16);
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = v16[i];
        }
        if (row < p.m && ws > 0) {
          uint32_t packed16[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            __nv_bfloat162 b2 = __floats2bfloat162_rn((__uint_as_float(v[2 * i]) * rs) * gs,
                                                      (__uint_as_float(v[2 * i + 1]) * rs) * gs);
            packed16[i] = *reinterpret_cast<uint32_t*>(&b2);
          }
          uint4* dst = reinterpret_cast<uint4*>(p.c + row * p.ldc + n0 + col);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (8 * i < ws)
              dst[i] = make_uint4(packed16[4 * i], packed16[4 * i + 1], packed16[4 * i + 2],
                                  packed16[4 * i + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tmem_empty(ab), 0u);  // to rank 0's MMA issuer
    }
  }
  tc_fence_before();
  __syncthreads();
  if (*abort) {
    // A wait ran out somewhere in the CTA: the last A load on each stage and
    // the MMAs already issued may still be in flight.  Wait for them (bounded)
    // before TMEM is freed and the CTAs' shared memory released.
    // (rank 1's A halves and tokens complete on rank 0's barriers: rank 0's
    // drain covers them, and rank 1 stays until the cluster barrier below)
    if (warp == 0 && lane == 0 && rank == 0)
      for (int g = a_issued > kStages ? a_issued - kStages : 0; g < a_issued; ++g)
        mbar_drain(full_a(g % kStages), (uint32_t)(g / kStages) & 1u, p.dev_status);
  }
  if (warp == 1 && lane == 0) {
    // every MMA issued (they read both CTAs' shared memory) has completed, and
    // its arrivals on both CTAs' barriers have landed, before either CTA moves
    // on to free its memory: rank 0 commits to drain_bar in both CTAs after
    // its last MMA and both wait for that arrival
    if (rank == 0) mma_commit_pair(drain_bar);
    mbar_drain(drain_bar, 0u, p.dev_status);
  }
  tc_fence_before();
  cluster_sync();  // neither CTA exits while the pair's MMAs or arrivals may touch it
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
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

namespace {

// Co-resident clusters of two CTAs (the persistent grid's pairs) for the
// kernel on the current device; queried once per (device, path) and then
// served from a table, so calls made while a stream is captured into a CUDA
// graph issue no CUDA API calls here.
int max_pairs(const void* kern, bool f16) {
  static int cache[64][2] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int& slot = cache[dev][f16 ? 1 : 0];
  if (slot > 0) return slot;
  if (nvfp4::occupancy(kern, kThreads, kSmemBytes) < 1) return 0;  // also raises the smem limit
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess) return 0;
  slot = clusters;
  return clusters;
}

// Pair tile width: the multiple of 16 in [128, 256] that minimises the
// scheduled work, waves x (BN + 16) -- whole waves of tiles over the pairs,
// each tile's time taken as its width plus a fixed per-tile share.
int pick_bn(int mtiles, int64_t n, int pairs) {
  int best = kMaxBN;
  int64_t best_cost = -1;
  for (int bn = kMaxBN; bn >= 128; bn -= 16) {
    const int64_t tiles = (int64_t)mtiles * nvfp4::cdiv(n, bn);
    const int64_t cost = nvfp4::cdiv(tiles, pairs) * (bn + 16);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

}  // namespace

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
  auto kern = f16 ? gemm_tcgen05_kernel<true> : gemm_tcgen05_kernel<false>;
  const int pairs_max = max_pairs(reinterpret_cast<const void*>(kern), f16);
  if (pairs_max < 1) return NVFP4_ERR_CUDA;
  GemmParams p;
  p.packed = w->packed;
  p.scales = w->scales;
  p.gscale = w->global_scale;
  p.c = reinterpret_cast<__nv_bfloat16*>(c);
  p.m = m;
  p.n = w->n;
  p.k = w->k;
  p.ldc = ldc;
  p.mtiles = (int)nvfp4::cdiv(m, 2 * BM);
  p.bn = pick_bn(p.mtiles, w->n, pairs_max);
  p.ntiles = (int)nvfp4::cdiv(w->n, p.bn);
  p.row_inv = row_inv;
  p.dev_status = dev_status;
  const int64_t tiles = (int64_t)p.mtiles * p.ntiles;
  if (tiles > 0x7FFFFFFF) return NVFP4_ERR_SHAPE;
  p.npairs = (int)(tiles < pairs_max ? tiles : pairs_max);  // persistent: one pair per two SMs
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * p.npairs));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, tmap, p) != cudaSuccess) return NVFP4_ERR_CUDA;
  return NVFP4_OK;
}
