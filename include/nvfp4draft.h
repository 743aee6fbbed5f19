/*
 * nvfp4draft.h -- C ABI of the GB300 (sm_103a) NVFP4 weight-only projection
 * library for a speculative-decoding draft head.
 *
 * NVFP4 weight format used throughout:
 *   packed  uint8 [n, k/2]  two E2M1 codes per byte; element 2j of a row in the
 *                           low nibble of byte j, element 2j+1 in the high one.
 *                           (The [N, K/2] layout is the one the prefill setup of
 *                           "spark_model/layers/qwen3_attention/prefill_weights.rs"
 *                           feeds its predequant kernel; 0.5 byte per weight as
 *                           the LM-head size log in "spark_model/layers/mtp_head/new.rs",
 *                           MtpHead::new, counts it.)
 *   scales  uint8 [n, k/16] one E4M3 scale per 16-element block along k, row-major.
 *   global  float           g = absmax(W) / (6 * 448).
 *   Dequantised weight: w[n][i] = g * e4m3(scales[n][i/16]) * e2m1(code[n][i]).
 *
 * Conventions shared by every call:
 *   - All pointers except those documented as host pointers are DEVICE
 *     pointers owned by the caller; the library allocates no memory and never
 *     synchronises: work is enqueued on ex->stream (a cudaStream_t; NULL =
 *     legacy default stream) and the call returns.  Its only state is caches
 *     (per-device SM count, per-kernel occupancy, the tensor-map encoder
 *     entry point) and the 256-byte scratch of w4a16_gemv_argmax_noalloc.
 *   - Arguments are checked on the host before anything is enqueued; a
 *     non-zero status means nothing was launched.  NVFP4_ERR_CUDA means a
 *     launch failed after validation (the CUDA error is left for the caller's
 *     cudaGetLastError).
 *   - ex->dev_status (nullable, device int32) receives conditions detected on
 *     the device (non-finite input to the quantiser, a bounded wait that gave
 *     up).  The library only ever writes non-zero codes there; the caller
 *     clears it.
 *   - Concurrent calls on different streams need distinct workspaces.
 *   - Weights are load-time constants.  The GEMV calls may read the quantised
 *     weight (codes, scales, global scale) and the segments' gamma while the
 *     previous kernel on the stream is still finishing (programmatic dependent
 *     launch: the next call's weight stream starts before this one ends);
 *     activations and gather indices are read only after it completed.  So
 *     the weight and gamma must not be written by the kernel that immediately
 *     precedes the call on the stream -- unless that kernel is
 *     nvfp4_quantize / fp8w_quantize, which make their output visible before
 *     releasing dependents.  Copies (cudaMemcpy*) and any other stream
 *     operation in between are fine.
 *   - No C++ exception crosses this interface.
 */
#ifndef NVFP4DRAFT_H
#define NVFP4DRAFT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define NVFP4_OK 0
#define NVFP4_ERR_NULL 1       /* a required pointer is NULL                 */
#define NVFP4_ERR_SHAPE 2      /* a size is out of range or not a multiple   */
#define NVFP4_ERR_ALIGN 3      /* a pointer or leading dimension misaligned  */
#define NVFP4_ERR_WORKSPACE 4  /* workspace missing, too small or misaligned */
#define NVFP4_ERR_CUDA 5       /* a kernel launch failed                     */
#define NVFP4_ERR_TIMEOUT 6    /* device: a bounded wait gave up; the call's
                                  outputs are not valid (a GEMV still returns
                                  its argmax workspace to zero)             */
#define NVFP4_ERR_NONFINITE 7  /* device: Inf/NaN in the quantiser's input   */
#define NVFP4_ERR_DTYPE 8      /* unknown output dtype                       */
#define NVFP4_ERR_INDEX 9      /* device: a gather index out of range; row 0 */

/* Output element types. */
#define NVFP4_DTYPE_F32 0
#define NVFP4_DTYPE_BF16 1

/* Largest activation batch of the GEMV calls (the pages' batch-16 and
 * batch-32 draft widths).  One launch takes up to 16 rows: one MMA column per
 * row, in groups of 8 columns that share each dequantised weight fragment;
 * wider batches, and batches whose activations exceed one CTA's shared memory
 * at large k, run as consecutive launches of row blocks on the caller's
 * stream (each streams the weights once). */
#define W4A16_GEMV_MAX_M 32
/* Largest total K of the GEMV calls (activations are staged on chip: the
 * FP16 activation fragments take 2 m k bytes of one CTA's shared memory next
 * to the weight ring; a batch whose fragments do not fit runs as row blocks of
 * 8, 4, ... rows, so every m <= W4A16_GEMV_MAX_M runs at every k up to this). */
#define W4A16_GEMV_MAX_K 16384
/* Workspace of w4a16_gemv_argmax: 16 64-bit keys (one launch's rows) + a
 * counter.  Zero it once when allocated; every completed call leaves it
 * zeroed. */
#define W4A16_ARGMAX_WS_BYTES 256
/* Most CTAs a GEMV launch uses, and the workspace of w4a16_gemv_argmax_ex
 * (keys + counter, then one (max, sum) pair per CTA and batch row). */
#define W4A16_GEMV_MAX_CTAS 1024
#define W4A16_ARGMAX_EX_WS_BYTES (W4A16_ARGMAX_WS_BYTES + W4A16_GEMV_MAX_CTAS * W4A16_GEMV_MAX_M * 8)
/* Optional larger GEMV workspace: with at least W4A16_GEMV_WS_BYTES(m, k)
 * bytes (16-byte aligned) and m >= 2, the GEMV calls normalise the
 * activations once in a small grid of their own (one CTA per batch row) and
 * every GEMV CTA copies the result, instead of each CTA normalising all rows
 * itself (both match the reference within the GEMV tolerance; the norm's
 * sum of squares may add its partials in another order).  Layout: the
 * argmax / log-prob area above, then the per-row scale carriers at
 * W4A16_GEMV_PREP_OFFSET and the FP16 fragments 256 bytes further on. */
#define W4A16_GEMV_PREP_OFFSET W4A16_ARGMAX_EX_WS_BYTES
#define W4A16_GEMV_WS_BYTES(m, k)                                                \
  ((size_t)W4A16_GEMV_PREP_OFFSET + 256 +                                        \
   ((size_t)(k) + 255) / 256 * 512 * (size_t)((m) <= 8 ? (m) : W4A16_GEMV_MAX_M))
/* Workspace of nvfp4_quantize when its absmax output is NULL. */
#define NVFP4_QUANTIZE_WS_BYTES 16
/* Optional workspace of w4a16_gemm that enables its FP16 staging path. */
#define W4A16_GEMM_WS_BYTES(m, k) ((size_t)(m) * (size_t)(k) * 2 + (size_t)(m) * 4 + 256)

/* A quantised weight (all device pointers, 16-byte aligned). */
typedef struct nvfp4_weight {
    const uint8_t *packed;       /* [n, k/2] E2M1 codes                */
    const uint8_t *scales;       /* [n, k/16] E4M3 block scales        */
    const float *global_scale;   /* 1 float: g                         */
    int64_t n;                   /* output features (rows)             */
    int64_t k;                   /* input features, multiple of 32     */
} nvfp4_weight;

/* One activation segment of the GEMV input.  The GEMV input row m is the
 * concatenation, in argument order, of every segment's row m, each optionally
 * RMS-normalised first:
 *     a = bf16( x * (1 / sqrt(mean(x^2) + eps)) * gamma )     (gamma != NULL)
 *     a = x                                                   (gamma == NULL)
 * with gamma applied as stored (the "vanilla" RMSNorm of the draft head in
 * "spark_model/layers/deepseek_v4_mtp.rs", constructor) and the embedding
 * segment first for the fc combiner (pre-fc norms, concat, fc, as the module
 * doc of "metrale_model_layers/layers/mtp_head.rs" orders the draft step). */
typedef struct w4a16_act_segment {
    const void *x;      /* BF16 [m, k_seg], row stride ld elements, 16-B aligned */
    int64_t k_seg;      /* multiple of 32                                         */
    int64_t ld;         /* row stride in elements, multiple of 8, >= k_seg        */
    const void *gamma;  /* BF16 [k_seg], 16-B aligned, or NULL for no norm        */
    float eps;
    /* Optional gather (embed_from_argmax of "metrale_model_layers/layers/
     * mtp_head.rs", fused into the activation load): with row_index != NULL,
     * x is a table of index_rows rows and row r of the segment is table row
     * row_index[r] -- e.g. the embedding of the token the previous
     * w4a16_gemv_argmax call wrote to its device argmax buffer, read after
     * that call completes (stream order), with no host round trip.  An index
     * outside [0, index_rows) reads row 0 and records NVFP4_ERR_INDEX. */
    const int32_t *row_index;  /* device int32 [m], 4-B aligned, or NULL      */
    int64_t index_rows;        /* rows of the table when row_index != NULL   */
} w4a16_act_segment;

/* An FP8 weight (the pages' second projection precision, see fp8w_quantize):
 * E4M3 codes [n, k] row-major, 16-byte aligned; one FP32 scale per row. */
typedef struct fp8w_weight {
    const uint8_t *codes;
    const float *row_scale;  /* device [n], 4-byte aligned */
    int64_t n, k;            /* k a multiple of 32; n * k < 2^32 */
} fp8w_weight;

/* Execution context. */
typedef struct nvfp4_exec {
    void *stream;           /* cudaStream_t                                  */
    void *workspace;        /* device, 16-byte aligned, see each call        */
    size_t workspace_bytes;
    int32_t *dev_status;    /* nullable device int32, see above              */
} nvfp4_exec;

/*
 * nvfp4_quantize -- load-time BF16 -> NVFP4 quantisation of w[n, k].
 * The two passes of the load path in "spark_model/layers/mtp_head/new.rs"
 * (MtpHead::new: the global-absmax kernel, then the BF16->NVFP4 kernel):
 *   amax = max |w|;  g = fl32(amax / 2688)
 *   per 16-block b of a row: s_b = E4M3_rne_satfinite(fl32(amax_b / fl32(6 g)))
 *                            (s_b = 0 when g == 0 or amax_b == 0)
 *   per element: d = fl32(e4m3(s_b) * g);
 *                code = d == 0 ? +0 : E2M1_rne_satfinite(fl32(x / d)) with the
 *                sign bit of x.
 *   w_bf16       device BF16 [n, k] row-major, 16-byte aligned.
 *   n >= 1, k >= 32, k % 32 == 0.
 *   packed       device uint8 [n, k/2] (16-byte aligned), written.
 *   scales       device uint8 [n, k/16], written.
 *   global_scale device float, written with g.
 *   absmax       device float or NULL; written with amax.  When NULL the
 *                workspace must hold NVFP4_QUANTIZE_WS_BYTES.
 * Non-finite input: results undefined, NVFP4_ERR_NONFINITE to dev_status.
 */
int nvfp4_quantize(const void *w_bf16, int64_t n, int64_t k, uint8_t *packed,
                   uint8_t *scales, float *global_scale, float *absmax,
                   const nvfp4_exec *ex);

/*
 * w4a16_gemv -- batched W4A16 GEMV, y[m, n] = g * sum_i a[m, i] * w~[n, i],
 * where w~ = e4m3(s) * e2m1(c) is exact in BF16 and the sum is accumulated in
 * FP32; the global scale multiplies the finished sum.  This is the NVFP4 arm
 * of the per-precision one-row GEMV of "metrale_model_layers/layers/mtp_head.rs"
 * (MtpHead::gemv -> w4a16_decode_gemv), batched to m <= 16 rows and with the
 * draft head's RMSNorm + concat fused into the activation load.
 *   seg, nseg     host array of 1 or 2 segments; sum of k_seg == w->k.
 *   m             1..W4A16_GEMV_MAX_M activation rows.
 *   w             host struct describing the weight; w->k <= W4A16_GEMV_MAX_K.
 *   y             device [m, ldy] of y_dtype (F32 or BF16, round-to-nearest-even),
 *                 ldy >= w->n.
 * Workspace: none required; with W4A16_GEMV_WS_BYTES(m, w->k) bytes the
 * activations are prepared once for all CTAs (both ways are within the GEMV
 * tolerance of the exact result; they may differ from each other in the last
 * bits, see W4A16_GEMV_WS_BYTES).
 */
int w4a16_gemv(const w4a16_act_segment *seg, int nseg, int m, const nvfp4_weight *w,
               void *y, int y_dtype, int64_t ldy, const nvfp4_exec *ex);

/*
 * w4a16_gemv_argmax -- the same GEMV with greedy argmax fused on the output:
 * argmax[r] = the lowest index n with y[r, n] maximal over the FP32 logits,
 * the scan of "spark_model/layers/deepseek_v4_mtp.rs" (argmax_grammar_masked:
 * strict '>' ascending from -inf, so NaN never wins and 0 comes back when no
 * logit exceeds -inf), applied to the reduced-vocab LM head's rows.
 *   logits        device float [m, ld_logits] or NULL (not written).
 *   argmax        device int32 [m].
 * Workspace: W4A16_ARGMAX_WS_BYTES, 16-byte aligned, zeroed once by the caller
 * when allocated; each completed call returns it to zero.
 */
int w4a16_gemv_argmax(const w4a16_act_segment *seg, int nseg, int m,
                      const nvfp4_weight *w, float *logits, int64_t ld_logits,
                      int32_t *argmax, const nvfp4_exec *ex);

/*
 * w4a16_gemv_argmax_ex -- w4a16_gemv_argmax with the two outputs the draft
 * loop asks of the LM head besides the token id:
 *   mask      device int32 [m, ld_mask] or NULL: grammar bitmask, bit n%32 of
 *             word n/32 of row r allows token n for batch row r (ld_mask >=
 *             ceil(n/32)).  A disallowed token never wins; a row with no
 *             allowed token returns index 0 -- the masked scan of
 *             argmax_grammar_masked in "spark_model/layers/deepseek_v4_mtp.rs",
 *             fused into the GEMV instead of run on the host.  Logits are
 *             written unmasked.
 *   logprob   device float [m] or NULL: top-1 log-probability of the chosen
 *             token, y[argmax] - log(sum exp(y)) over the allowed tokens; NaN
 *             when no token is allowed.  It is what the batched
 *             argmax_bf16_batch_lp kernel of "metrale_model_layers/layers/
 *             mtp_head.rs" (MtpHead fields) writes per row, and what the draft
 *             confidence stop there reads (last_conf_bits).  FP32 exp/log; the
 *             per-CTA partials are combined in a fixed order.
 * Workspace: W4A16_ARGMAX_EX_WS_BYTES, 16-byte aligned, its first
 * W4A16_ARGMAX_WS_BYTES zeroed once when allocated (each completed call
 * returns them to zero); the rest is scratch that every call overwrites.
 */
int w4a16_gemv_argmax_ex(const w4a16_act_segment *seg, int nseg, int m, const nvfp4_weight *w,
                         float *logits, int64_t ld_logits, int32_t *argmax, float *logprob,
                         const int32_t *mask, int64_t ld_mask, const nvfp4_exec *ex);

/*
 * w4a16_gemv_argmax_noalloc -- w4a16_gemv_argmax for callers that cannot
 * allocate device memory.  The pages have no counterpart of this call.
 * Some callers cannot call cudaMalloc at call time: a serving loop running
 * under a fixed device-memory budget handed out up front, a host framework
 * whose allocator forbids side allocations, or code that must not hit the
 * implicit device synchronisation of cudaMalloc/cudaFree in the decode path.
 * This variant takes no workspace: its argmax scratch (W4A16_GEMV_MAX_M keys
 * and a counter) is a fixed 256-byte __device__ array inside the library,
 * which every GPU that loads the library keeps until the process exits.
 *   Arguments as w4a16_gemv_argmax, except: no nvfp4_exec; stream is a
 *   cudaStream_t (NULL = legacy default stream); dev_status is nullable.
 *   m > W4A16_GEMV_MAX_M (beyond the scratch) -> NVFP4_ERR_SHAPE.
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  Under
 * lazy module loading (the CUDA default) that first call may also load the
 * library's device code, which allocates device memory and may synchronise:
 * a caller with a fixed memory budget makes one call at start-up, before the
 * budget is handed out.  The stream must belong to the current device
 * (otherwise NVFP4_ERR_CUDA, nothing launched).  Each call clears the scratch
 * on its stream first.  All calls share the array, so calls that overlap on
 * the GPU (other streams, other host threads) race.  After that first call it
 * allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 */
int w4a16_gemv_argmax_noalloc(const w4a16_act_segment *seg, int nseg, int m,
                              const nvfp4_weight *w, float *logits, int64_t ld_logits,
                              int32_t *argmax, void *stream, int32_t *dev_status);

/*
 * w4a16_gemm -- prefill W4A16 GEMM, C[m, n] = bf16( g * A[m, :] . w~[n, :] ),
 * w~ dequantised exactly to BF16 and multiplied with BF16 tensor-core MMAs
 * accumulating in FP32, in 128-row tiles of A.  This is the lossless
 * "FP4->BF16 dequant + BF16 MMA" numerics of the M=128 prefill GEMM dispatch in
 * "spark_model/layers/qwen3_attention/prefill_weights.rs"
 * (w4a16_gemm_m128_dispatch, BF16 tensor-core variant).
 *   a_bf16   device BF16 [m, lda], 16-byte aligned, lda % 8 == 0, lda >= k.
 *   m >= 1 (any; the last tile is masked); w->n % 128 == 0; w->k % 64 == 0.
 *   c_bf16   device BF16 [m, ldc], 16-byte aligned, ldc % 8 == 0, ldc >= n.
 *   w->scales 4-byte aligned.
 * Workspace (optional): with at least W4A16_GEMM_WS_BYTES(m, k) bytes (16-byte
 * aligned) the activations are first staged there as FP16, each row times an
 * exact power of two that puts its largest magnitude in [2^14, 2^15) (exact
 * for every activation within 2^-31 of the row maximum; smaller ones round at
 * that level), and the weights are dequantised to FP16 with the hardware E2M1
 * conversion for an FP16 x FP16 -> FP32 MMA; the row scale is removed from the
 * FP32 sum.  Without it, the BF16 operands go to a BF16 MMA directly.  Both
 * paths multiply exact weight values; they differ only in how activations far
 * below their row's maximum are rounded.
 * Waits inside the kernel are bounded; one that runs out writes
 * NVFP4_ERR_TIMEOUT to ex->dev_status and leaves C incomplete.
 */
int w4a16_gemm(const void *a_bf16, int64_t m, int64_t lda, const nvfp4_weight *w,
               void *c_bf16, int64_t ldc, const nvfp4_exec *ex);

/*
 * FP8 weight variant of the GEMV path: MtpHead::new in
 * "spark_model/layers/mtp_head/new.rs" resolves gemv_fp8w's
 * quantize_bf16_to_fp8 beside the NVFP4 pair, and its MtpQuantization::Fp8
 * arm resolves dense_gemv_fp8w; the pages print no formula.  Plainest reading
 * of a single quantise kernel (no separate global-absmax pass): one binary32
 * scale per output row,
 *     s_n = fl32(amax_n / 448),   c = E4M3_RNE_SATFINITE(fl32(x / s_n))
 * (sign of x, all codes +0 when s_n == 0), and
 *     y[m, n] = s_n * sum_i a[m, i] * e4m3(c[n, i])   (FP32 accumulation).
 *
 * fp8w_quantize -- BF16 w [n, k] (16-B aligned, k % 32 == 0) -> codes [n, k]
 *   (16-B aligned) and row_scale [n].  One warp per row.  Non-finite input:
 *   results undefined, NVFP4_ERR_NONFINITE to dev_status.  No workspace.
 * fp8w_gemv, fp8w_gemv_argmax -- the same contracts (segments, RMSNorm +
 *   concat + gather, outputs, argmax ties, workspaces) as w4a16_gemv and
 *   w4a16_gemv_argmax, with the FP8 weight.
 */
int fp8w_quantize(const void *w_bf16, int64_t n, int64_t k, uint8_t *codes, float *row_scale,
                  const nvfp4_exec *ex);
int fp8w_gemv(const w4a16_act_segment *seg, int nseg, int m, const fp8w_weight *w, void *y,
              int y_dtype, int64_t ldy, const nvfp4_exec *ex);
int fp8w_gemv_argmax(const w4a16_act_segment *seg, int nseg, int m, const fp8w_weight *w,
                     float *logits, int64_t ld_logits, int32_t *argmax, const nvfp4_exec *ex);
/* fp8w_gemv_argmax_ex -- w4a16_gemv_argmax_ex (grammar mask, top-1
 * log-probability) with the FP8 weight. */
int fp8w_gemv_argmax_ex(const w4a16_act_segment *seg, int nseg, int m, const fp8w_weight *w,
                        float *logits, int64_t ld_logits, int32_t *argmax, float *logprob,
                        const int32_t *mask, int64_t ld_mask, const nvfp4_exec *ex);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4DRAFT_H */
