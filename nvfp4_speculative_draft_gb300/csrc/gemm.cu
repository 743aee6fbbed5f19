// gemm.cu -- prefill W4A16 GEMM, C = bf16(g * A . w~^T), w~ = e4m3(s) * e2m1(c).
//
// First correct version on CUDA cores (64x64 output tiles, FP32 FMA over the
// exactly dequantised weights); the tensor-core (tcgen05/TMEM) kernel replaces
// it.  Numerics follow the lossless FP4->BF16 dequant + BF16 product of the
// M=128 prefill dispatch in "spark_model/layers/qwen3_attention/prefill_weights.rs".
#include <cuda_fp8.h>

#include "common.cuh"

namespace {

constexpr int BM = 64, BN = 64, BK = 32;

__device__ __forceinline__ float e2m1_val(uint32_t c) {
  const float mag[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
  const float v = mag[c & 7];
  return (c & 8) ? -v : v;
}

__global__ void __launch_bounds__(256)
gemm_simt_kernel(const __nv_bfloat16* __restrict__ A, int64_t M, int64_t lda,
                 const uint8_t* __restrict__ packed, const uint8_t* __restrict__ scales,
                 const float* __restrict__ gscale, int64_t N, int64_t K,
                 __nv_bfloat16* __restrict__ C, int64_t ldc) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int64_t m0 = (int64_t)blockIdx.y * BM, n0 = (int64_t)blockIdx.x * BN;
  float acc[4][4] = {};
  for (int64_t k0 = 0; k0 < K; k0 += BK) {
    for (int e = threadIdx.x; e < BM * BK; e += 256) {
      const int r = e / BK, kk = e % BK;
      const int64_t gm = m0 + r;
      As[kk][r] = gm < M ? __bfloat162float(A[gm * lda + k0 + kk]) : 0.f;
    }
    for (int e = threadIdx.x; e < BN * BK; e += 256) {
      const int r = e / BK, kk = e % BK;
      const int64_t gn = n0 + r, gk = k0 + kk;
      const uint32_t byte = packed[gn * (K / 2) + gk / 2];
      const uint32_t code = (gk & 1) ? (byte >> 4) : (byte & 15u);
      const __half_raw sh =
          __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)scales[gn * (K / 16) + gk / 16], __NV_E4M3);
      Bs[kk][r] = e2m1_val(code) * __half2float(__half(sh));
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  const float g = *gscale;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t gm = m0 + ty * 4 + i;
    if (gm >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) C[gm * ldc + n0 + tx * 4 + j] = __float2bfloat16_rn(acc[i][j] * g);
  }
}

}  // namespace

int launch_gemm(const void* a, int64_t m, int64_t lda, const nvfp4_weight* w, void* c,
                int64_t ldc, int32_t* dev_status, cudaStream_t stream) {
  (void)dev_status;
  dim3 grid((unsigned)(w->n / BN), (unsigned)nvfp4::cdiv(m, BM));
  gemm_simt_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<const __nv_bfloat16*>(a), m, lda,
                                             w->packed, w->scales, w->global_scale, w->n, w->k,
                                             reinterpret_cast<__nv_bfloat16*>(c), ldc);
  if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
  return NVFP4_OK;
}
