// noalloc.cu -- w4a16_gemv_argmax_noalloc: the fused GEMV + argmax without a
// caller-provided workspace, for callers that cannot allocate device memory.
//
// The argmax pass needs a few bytes of device scratch (one 64-bit key per
// batch row and a completion counter).  w4a16_gemv_argmax takes them from the
// caller's workspace; this variant keeps them in a file-scope __device__ array
// instead, so nothing is allocated at call time.  Every GPU that loads this
// library holds the array (kNoallocScratchBytes) until the process exits.
//
// Host code cannot use the array's name as a device address: on the host the
// symbol is only a stand-in.  The device address is obtained once per device
// with cudaGetSymbolAddress, with that device current, on the first call made
// on it; the first call on each device should therefore come before any stream
// capture.  Under lazy module loading (the CUDA default) that first call may
// also load the library's device code, which allocates device memory and may
// synchronise: a caller with a fixed memory budget makes one call at start-up.
// The stream must belong to the current device.  Each call clears the keys and
// counter on its stream before the
// kernel runs.  All calls share the one array: calls that overlap on the GPU
// (concurrent streams, or several host threads) race on it.
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kNoallocScratchBytes = 256;  // >= W4A16_ARGMAX_WS_BYTES
static_assert(kNoallocScratchBytes >= W4A16_ARGMAX_WS_BYTES, "argmax scratch too small");

static __device__ __align__(256) unsigned char g_argmax_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (set up once),
// which must also be the device of `stream`: the scratch of one device is
// not the scratch of another.
int scratch_for_current_device(cudaStream_t stream, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_CUDA;
  if (stream != nullptr) {
    int sdev = -1;
    if (cudaStreamGetDevice(stream, &sdev) != cudaSuccess || sdev != dev) return NVFP4_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_argmax_scratch) != cudaSuccess || ptr == nullptr)
      return NVFP4_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return NVFP4_OK;
}

}  // namespace

extern "C" int w4a16_gemv_argmax_noalloc(const w4a16_act_segment* seg, int nseg, int m,
                                         const nvfp4_weight* w, float* logits, int64_t ld_logits,
                                         int32_t* argmax, void* stream, int32_t* dev_status) {
  int rc = nvfp4::check_weight(w);
  if (rc) return rc;
  // m beyond W4A16_GEMV_MAX_M is rejected here; a launch takes at most 16 rows, one key each
  rc = nvfp4::check_segments(seg, nseg, m, w->k);
  if (rc) return rc;
  if (argmax == nullptr) return NVFP4_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(argmax) & 3u) ||
      (logits != nullptr && (reinterpret_cast<uintptr_t>(logits) & 3u)))
    return NVFP4_ERR_ALIGN;
  if (logits != nullptr && ld_logits < w->n) return NVFP4_ERR_SHAPE;
  if (w->n > 0x7FFFFFFFLL) return NVFP4_ERR_SHAPE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  void* scratch = nullptr;
  rc = scratch_for_current_device(st, &scratch);
  if (rc) return rc;
  if (cudaMemsetAsync(scratch, 0, W4A16_ARGMAX_WS_BYTES, st) != cudaSuccess) return NVFP4_ERR_CUDA;
  return launch_gemv(seg, nseg, m, ref_of(w), logits, NVFP4_DTYPE_F32, ld_logits, true, argmax, scratch,
                     W4A16_ARGMAX_WS_BYTES, dev_status, st);
}
