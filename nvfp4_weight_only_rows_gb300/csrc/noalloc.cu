// noalloc.cu -- w4a16_lm_head_noalloc: the W4A16 lm_head product for callers
// that cannot hand the library a workspace.
//
// Who needs this: runtimes that fix their whole device-memory budget when
// they start and forbid any later cudaMalloc (which can also synchronize the
// device and stall a serving loop), and plain C callers of this library that
// have no device allocator of their own to carve a workspace from.  This
// entry point keeps its scratch in one static device array of this file
// instead, so the caller passes only inputs and outputs.
//
// The array (NVFP4_NOALLOC_SCRATCH_BYTES, 8 MiB) lives in every GPU that
// loads the library until the process exits.  All calls share it: the
// kernels write every byte before they read it (the rescaled activations,
// the token multipliers, the split-K partials), the status word and the
// split-K counters are cleared at the start of each call, but two calls that
// overlap on the GPU (different streams, no ordering between them) race on it.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"

namespace nvfp4 {
size_t lm_head_workspace_bytes(int64_t M, int64_t N, int64_t K, bool argmax);

// The fixed scratch.  In host code `g_noalloc_scratch` is only a host-side
// stand-in for the symbol; its device address comes from
// cudaGetSymbolAddress (below), once per device.
static __device__ __align__(256) uint8_t g_noalloc_scratch[NVFP4_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
static std::mutex g_scratch_mu;
static void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up on
// the first call made with that device current, then cached).
static nvfp4_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return NVFP4_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return NVFP4_OK;
}

}  // namespace nvfp4

extern "C" nvfp4_status w4a16_lm_head_noalloc(const void* x, int64_t M, int64_t K,
                                              const uint8_t* packed, const uint8_t* scales,
                                              const float* global_scale, int64_t N,
                                              void* logits, int out_dtype, void* stream) {
  using namespace nvfp4;
  if (M < 0 || N < 0 || K < 16 || K % 16 != 0) return NVFP4_ERR_SHAPE;
  if (out_dtype != NVFP4_OUT_F32 && out_dtype != NVFP4_OUT_BF16) return NVFP4_ERR_DTYPE;
  if (M == 0 || N == 0) return NVFP4_OK;
  // M * K decides the scratch: reject what the fixed array cannot hold
  if (lm_head_workspace_bytes(M, N, K, false) > NVFP4_NOALLOC_SCRATCH_BYTES)
    return NVFP4_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  nvfp4_status st = scratch_for_current_device(&scratch);
  if (st != NVFP4_OK) return st;
  // the usual entry point does the remaining checks and the launches
  return w4a16_lm_head(x, M, K, packed, scales, global_scale, N, logits, out_dtype, scratch,
                       NVFP4_NOALLOC_SCRATCH_BYTES, stream);
}
