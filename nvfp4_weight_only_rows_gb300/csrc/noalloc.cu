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
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "common.cuh"

namespace nvfp4 {
size_t lm_head_workspace_bytes(int64_t M, int64_t N, int64_t K, bool argmax);

// The fixed scratch.  In host code `g_noalloc_scratch` is only a host-side
// stand-in for the symbol; its device address comes from
// cudaGetSymbolAddress (below), once per CUDA context.
static __device__ __align__(256) uint8_t g_noalloc_scratch[NVFP4_NOALLOC_SCRATCH_BYTES];

// The symbol has one address per CUDA context (each context loads its own
// copy of the module), so the cache is keyed by the context current at the
// call: the primary context of each device, or one the caller made current.
// Lookups read the published entries without a lock; only a first lookup in
// a new context takes the mutex and appends an entry.
constexpr int kMaxContexts = 64;
struct ScratchEntry {
  std::atomic<CUcontext> ctx{nullptr};
  void* ptr = nullptr;
};
static ScratchEntry g_entries[kMaxContexts];
static std::atomic<int> g_n_entries{0};
static std::mutex g_scratch_mu;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

static CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Device address of the scratch array in the current context.  With no
// context current yet (a first CUDA call of the thread), the symbol lookup
// makes the device's primary context current, and the context is read after.
static nvfp4_status scratch_for_current_context(void** out) {
  CtxGetCurrentFn get = ctx_get_current();
  CUcontext ctx = nullptr;
  if (!get || get(&ctx) != CUDA_SUCCESS) return NVFP4_ERR_CUDA;
  if (!ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p ||
        get(&ctx) != CUDA_SUCCESS || !ctx)
      return NVFP4_ERR_CUDA;
  }
  const int n = g_n_entries.load(std::memory_order_acquire);
  for (int i = 0; i < n; ++i)
    if (g_entries[i].ctx.load(std::memory_order_acquire) == ctx) {
      *out = g_entries[i].ptr;
      return NVFP4_OK;
    }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  const int m = g_n_entries.load(std::memory_order_relaxed);
  for (int i = 0; i < m; ++i)
    if (g_entries[i].ctx.load(std::memory_order_relaxed) == ctx) {
      *out = g_entries[i].ptr;
      return NVFP4_OK;
    }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return NVFP4_ERR_CUDA;
  if (m < kMaxContexts) {  // publish: the pointer first, then the context, then the count
    g_entries[m].ptr = p;
    g_entries[m].ctx.store(ctx, std::memory_order_release);
    g_n_entries.store(m + 1, std::memory_order_release);
  }
  *out = p;
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
  // M * K (and, for K % 256 != 0, the staged weight rows) decide the
  // scratch: reject what the fixed array cannot hold
  if (lm_head_workspace_bytes(M, N, K, false) > NVFP4_NOALLOC_SCRATCH_BYTES)
    return NVFP4_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  nvfp4_status st = scratch_for_current_context(&scratch);
  if (st != NVFP4_OK) return st;
  // the usual entry point does the remaining checks and the launches
  return w4a16_lm_head(x, M, K, packed, scales, global_scale, N, logits, out_dtype, scratch,
                       NVFP4_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" nvfp4_status w4a16_lm_head_noalloc_status(int32_t* status_out, void* stream) {
  using namespace nvfp4;
  if (!status_out) return NVFP4_ERR_NULL;
  void* scratch = nullptr;
  nvfp4_status st = scratch_for_current_context(&scratch);
  if (st != NVFP4_OK) return st;
  // the status word is the first word of the scratch, as of any workspace
  return nvfp4_read_device_status(scratch, status_out, stream);
}
