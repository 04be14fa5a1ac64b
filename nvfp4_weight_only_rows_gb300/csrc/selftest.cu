// selftest.cu -- nvfp4_selftest_bounded_wait: check, on the device, that the
// library's pipeline waits give up instead of hanging; nvfp4_selftest_topk_bins:
// check, on the host, the fused top-k's histogram bins against the order keys.
//
// The kernel waits on an mbarrier phase that nothing completes, with the same
// bounded wait (mbar_wait) every kernel of this library uses, and then on a
// global flag that nothing sets.  Both waits must run out after the given
// limit, raise NVFP4_ERR_TIMEOUT in the workspace status word and return, so
// the CUDA context stays usable.  No fault, trap or unbounded loop is involved.
#include <cuda_runtime.h>

#include "common.cuh"
#include "gemm_common.cuh"

namespace nvfp4 {

__global__ void nvfp4_wait_selftest_kernel(int32_t* status, const uint32_t* never_set,
                                           uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int32_t abort_flag;
  if (threadIdx.x == 0) {
    *status = NVFP4_OK;
    mbar_init(&bar, 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  WaitCtl wc{status, &abort_flag, limit_ns};
  // 1) phase 0 of a fresh barrier with one expected arrival that never comes
  const bool done = mbar_wait(&bar, 0, wc);
  // 2) a global flag nobody writes (a fresh limit: the abort flag is cleared)
  __syncthreads();
  if (threadIdx.x == 0) abort_flag = 0;
  __syncthreads();
  bool seen = false;
  const uint64_t t0 = globaltimer_ns();
  while (!seen && globaltimer_ns() - t0 <= limit_ns) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(never_set) : "memory");
    seen = v != 0;
  }
  if (!seen) raise_status(status, NVFP4_ERR_TIMEOUT);
  (void)done;
}

}  // namespace nvfp4

extern "C" nvfp4_status nvfp4_selftest_bounded_wait(void* workspace, size_t workspace_bytes,
                                                    int64_t limit_us, void* stream) {
  using namespace nvfp4;
  if (!workspace) return NVFP4_ERR_NULL;
  if (workspace_bytes < kWsHeader) return NVFP4_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return NVFP4_ERR_ALIGN;
  if (limit_us <= 0 || limit_us > 10000000) return NVFP4_ERR_SHAPE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* status = reinterpret_cast<int32_t*>(ws);
  uint32_t* flag = reinterpret_cast<uint32_t*>(ws + 128);  // inside the header, never set
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(flag, 0, sizeof(uint32_t), s) != cudaSuccess) return NVFP4_ERR_CUDA;
  nvfp4_wait_selftest_kernel<<<1, 32, 0, s>>>(status, flag, (uint64_t)limit_us * 1000ull);
  if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
  return NVFP4_OK;
}

// Every 32-bit order key, in increasing order: its histogram bin never
// decreases, and the lower edge of its bin (the threshold a raise to that
// bin sets) never exceeds it; each bin's edge lies in the bin itself, and
// the edges increase with the bin.  The first key that breaks a rule is
// returned, -1 when none does.
extern "C" int64_t nvfp4_selftest_topk_bins(void) {
  using namespace nvfp4;
  uint32_t prev = 0, edge_hi = 0;
  for (uint64_t k = 0; k <= 0xFFFFFFFFull; ++k) {
    const uint32_t ok = (uint32_t)k;
    const uint32_t b = topk_bin(ok);
    if (b < prev || b >= (uint32_t)kHistBins) return (int64_t)ok;
    if (b != prev || k == 0) edge_hi = (uint32_t)(topk_edge(b) >> 32);
    if (edge_hi > ok) return (int64_t)ok;
    prev = b;
  }
  for (uint32_t b = 1; b < (uint32_t)kHistBins; ++b) {
    const uint32_t e = (uint32_t)(topk_edge(b) >> 32);
    if (topk_bin(e) != b || topk_edge(b) <= topk_edge(b - 1)) return (int64_t)e;
  }
  return -1;
}
