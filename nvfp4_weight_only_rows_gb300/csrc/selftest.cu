// selftest.cu -- nvfp4_selftest_bounded_wait: check, on the device, that the
// library's pipeline waits give up instead of hanging; nvfp4_selftest_topk_bins:
// check, on the host, the fused top-k's histogram bins against the order keys;
// nvfp4_selftest_schedule: check, on the host, the persistent GEMM's split of
// its units into whole-unit waves and a (skewed) stream-K tail.
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

// The persistent schedule's host split (schedule_units) over a spread of
// unit counts, grids, stages per unit and skew bounds: the whole-unit waves
// and the tail cover every stage once; the tail ranges are contiguous, each
// at least one unit long, so that a unit is cut at most once (the pairwise
// partial combine relies on it); an unskewed split is the even one.
// Returns -1 when every case passes, else the index of the first failing
// case.
extern "C" int64_t nvfp4_selftest_schedule(void) {
  using namespace nvfp4;
  const int64_t units[] = {1, 2, 3, 7, 31, 100, 151, 152, 153, 303, 304, 305, 457, 1002, 1003,
                           2004, 4096, 16032};
  const int64_t grids[] = {1, 2, 7, 76, 148, 152};
  const int n_kbs[] = {1, 2, 3, 16, 32};
  const uint32_t skews[] = {0, 4, 8, 16};
  int64_t idx = 0;
  for (int64_t nu : units)
    for (int64_t grid : grids)
      for (int n_kb : n_kbs)
        for (uint32_t skew : skews) {
          ++idx;
          if (grid > nu) continue;  // the launch never runs more CTAs than units
          GemmArgs a = {};
          a.n_units = nu;
          a.n_kb = n_kb;
          schedule_units(a, grid, skew);
          const uint64_t total = (uint64_t)nu * n_kb;
          if ((int64_t)a.n_dp * grid > nu || a.tail_skew > skew) return idx;
          if (a.tail_s0 != (uint64_t)a.n_dp * grid * n_kb || a.tail_s0 + a.tail_len != total)
            return idx;
          uint64_t prev = 0;
          for (int64_t c = 0; c < grid; ++c) {
            const uint64_t b0 = tail_bound(a.tail_len, grid, a.tail_skew, c);
            const uint64_t b1 = tail_bound(a.tail_len, grid, a.tail_skew, c + 1);
            if (b0 != prev || b1 < b0) return idx;
            if (a.tail_skew == 0 && b1 != a.tail_len * (c + 1) / grid) return idx;
            // a range of at least one unit (ranges of a tail shorter than
            // the grid are the even split, as before any skew)
            if (a.tail_skew > 0 && b1 - b0 < (uint64_t)n_kb) return idx;
            prev = b1;
          }
          if (prev != a.tail_len) return idx;
          // no tail unit cut twice: the CTAs whose ranges touch each unit
          if (a.tail_len >= (uint64_t)grid * n_kb) {
            for (uint64_t u = 0; u < a.tail_len / n_kb; ++u) {
              int touch = 0;
              for (int64_t c = 0; c < grid; ++c) {
                const uint64_t b0 = tail_bound(a.tail_len, grid, a.tail_skew, c);
                const uint64_t b1 = tail_bound(a.tail_len, grid, a.tail_skew, c + 1);
                if (b0 < (u + 1) * n_kb && b1 > u * n_kb) ++touch;
              }
              if (touch > 2) return idx;
            }
          }
        }
  return -1;
}

