// topk.cu -- the selection step of the fused top-k: the GEMM epilogue has
// appended, per token, every logit that reached the token's running
// threshold (a superset of its k largest); here one CTA per token picks the
// exact k largest candidate keys, sorts them (larger logit first, of equal
// logits the smaller row; a NaN above every number) and writes their rows
// and logits.
#include "gemm_common.cuh"

namespace nvfp4 {

constexpr int kSelThreads = 512;
constexpr int kSelCap = 8192;  // candidates at or above the threshold held in shared memory

__global__ void __launch_bounds__(kSelThreads) topk_select_kernel(
    const unsigned long long* __restrict__ lines, const unsigned long long* __restrict__ cand,
    int64_t N, int k, int64_t* __restrict__ ids, float* __restrict__ vals) {
  // the candidates come from the GEMM, which may still be running
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ unsigned long long s_keys[];  // kSelCap
  __shared__ uint32_t hist[256];
  __shared__ unsigned long long s_top[kTopkMax];
  __shared__ uint32_t s_n, s_m, s_need, s_match;
  __shared__ unsigned long long s_prefix;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t tok = blockIdx.x;
  const unsigned long long T = __ldcg(lines + tok * kKeyStride);
  const uint32_t cnt = __ldcg(reinterpret_cast<const uint32_t*>(lines + tok * kKeyStride + 1));
  const int64_t n = cnt < (uint64_t)N ? (int64_t)cnt : N;
  const unsigned long long* src = cand + tok * N;
  if (tid == 0) {
    s_n = 0;
    s_prefix = 0;
    s_need = (uint32_t)k;
    s_match = 0;
  }
  __syncthreads();

  // 1. the candidates at or above the final threshold (the token's k largest
  // among them), gathered into shared memory while they fit
  for (int64_t i0 = 0; i0 < n; i0 += blockDim.x) {
    const int64_t i = i0 + tid;
    const unsigned long long key = i < n ? __ldcg(src + i) : 0ull;
    const bool keep = i < n && key >= T;
    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, keep);
    uint32_t pos0 = 0;
    if (lane == 0 && bal) pos0 = atomicAdd(&s_n, (uint32_t)__popc(bal));
    pos0 = __shfl_sync(0xFFFFFFFFu, pos0, 0);
    const uint32_t pos = pos0 + __popc(bal & ((1u << lane) - 1u));
    if (keep && pos < (uint32_t)kSelCap) s_keys[pos] = key;
  }
  __syncthreads();
  const uint32_t m = s_n;
  const bool in_smem = m <= (uint32_t)kSelCap;
  // every key of the list: shared memory, or (more than kSelCap of them)
  // the global candidates again, filtered the same way
  auto for_each_key = [&](auto&& f) {
    if (in_smem) {
      for (uint32_t i = tid; i < m; i += blockDim.x) f(s_keys[i]);
    } else {
      for (int64_t i = tid; i < n; i += blockDim.x) {
        const unsigned long long key = __ldcg(src + i);
        if (key >= T) f(key);
      }
    }
  };

  // 2. the k-th largest key, a byte at a time from the top: the histogram of
  // the next byte over the keys that match the bytes chosen so far
  unsigned long long prefix = 0, mask = 0;
  uint32_t need = (uint32_t)k;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for_each_key([&](unsigned long long key) {
      if ((key & mask) == prefix) atomicAdd(&hist[(uint32_t)(key >> shift) & 255u], 1u);
    });
    __syncthreads();
    if (warp == 0) {
      // lane l holds bins 255 - 8l down to 248 - 8l; an inclusive scan over
      // the lanes counts the keys in higher bins
      uint32_t c[8], sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[255 - 8 * lane - j];
        sum += c[j];
      }
      uint32_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t excl = incl - sum;
      if (excl < need && need <= incl) {
        uint32_t acc = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (acc + c[j] >= need) {
            s_prefix = prefix | ((unsigned long long)(255 - 8 * lane - j) << shift);
            s_need = need - acc;
            s_match = c[j];
            break;
          }
          acc += c[j];
        }
      }
    }
    __syncthreads();
    prefix = s_prefix;
    need = s_need;
    mask |= 0xFFull << shift;
    // all keys that match the prefix are among the k largest: the rest of
    // the key does not matter
    if (s_match == need) break;
  }

  // 3. exactly k keys reach `prefix` (the bytes below it read as zero)
  if (tid == 0) s_m = 0;
  const int P = k <= 1 ? 1 : 1 << (32 - __clz(k - 1));  // k rounded up to a power of two
  for (int i = k + tid; i < P; i += blockDim.x) s_top[i] = 0ull;  // below every key
  __syncthreads();
  for_each_key([&](unsigned long long key) {
    if (key >= prefix) {
      const uint32_t pos = atomicAdd(&s_m, 1u);
      if (pos < (uint32_t)kTopkMax) s_top[pos] = key;
    }
  });
  __syncthreads();

  // 4. bitonic sort, largest key first
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < P / 2; i += blockDim.x) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const unsigned long long a = s_top[lo], b = s_top[hi];
        if ((a < b) == desc) {
          s_top[lo] = b;
          s_top[hi] = a;
        }
      }
      __syncthreads();
    }
  }
  for (int j = tid; j < k; j += blockDim.x) {
    const unsigned long long key = s_top[j];
    ids[tok * k + j] = (int64_t)(uint32_t)~(uint32_t)key;
    if (vals) vals[tok * k + j] = key_value((uint32_t)(key >> 32));
  }
}

cudaError_t topk_select_launch(const unsigned long long* lines, const unsigned long long* cand,
                               int64_t M, int64_t N, int k, int64_t* ids, float* vals,
                               cudaStream_t stream) {
  const size_t smem = (size_t)kSelCap * sizeof(unsigned long long);
  static const cudaError_t attr_err = cudaFuncSetAttribute(
      topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (attr_err != cudaSuccess) return attr_err;
  PdlLaunch l(dim3((unsigned)M), dim3(kSelThreads), smem, stream);
  return cudaLaunchKernelEx(&l.cfg, topk_select_kernel, lines, cand, N, k, ids, vals);
}

}  // namespace nvfp4
