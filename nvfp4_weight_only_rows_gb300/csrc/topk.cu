// topk.cu -- the selection step of the fused top-k: the GEMM epilogue has
// kept, per token, every logit that reached the token's running threshold
// (a superset of its k largest; the order key of row n in slot n, flagged
// in the word of its 32-row group); here one CTA per token picks the exact k
// largest candidate keys, sorts them (larger logit first, of equal logits
// the smaller row; a NaN above every number) and writes their rows and
// logits.
//
// The kernel runs once per call, briefly and cold, so its code is kept
// small (instruction fetch, not memory, bounds a bloated version): the
// common path gathers the few candidates at or above the final threshold
// into shared memory and ranks them with one warp; a byte-wise radix
// select over the candidates covers the rare token with more of them.
#include "gemm_common.cuh"

namespace nvfp4 {

constexpr int kSelThreads = 256;
constexpr int kSelCap = 8192;  // candidates at or above the threshold held in shared memory
constexpr int kGW = 16;        // group words per lane loaded before any is used
constexpr int kSelU = 4;       // groups whose candidate loads are in flight together
constexpr int kRankMax = 512;  // at most this many keys: selection by rank (one warp)

// Every candidate key of one token at or above T, through the group words,
// one thread at a time (the overflow path only).
template <typename F>
__device__ __noinline__ void topk_scan_slow(const uint2* gw, const uint32_t* src, int64_t G,
                                            int64_t N, unsigned long long T, F f) {
  const uint32_t t_hi = (uint32_t)(T >> 32);
#pragma unroll 1
  for (int64_t g = threadIdx.x; g < G; g += blockDim.x) {
    const uint2 w = __ldcg(gw + g);
    if (w.x < t_hi) continue;
    uint32_t bits = w.y;
#pragma unroll 1
    while (bits) {
      const int b = __ffs(bits) - 1;
      bits &= bits - 1;
      const int64_t slot = g * 32 + b;
      if (slot >= N) break;
      const unsigned long long key =
          ((unsigned long long)__ldcg(src + slot) << 32) | (uint32_t)~(uint32_t)slot;
      if (key >= T) f(key);
    }
  }
}

__global__ void __launch_bounds__(kSelThreads) topk_select_kernel(
    const unsigned long long* __restrict__ lines, const uint2* __restrict__ grp,
    const uint32_t* __restrict__ cand, int64_t N, int k, int64_t* __restrict__ ids,
    float* __restrict__ vals) {
  // the candidates come from the GEMM, which may still be running
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ unsigned long long s_keys[];  // kSelCap
  __shared__ uint32_t hist[256];
  __shared__ unsigned long long s_top[kTopkMax];
  __shared__ uint32_t s_n, s_m, s_need, s_match;
  __shared__ unsigned long long s_prefix;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_warps = blockDim.x >> 5;
  const int64_t tok = blockIdx.x;
  const unsigned long long T = __ldcg(lines + tok * kKeyStride);
  const uint32_t t_hi = (uint32_t)(T >> 32);  // key >= T  <=>  order key >= t_hi
  const int64_t G = (N + 31) / 32;
  const uint2* gw = grp + tok * G;
  const uint32_t* src = cand + tok * N;
  if (tid == 0) {
    s_n = 0;
    s_prefix = 0;
    s_need = (uint32_t)k;
    s_match = 0;
  }
  __syncthreads();

  // 1. the candidates at or above T, into shared memory while they fit:
  // each lane loads kGW group words at once (a warp covers 32 x kGW
  // groups) and keeps a mask of those whose largest candidate reaches T;
  // then, kSelU groups at a time, the warp loads their flagged slots
  // (lane l: slot 32g + l) and appends the keys that reach T
  for (int64_t g0 = (int64_t)warp * 32 * kGW; g0 < G; g0 += (int64_t)n_warps * 32 * kGW) {
    uint32_t bits[kGW];
    uint32_t pass = 0;  // bit u: group g0 + 32u + lane has a candidate at or above T
#pragma unroll
    for (int u = 0; u < kGW; ++u) {
      const int64_t g = g0 + u * 32 + lane;
      const uint2 w = g < G ? __ldcg(gw + g) : make_uint2(0u, 0u);
      bits[u] = w.y;
      if (w.y != 0u && w.x >= t_hi) pass |= 1u << u;
    }
#pragma unroll 1
    while (__any_sync(0xFFFFFFFFu, pass != 0u)) {
      unsigned long long key[kSelU];
      bool keep[kSelU];
#pragma unroll
      for (int v = 0; v < kSelU; ++v) {
        // the next flagged group: lowest lane with one, its lowest u
        const uint32_t who = __ballot_sync(0xFFFFFFFFu, pass != 0u);
        keep[v] = false;
        key[v] = 0ull;
        if (who) {
          const int src_lane = __ffs(who) - 1;
          const int my_u = pass ? __ffs(pass) - 1 : 0;
          uint32_t my_bits = 0;
#pragma unroll
          for (int u = 0; u < kGW; ++u) my_bits = u == my_u ? bits[u] : my_bits;
          const int u = __shfl_sync(0xFFFFFFFFu, my_u, src_lane);
          const uint32_t bj = __shfl_sync(0xFFFFFFFFu, my_bits, src_lane);
          if (lane == src_lane) pass &= pass - 1;
          const int64_t slot = (g0 + u * 32 + src_lane) * 32 + lane;
          keep[v] = ((bj >> lane) & 1u) && slot < N;
          if (keep[v])
            key[v] = ((unsigned long long)__ldcg(src + slot) << 32) | (uint32_t)~(uint32_t)slot;
        }
      }
#pragma unroll
      for (int v = 0; v < kSelU; ++v) {
        const bool kv = keep[v] && key[v] >= T;
        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, kv);
        if (bal == 0) continue;  // warp-uniform
        uint32_t pos0 = 0;
        if (lane == 0) pos0 = atomicAdd(&s_n, (uint32_t)__popc(bal));
        pos0 = __shfl_sync(0xFFFFFFFFu, pos0, 0);
        const uint32_t pos = pos0 + __popc(bal & ((1u << lane) - 1u));
        if (kv && pos < (uint32_t)kSelCap) s_keys[pos] = key[v];
      }
    }
  }
  __syncthreads();
  const uint32_t m = s_n;

  // 2a. few keys (the usual case): each key's rank is the number of larger
  // keys (they are distinct); the keys of rank < k go straight to their
  // place in the output
  if (m <= (uint32_t)kRankMax) {
    if (warp != 0) return;  // one warp: lane l ranks keys l, l + 32, ...
    for (int j = lane; j < k; j += 32) s_top[j] = 0ull;
    __syncwarp();
#pragma unroll 1
    for (uint32_t i = lane; i < m; i += 32) {
      const unsigned long long key = s_keys[i];
      uint32_t rank = 0;
#pragma unroll 8
      for (uint32_t j = 0; j < m; ++j) rank += s_keys[j] > key ? 1u : 0u;
      if (rank < (uint32_t)k) s_top[rank] = key;
    }
    __syncwarp();
    for (int j = lane; j < k; j += 32) {
      const unsigned long long key = s_top[j];
      ids[tok * k + j] = (int64_t)(uint32_t)~(uint32_t)key;
      if (vals) vals[tok * k + j] = key_value((uint32_t)(key >> 32));
    }
    return;
  }

  // 2b. the k-th largest key, a byte at a time from the top: the histogram
  // of the next byte over the keys that match the bytes chosen so far (over
  // shared memory, or, past kSelCap keys, the candidates again)
  const bool in_smem = m <= (uint32_t)kSelCap;
  unsigned long long prefix = 0, mask = 0;
  uint32_t need = (uint32_t)k;
#pragma unroll 1
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    auto count = [&](unsigned long long key) {
      if ((key & mask) == prefix) atomicAdd(&hist[(uint32_t)(key >> shift) & 255u], 1u);
    };
    if (in_smem) {
      for (uint32_t i = tid; i < m; i += blockDim.x) count(s_keys[i]);
    } else {
      topk_scan_slow(gw, src, G, N, T, count);
    }
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
#pragma unroll 1
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
  auto collect = [&](unsigned long long key) {
    if (key >= prefix) {
      const uint32_t pos = atomicAdd(&s_m, 1u);
      if (pos < (uint32_t)kTopkMax) s_top[pos] = key;
    }
  };
  if (in_smem) {
    for (uint32_t i = tid; i < m; i += blockDim.x) collect(s_keys[i]);
  } else {
    topk_scan_slow(gw, src, G, N, T, collect);
  }
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

cudaError_t topk_select_launch(const unsigned long long* lines, const uint2* grp,
                               const uint32_t* cand, int64_t M, int64_t N, int k, int64_t* ids,
                               float* vals, cudaStream_t stream) {
  const size_t smem = (size_t)kSelCap * sizeof(unsigned long long);
  static std::atomic<uint64_t> limit_set{0};
  const cudaError_t attr_err =
      smem_limit_once(limit_set, reinterpret_cast<const void*>(topk_select_kernel), smem);
  if (attr_err != cudaSuccess) return attr_err;
  PdlLaunch l(dim3((unsigned)M), dim3(kSelThreads), smem, stream);
  return cudaLaunchKernelEx(&l.cfg, topk_select_kernel, lines, grp, cand, N, k, ids, vals);
}

}  // namespace nvfp4
