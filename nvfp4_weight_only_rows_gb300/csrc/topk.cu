// topk.cu -- the selection steps of the fused top-k, one CTA per token
// each, both writing the rows and logits of the token's k largest, sorted
// (larger logit first, of equal logits the smaller row; a NaN above every
// number):
// - topk_select_kernel, beyond 256 tokens: the GEMM epilogue has kept, per
//   token, every logit that reached the token's running threshold (a
//   superset of its k largest; the order key of row n in slot n, flagged in
//   the word of its 32-row group, a word written only for groups with
//   candidates and marked in the token's group bitmap), and this kernel
//   picks the exact k largest of those keys;
// - topk_logits_kernel (after "from logits" below), up to 256 tokens: the
//   GEMM has written the fp32 logits and the largest of every 32 rows, and
//   this kernel bounds the k-th largest from those maxima and ranks the few
//   logits that reach the bound.
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
__device__ __noinline__ void topk_scan_slow(const uint2* gw, const uint32_t* gbits,
                                            const uint32_t* src, int64_t G, int64_t N,
                                            unsigned long long T, F f) {
  const uint32_t t_hi = (uint32_t)(T >> 32);
#pragma unroll 1
  for (int64_t g = threadIdx.x; g < G; g += blockDim.x) {
    if (((__ldcg(gbits + (g >> 5)) >> (g & 31)) & 1u) == 0u) continue;  // no word this call
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
    const uint32_t* __restrict__ cand, const uint32_t* __restrict__ tk_hist, int hstride,
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
  const int n_warps = blockDim.x >> 5;
  const int64_t tok = blockIdx.x;
  const unsigned long long T = __ldcg(lines + tok * kKeyStride);
  const uint32_t t_hi = (uint32_t)(T >> 32);  // key >= T  <=>  order key >= t_hi
  const int64_t G = (N + 31) / 32;
  const uint2* gw = grp + tok * G;
  const uint32_t* gbits = tk_hist + tok * hstride + kHistWords;  // groups with a word this call
  const int64_t GB = (G + 31) / 32;
  const uint32_t* src = cand + tok * N;
  if (tid == 0) {
    s_n = 0;
    s_prefix = 0;
    s_need = (uint32_t)k;
    s_match = 0;
  }
  __syncthreads();

  // 1. the candidates at or above T, into shared memory while they fit:
  // lane u < kGW loads the bitmap word of the warp's groups 32 u .. 32 u +
  // 31, then each lane loads the words of its kGW groups that have one (a
  // warp covers 32 x kGW groups) and keeps a mask of those whose largest
  // candidate reaches T;
  // then, kSelU groups at a time, the warp loads their flagged slots
  // (lane l: slot 32g + l) and appends the keys that reach T
  for (int64_t g0 = (int64_t)warp * 32 * kGW; g0 < G; g0 += (int64_t)n_warps * 32 * kGW) {
    uint32_t bits[kGW];
    uint32_t pass = 0;  // bit u: group g0 + 32u + lane has a candidate at or above T
    const int64_t bw = (g0 >> 5) + lane;
    const uint32_t my_bm = lane < kGW && bw < GB ? __ldcg(gbits + bw) : 0u;
#pragma unroll
    for (int u = 0; u < kGW; ++u) {
      const int64_t g = g0 + u * 32 + lane;
      const bool has = (__shfl_sync(0xFFFFFFFFu, my_bm, u) >> lane) & 1u;
      const uint2 w = has ? __ldcg(gw + g) : make_uint2(0u, 0u);
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
      topk_scan_slow(gw, gbits, src, G, N, T, count);
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
    topk_scan_slow(gw, gbits, src, G, N, T, collect);
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
                               const uint32_t* cand, const uint32_t* hist, int hstride, int64_t M,
                               int64_t N, int k, int64_t* ids, float* vals, cudaStream_t stream) {
  const size_t smem = (size_t)kSelCap * sizeof(unsigned long long);
  static std::atomic<uint64_t> limit_set{0};
  const cudaError_t attr_err =
      smem_limit_once(limit_set, reinterpret_cast<const void*>(topk_select_kernel), smem);
  if (attr_err != cudaSuccess) return attr_err;
  PdlLaunch l(dim3((unsigned)M), dim3(kSelThreads), smem, stream);
  return cudaLaunchKernelEx(&l.cfg, topk_select_kernel, lines, grp, cand, hist, hstride, N, k,
                            ids, vals);
}

// ------------------------------------------------------------ from logits
// Top-k of decode-sized products: the GEMM writes the fp32 logits (M x N, a
// few tens of MB next to hundreds of MB of weights) and, per token, the
// largest order key of every 32 rows (its epilogue warps hold 32
// consecutive rows); then one CTA per token selects:
// 1. the super-group maxima: the largest of every sg consecutive group
//    maxima, sg the widest power of two up to 32 that leaves at least 2k of
//    them, or the narrowest that leaves at most 256 (at least k of them
//    whenever the token has k groups);
// 2. the bound: the k-th largest super-group maximum (warp 0 sorts them in
//    registers).  Each super-group maximum is a logit of its own rows, so
//    at least k logits reach the bound and the k-th largest logit is not
//    below it; with fewer than k groups the bound is 0 (every logit);
// 3. the hot groups: those whose maximum reaches the bound (the others hold
//    no logit that does);
// 4. their logits that reach the bound (a few more than k: with s
//    super-groups, about -s ln(1 - k / s)); up to 128 of them warp 0 sorts
//    in registers, up to kRankCap the block ranks them against each other.
// The keys (order key << 32 | ~row) are distinct, so the answer is that of
// a sort of the fp32 logits, bit for bit.  A radix select over all N keys
// takes over where more than kHotCap groups or kRankCap logits reach the
// bound (heavily tied logits, or a vocabulary of few groups).
constexpr int kRankCap = 512;     // keys ranked against each other in shared memory
constexpr int kDigitBits = 11;    // radix digit: 2048 bins (a quarter octave at the top)
constexpr int kBins = 1 << kDigitBits;
constexpr int kSuperCap = 256;    // super-group maxima (sorted by one warp, 8 per lane)
constexpr int kHotCap = 2048;     // groups whose maximum reaches the bound

__device__ __forceinline__ unsigned long long logit_key(float v, uint32_t n) {
  return ((unsigned long long)logit_order(v) << 32) | (uint32_t)~n;
}

// Every one of the `count` distinct keys in `keys` (shared memory, count <=
// kRankCap) against the others: out[r] receives the key of rank r < want.
template <int T>
__device__ void rank_keys(const unsigned long long* keys, int count, int want,
                          unsigned long long* out) {
  for (int i = threadIdx.x; i < count; i += T) {
    const unsigned long long kk = keys[i];
    int rank = 0;
#pragma unroll 8
    for (int j = 0; j < count; ++j) rank += keys[j] > kk ? 1 : 0;
    if (rank < want) out[rank] = kk;
  }
  __syncthreads();
}

// The `want` largest of the `count` distinct keys key_at(i) (whole block of
// T threads, want <= count, want <= kTopkMax): an 11-bit digit at a time
// from the top, the histogram of the next digit over the keys inside the
// range chosen so far picks the digit of the want-th largest, until the keys
// at or above that prefix (zeros below it) are few enough to rank.
template <int T, typename KeyAt>
__device__ void select_largest(KeyAt key_at, int count, int want, unsigned long long* out,
                               unsigned long long* s_rank, uint32_t* hist) {
  __shared__ unsigned long long s_prefix;
  __shared__ uint32_t s_need, s_above, s_bin, s_n;
  constexpr int kBinsPerThread = kBins / T;
  __shared__ uint32_t s_warp[T / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned long long prefix = 0ull, mask = 0ull;
  // need: keys still to find inside the range; above: keys above the range
  uint32_t need = (uint32_t)want, above = 0;
  if (count > kRankCap) {
#pragma unroll 1
    for (int top = 64; top > 0; top -= kDigitBits) {
      const int width = top < kDigitBits ? top : kDigitBits;
      const int shift = top - width;
      for (int i = tid; i < kBins; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      for (int i = tid; i < count; i += blockDim.x) {
        const unsigned long long kk = key_at(i);
        if ((kk & mask) == prefix)
          atomicAdd(&hist[(uint32_t)(kk >> shift) & ((1u << width) - 1u)], 1u);
      }
      __syncthreads();
      // thread t holds the kBinsPerThread bins below kBins - kBinsPerThread t
      // (from the top); a block scan from the top counts the range's keys in
      // higher bins
      uint32_t c[kBinsPerThread], sum = 0;
#pragma unroll
      for (int j = 0; j < kBinsPerThread; ++j) {
        c[j] = hist[kBins - 1 - kBinsPerThread * tid - j];
        sum += c[j];
      }
      uint32_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) s_warp[warp] = incl;
      __syncthreads();
      for (int w = 0; w < warp; ++w) incl += s_warp[w];
      const uint32_t excl = incl - sum;
      if (excl < need && need <= incl) {
        uint32_t acc = excl;
#pragma unroll 1
        for (int j = 0; j < kBinsPerThread; ++j) {
          if (acc + c[j] >= need) {
            const uint32_t bin = kBins - 1 - kBinsPerThread * tid - j;
            s_prefix = prefix | ((unsigned long long)bin << shift);
            s_need = need - acc;
            s_above = above + acc;
            s_bin = c[j];
            break;
          }
          acc += c[j];
        }
      }
      __syncthreads();
      prefix = s_prefix;
      need = s_need;
      above = s_above;
      mask |= ((1ull << width) - 1ull) << shift;
      // the keys at or above the new prefix: those above its range and its bin
      if (above + s_bin <= (uint32_t)kRankCap) break;
    }
  }
  // the keys at or above `prefix` (all of them when count <= kRankCap)
  if (tid == 0) s_n = 0;
  __syncthreads();
  for (int i = tid; i < count; i += blockDim.x) {
    const unsigned long long kk = key_at(i);
    if (kk >= prefix) {
      const uint32_t pos = atomicAdd(&s_n, 1u);
      if (pos < (uint32_t)kRankCap) s_rank[pos] = kk;
    }
  }
  __syncthreads();
  rank_keys<T>(s_rank, (int)min(s_n, (uint32_t)kRankCap), want, out);
}

// Sorts the 32 R values a warp holds (R per lane, element lane R + r) into
// descending order in registers: a bitonic network, partners R or more
// elements apart exchanged by shuffles, nearer ones inside the lane.
template <int R, typename V>
__device__ __forceinline__ void warp_sort_desc(V (&a)[R], int lane) {
#pragma unroll
  for (int s = 2; s <= 32 * R; s <<= 1) {
#pragma unroll
    for (int d = s >> 1; d > 0; d >>= 1) {
      if (d >= R) {
        const bool lower = (lane & (d / R)) == 0;
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const bool desc = ((lane * R + r) & s) == 0;
          const V other = __shfl_xor_sync(0xFFFFFFFFu, a[r], d / R);
          a[r] = lower == desc ? (a[r] > other ? a[r] : other) : (a[r] < other ? a[r] : other);
        }
      } else {
#pragma unroll
        for (int r = 0; r < R; ++r) {
          if ((r & d) == 0) {
            const bool desc = ((lane * R + r) & s) == 0;
            const V x = a[r], y = a[r + d];
            if ((x < y) == desc) {
              a[r] = y;
              a[r + d] = x;
            }
          }
        }
      }
    }
  }
}

// The n values src[0, n) (shared memory, n <= 32 R) sorted by one warp,
// larger first (zeros pad the rest); returns the one at position `pos`.
template <int R, typename V>
__device__ __forceinline__ V warp_kth(const V* src, int n, int pos, int lane) {
  V a[R];
#pragma unroll
  for (int r = 0; r < R; ++r) a[r] = lane * R + r < n ? src[lane * R + r] : V(0);
  warp_sort_desc<R>(a, lane);
  V mine = a[0];
#pragma unroll
  for (int r = 1; r < R; ++r) mine = r == pos % R ? a[r] : mine;
  return __shfl_sync(0xFFFFFFFFu, mine, pos / R);
}

// Keys src[0, n) (shared memory, distinct, n <= 32 R) sorted by one warp;
// the first k (k <= n) go to ids / vals of token m.
template <int R>
__device__ __forceinline__ void warp_sort_out(const unsigned long long* src, int n, int k,
                                              int64_t m, int64_t* ids, float* vals, int lane) {
  unsigned long long a[R];
#pragma unroll
  for (int r = 0; r < R; ++r) a[r] = lane * R + r < n ? src[lane * R + r] : 0ull;
  warp_sort_desc<R>(a, lane);
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int e = lane * R + r;
    if (e < k) {
      ids[m * k + e] = (int64_t)(uint32_t)~(uint32_t)a[r];
      if (vals) vals[m * k + e] = key_value((uint32_t)(a[r] >> 32));
    }
  }
}

// Appends `key` to s_list (capacity kRankCap; the count in *s_n keeps
// growing past it) where `take`; the whole warp calls it.
__device__ __forceinline__ void append_key(bool take, unsigned long long key,
                                           unsigned long long* s_list, uint32_t* s_n) {
  const uint32_t bal = __ballot_sync(0xFFFFFFFFu, take);
  if (bal == 0u) return;
  const int lane = threadIdx.x & 31;
  uint32_t pos0 = 0;
  if (lane == 0) pos0 = atomicAdd(s_n, (uint32_t)__popc(bal));
  pos0 = __shfl_sync(0xFFFFFFFFu, pos0, 0);
  const uint32_t pos = pos0 + __popc(bal & ((1u << lane) - 1u));
  if (take && pos < (uint32_t)kRankCap) s_list[pos] = key;
}

// Group maxima a thread holds: a token's ceil(N / 32) <= 8192 of them.
template <int T>
constexpr int groups_per_thread() { return (int)(kTopkLogitsMaxN / 32) / T; }

template <int T>
__global__ void __launch_bounds__(T) topk_logits_kernel(
    const float* __restrict__ logits, const uint32_t* __restrict__ gmax, int64_t N, int k,
    int64_t* __restrict__ ids, float* __restrict__ vals) {
  // the logits and group maxima come from the GEMM, which may still be running
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int kPer = groups_per_thread<T>();
  __shared__ unsigned long long s_rank[kRankCap];
  __shared__ unsigned long long s_out[kTopkMax];
  __shared__ uint32_t hist[kBins];
  __shared__ uint32_t s_super[kSuperCap];
  __shared__ uint32_t s_hot[kHotCap];
  __shared__ uint32_t s_bound, s_n, s_nhot;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lt = (1u << lane) - 1u;
  const int64_t m = blockIdx.x;
  const int G = (int)((N + 31) / 32);
  const float* src = logits + m * N;
  const uint32_t* gm = gmax + m * (int64_t)G;
  // 1. the group maxima (group tid + j T), all loads in flight together
  uint32_t g[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int i = tid + j * T;
    g[j] = i < G ? __ldcg(gm + i) : 0u;
  }
  int sg = 32;
  while (sg > 1 && (G + sg - 1) / sg < 2 * k && (G + sg / 2 - 1) / (sg / 2) <= kSuperCap) sg >>= 1;
  const int n_super = (G + sg - 1) / sg;
  // warp w holds groups j T + 32 w + lane in step j: a 32-group super-group,
  // or 32 / sg of them
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int i = tid + j * T;
    if (j * T + warp * 32 < G) {  // warp-uniform
      if (sg == 32) {
        const uint32_t mx = __reduce_max_sync(0xFFFFFFFFu, g[j]);
        if (lane == 0) s_super[i >> 5] = mx;
      } else {
        uint32_t mx = g[j];
        for (int o = 1; o < sg; o <<= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        if ((lane & (sg - 1)) == 0 && i < G) s_super[i / sg] = mx;
      }
    }
  }
  if (tid == 0) {
    s_n = 0;
    s_nhot = 0;
    s_bound = 0u;  // fewer than k groups: every logit is a candidate
  }
  __syncthreads();
  // 2. the bound: the k-th largest super-group maximum, sorted by warp 0
  if (warp == 0 && n_super >= k) {
    const uint32_t b = n_super <= 128 ? warp_kth<4>(s_super, n_super, k - 1, lane)
                                      : warp_kth<8>(s_super, n_super, k - 1, lane);
    if (lane == 0) s_bound = b;
  }
  __syncthreads();
  const uint32_t bound = s_bound;
  // 3. the hot groups, appended to s_hot (one shared counter per warp step)
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int i = tid + j * T;
    const bool hot = i < G && g[j] >= bound;
    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, hot);
    if (bal != 0u) {
      uint32_t pos0 = 0;
      if (lane == 0) pos0 = atomicAdd(&s_nhot, (uint32_t)__popc(bal));
      pos0 = __shfl_sync(0xFFFFFFFFu, pos0, 0);
      const uint32_t at = pos0 + __popc(bal & lt);
      if (hot && at < (uint32_t)kHotCap) s_hot[at] = (uint32_t)i;
    }
  }
  __syncthreads();
  const uint32_t n_hot = s_nhot;
  // 4. the hot groups' logits that reach the bound: a warp per group, two
  // groups' loads in flight per warp
  bool ranked = false;
  if (n_hot <= (uint32_t)kHotCap) {
    constexpr int kW = T / 32;
    for (int h0 = warp; h0 < (int)n_hot; h0 += 2 * kW) {
      float v[2];
      int64_t row[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int h = h0 + u * kW;
        row[u] = h < (int)n_hot ? (int64_t)s_hot[h] * 32 + lane : N;
        v[u] = row[u] < N ? __ldcg(src + row[u]) : 0.0f;
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const unsigned long long key = logit_key(v[u], (uint32_t)row[u]);
        append_key(row[u] < N && (uint32_t)(key >> 32) >= bound, key, s_rank, &s_n);
      }
    }
    __syncthreads();
    const int n_cand = (int)s_n;
    // 5. few candidates (the usual case): warp 0 sorts them and writes the k best
    if (n_cand <= 128) {
      if (warp == 0) {
        if (n_cand <= 64) warp_sort_out<2>(s_rank, n_cand, k, m, ids, vals, lane);
        else warp_sort_out<4>(s_rank, n_cand, k, m, ids, vals, lane);
      }
      return;
    }
    if (n_cand <= kRankCap) {
      rank_keys<T>(s_rank, n_cand, k, s_out);
      ranked = true;
    }
  }
  if (!ranked)  // block-uniform
    select_largest<T>([&](int i) { return logit_key(__ldcg(src + i), (uint32_t)i); }, (int)N, k,
                      s_out, s_rank, hist);
  for (int j = tid; j < k; j += T) {
    const unsigned long long kk = s_out[j];
    ids[m * k + j] = (int64_t)(uint32_t)~(uint32_t)kk;
    if (vals) vals[m * k + j] = key_value((uint32_t)(kk >> 32));
  }
}

cudaError_t topk_logits_launch(const float* logits, const uint32_t* gmax, int64_t M, int64_t N,
                               int k, int64_t* ids, float* vals, cudaStream_t stream) {
  PdlLaunch l(dim3((unsigned)M), dim3(1024), 0, stream);
  return cudaLaunchKernelEx(&l.cfg, topk_logits_kernel<1024>, logits, gmax, N, k, ids, vals);
}

}  // namespace nvfp4
