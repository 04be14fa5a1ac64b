// gemm_common.cuh -- the parts of the persistent tcgen05 lm_head GEMMs that
// the W4A16 (NVFP4 weights) and W8A8 (fp8 weights) products share: kernel
// arguments, the unit schedule (strided whole units, then a stream-K tail),
// bounded warp-level waits, the epilogue role (TMEM drain, per-token and
// per-row scales, split-unit combine, logits stores or the fused greedy
// argmax) and the host-side tensor-map and workspace helpers.
//
// A unit is 128 vocabulary rows x BN tokens; the MMA runs in the swapped
// orientation D[row, token], so D lives in TMEM with one lane per row.
#pragma once

#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <type_traits>
#include <mutex>

#include "common.cuh"

namespace nvfp4 {

constexpr int kRows = 128;   // vocabulary rows per unit (MMA M)
constexpr int kKB = 256;     // k per pipeline stage
constexpr int kMaxBN = 128;  // largest token tile
constexpr int kWideBN = 256;  // the W8A8 prefill's token tile (its TMEM holds no scales)
constexpr int kOutArgmax = 2;   // third output mode (after NVFP4_OUT_F32, NVFP4_OUT_BF16)
constexpr int kOutTopk = 3;     // fourth: the k largest logits of each token
constexpr int kOutLogitsGroups = 4;  // fifth: fp32 logits and their 32-row maxima (grp_max)
constexpr int kKeyStride = 16;  // argmax / top-k: one 128-byte line of per-token state (spreads the atomics)
constexpr int kTopkMax = 128;   // largest k of the fused top-k
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per pipeline wait

struct GemmArgs {
  int64_t M, N, K;
  int BN;              // token tile, multiple of 16, <= 128
  int n_ttiles;        // token tiles
  int64_t n_units;     // weight tiles x token tiles
  int n_kb;            // 256-k stages per unit
  uint32_t n_dp;       // whole units per CTA in strided waves (unit c + j * grid)
  uint64_t tail_s0;    // first stage of the stream-K tail (unit-major, k-minor)
  uint64_t tail_len;   // stages in the tail, split over the grid (see tail_bound)
  uint32_t tail_skew;  // 0: an even split; a: CTA c's share falls linearly by a / 64 each side
  uint32_t tmem_cols;  // allocated TMEM columns
  uint32_t dbuf_log2;  // accumulator buffers in TMEM: 1 << dbuf_log2 (2 or 4)
  const float* tok_scale;
  void* out;
  int32_t* status;
  uint32_t* split_cnt;    // [grid][4] arrivals at a split unit, per TMEM lane quadrant
  uint32_t* split_ready;  // [grid][4] the first arriver's partial is in split_part
  float* split_part;      // [grid][4][BN][32] fp32 partial accumulators
  // greedy argmax output mode only
  unsigned long long* am_keys;  // [m_pad * kKeyStride] per-token maxima (order key << 32 | ~n),
                                // zeroed per call by the prep kernel
  uint32_t* am_done;            // CTAs that have finished, zeroed per call
  int64_t* am_idx;              // [M] result: vocabulary row of the largest logit
  float* am_val;                // [M] result: that logit (may be null)
  // top-k output mode only (am_keys then holds per token line: word 0 the
  // threshold key, a lower bound of the token's k-th largest candidate
  // key; the low half of word 2 the largest candidate order key)
  uint32_t* tk_cand;            // [M][N] candidate order keys, slot n for row n
  uint2* tk_grp;                // [M][tk_groups] per 32 rows: {largest candidate order key,
                                //   bit j: slot 32g + j holds a candidate}
  int64_t tk_groups;            // ceil(N / 32)
  uint32_t* tk_hist;            // [m_pad][tk_hstride] per token: the histogram of the
                                //   largest key of each candidate group (kHistWords), then
                                //   one bit per group whose word this call wrote
  int tk_hstride;               // u32 per token in tk_hist
  int tk_k;                     // k, 1 .. kTopkMax
  const float* row_scale;       // [N] per-row weight scale (fp8 weights), else null
  // output mode kOutLogitsGroups only: per token, the largest order key
  // (logit_order) of every 32 rows of the fp32 logits, [M][ceil(N / 32)]
  uint32_t* grp_max;
  // grouped product (experts) only
  const int32_t* grp_off;       // [n_groups + 1] token row offsets of the groups
  const float* grp_global;      // [n_groups] per-group weight global scale
  int n_groups;
};

constexpr int kMaxGroups = 256;  // experts of one grouped call

// The schedule of a call.  For the plain product it comes from the host
// (GemmArgs); for the grouped product every CTA derives it on the device
// from the group offsets (shared memory), so the host never reads them.
struct Sched {
  uint32_t n_dp;      // whole units per CTA in strided waves
  uint32_t grid;      // CTAs that take part (blockIdx.x >= grid: no work)
  uint64_t tail_s0;   // first stage of the stream-K tail
  uint64_t tail_len;  // stages in the tail
  uint32_t tail_skew;  // as GemmArgs::tail_skew
  uint32_t nt;        // grouped: weight tiles per group
  const uint32_t* unit_pre;  // grouped: [n_groups + 1] prefix of units per group (shared)
  const int32_t* off;        // grouped: [n_groups + 1] token row offsets (shared)
  uint32_t units_end;  // the waves take units below this index (their last wave may be partial)
  const uint2* grp_tab;      // grouped: this CTA's wave unit j (shared), j < n_tab: {group |
                             //   reused << 31, weight tile | token tile << 16}
  uint32_t n_tab;
};

constexpr int kGrpTab = 64;  // grouped: wave units per CTA whose place is looked up, not searched

__device__ __forceinline__ Sched plain_sched(const GemmArgs& p) {
  return Sched{p.n_dp, gridDim.x, p.tail_s0, p.tail_len, p.tail_skew, 0u, nullptr, nullptr,
               p.n_dp * gridDim.x, nullptr, 0u};
}

// Where a unit lives: its first weight row (the TMA coordinate), first
// output column, token rows [t0, t_end) of its group, and whether its
// weight tile is read by more than one token tile.
struct UnitGeom {
  int64_t w_row, n0, t0, t_end;
  bool reused;
};

// Grouped: the group e with unit_pre[e] <= u < unit_pre[e + 1] (binary search).
__device__ __forceinline__ int unit_group(const GemmArgs& p, const uint32_t* unit_pre, uint32_t u) {
  int lo = 0, hi = p.n_groups;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (unit_pre[mid] <= u) lo = mid; else hi = mid;
  }
  return lo;
}

// j: the piece's index in the CTA's sequence (the first n_tab pieces are its
// wave units, whose group and tiles the schedule build put in grp_tab)
template <bool kGrouped>
__device__ __forceinline__ UnitGeom unit_geom(const GemmArgs& p, const Sched& s, uint32_t u,
                                              uint32_t j = 0xFFFFFFFFu) {
  UnitGeom g;
  if constexpr (!kGrouped) {
    g.n0 = g.w_row = (int64_t)(u / p.n_ttiles) * kRows;
    g.t0 = (int64_t)(u % p.n_ttiles) * p.BN;
    g.t_end = p.M;
    g.reused = p.n_ttiles > 1;
  } else {
    int lo;
    uint32_t wt, tt;
    if (j < s.n_tab) {
      const uint2 e = s.grp_tab[j];
      lo = (int)(e.x & 0x7FFFFFFFu);
      wt = e.y & 0xFFFFu;
      tt = e.y >> 16;
      g.reused = (e.x >> 31) != 0u;
    } else {
      lo = unit_group(p, s.unit_pre, u);
      const uint32_t local = u - s.unit_pre[lo];
      const uint32_t ttc = (s.unit_pre[lo + 1] - s.unit_pre[lo]) / s.nt;  // token tiles of group lo
      wt = local / ttc;
      tt = local % ttc;
      g.reused = ttc > 1;
    }
    g.n0 = (int64_t)wt * kRows;
    g.w_row = (int64_t)lo * p.N + g.n0;
    g.t0 = s.off[lo] + (int64_t)tt * p.BN;
    g.t_end = s.off[lo + 1] > s.off[lo] ? s.off[lo + 1] : s.off[lo];  // offsets are within [0, M]
  }
  return g;
}

// Grouped product: the whole block loads the group offsets into `off`,
// each clamped to [0, M] (so no token row outside [0, M) is ever touched,
// even for offsets that break the non-decreasing contract), then a block
// barrier; warp 0 then derives the schedule (before the block barrier that
// publishes it).  Units of group e: weight tiles x ceil(rows_e / BN), BN a
// power of two.
__device__ __forceinline__ void grouped_offsets_load(const GemmArgs& p, int32_t* off) {
  for (int e = threadIdx.x; e <= p.n_groups; e += blockDim.x) {
    const int32_t o = p.grp_off[e];
    off[e] = o < 0 ? 0 : (o > p.M ? (int32_t)p.M : o);
  }
}

// Warp 0 (all lanes): lane l takes a contiguous run of groups, the warp
// scans the run totals.
__device__ __forceinline__ void grouped_sched_build(const GemmArgs& p, Sched* s, uint32_t* unit_pre,
                                                    const int32_t* off, uint2* grp_tab,
                                                    uint32_t n_kb, int lane) {
  const uint32_t nt = (uint32_t)((p.N + kRows - 1) / kRows);
  const int shift = __ffs(p.BN) - 1;  // BN = 1 << shift
  const int E = p.n_groups;
  const int per = (E + 31) / 32;
  const int e0 = lane * per, e1 = min(E, e0 + per);
  uint32_t run = 0;
  for (int e = e0; e < e1; ++e) {
    const int32_t rows = off[e + 1] > off[e] ? off[e + 1] - off[e] : 0;
    run += nt * (uint32_t)((rows + p.BN - 1) >> shift);
  }
  uint32_t incl = run;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += v;
  }
  uint32_t acc = incl - run;  // units before this lane's run
  for (int e = e0; e < e1; ++e) {
    unit_pre[e] = acc;
    const int32_t rows = off[e + 1] > off[e] ? off[e + 1] - off[e] : 0;
    acc += nt * (uint32_t)((rows + p.BN - 1) >> shift);
  }
  const uint32_t n_units = __shfl_sync(0xFFFFFFFFu, incl, 31);
  if (lane == 0) unit_pre[E] = n_units;
  __syncwarp();
  const uint32_t grid = n_units < gridDim.x ? n_units : gridDim.x;
  uint32_t n_dp, units_end;
  uint64_t tail_s0, tail_len;
  if (grid > 0 && (n_kb <= 4 || n_units >= 8 * grid)) {
    // short units, or many per CTA: whole units only, the last wave partial
    // (a CTA ends at most one unit after another; splitting the last units
    // would cost each cut unit a partial tile through global memory; same
    // box, 64 tokens of a 128-expert top-8 layer: w2 35.4 -> 32.9 us,
    // w13 48.1 -> 47.2 us)
    n_dp = (n_units + grid - 1) / grid;
    units_end = n_units;
    tail_s0 = (uint64_t)n_units * n_kb;
    tail_len = 0;
  } else {
    const uint32_t dp = (grid > 0 && n_units >= 2 * grid) ? n_units / grid - 1 : 0;
    n_dp = dp;
    units_end = dp * grid;
    tail_s0 = (uint64_t)dp * grid * n_kb;
    tail_len = (uint64_t)(n_units - dp * grid) * n_kb;
  }
  // where this CTA's wave units lie (group, weight tile, token tile), one
  // search per lane; weight and token tiles must fit 16 bits each
  const bool fits = nt <= 0xFFFFu && ((uint64_t)p.M + p.BN - 1) / p.BN <= 0xFFFFu;
  const uint32_t n_tab = fits ? (n_dp < (uint32_t)kGrpTab ? n_dp : (uint32_t)kGrpTab) : 0u;
  for (uint32_t j = (uint32_t)lane; j < n_tab; j += 32) {
    const uint32_t u = blockIdx.x + j * grid;
    uint2 e = make_uint2(0u, 0u);
    if (u < units_end) {
      const int lo = unit_group(p, unit_pre, u);
      const uint32_t local = u - unit_pre[lo];
      const uint32_t ttc = (unit_pre[lo + 1] - unit_pre[lo]) / nt;
      e = make_uint2((uint32_t)lo | (ttc > 1 ? 0x80000000u : 0u),
                     (local / ttc) | ((local % ttc) << 16));
    }
    grp_tab[j] = e;
  }
  if (lane != 0) return;
  s->grid = grid;
  s->n_dp = n_dp;
  s->units_end = units_end;
  s->tail_s0 = tail_s0;
  s->tail_len = tail_len;
  s->tail_skew = 0;
  s->nt = nt;
  s->unit_pre = unit_pre;
  s->off = off;
  s->grp_tab = grp_tab;
  s->n_tab = blockIdx.x < grid ? n_tab : 0u;
}

// one lane of a converged warp (the lowest active lane)
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b32 r;\n\t"
      "elect.sync r|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// Before a producer warp exits, wait (bounded) until the last TMA load it
// issued into each ring slot has landed, so no copy targets freed memory.
__device__ __forceinline__ void drain_loads(uint64_t* full, uint32_t n_slots, uint32_t issued,
                                            int /*arrivals*/, int32_t* status) {
  volatile int32_t zero = 0;
  WaitCtl drain{status, &zero, 100000000ull};
  for (uint32_t s = 0; s < n_slots && s < issued; ++s) {
    const uint32_t fills = issued / n_slots + (s < issued % n_slots ? 1u : 0u);
    mbar_wait(&full[s], (fills - 1) & 1, drain);
  }
}

// Wait until the preceding kernel in the stream (launched with programmatic
// stream serialization) has completed and its writes are visible.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Poll a global flag (acquire) until it is non-zero, at most the wait limit.
// The writer is a CTA that has already announced itself, so this is short.
__device__ __forceinline__ bool spin_until_set(const uint32_t* flag, const WaitCtl& w) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
  if (v) return __all_sync(0xFFFFFFFFu, true);
  const uint64_t t0 = globaltimer_ns();
  bool ok = true;
  for (uint32_t it = 1;; ++it) {
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    if (v) break;
    if ((it & 63u) == 0 && globaltimer_ns() - t0 > w.limit_ns) {
      raise_status(w.status, NVFP4_ERR_TIMEOUT);
      *w.abort = 1;
      ok = false;
      break;
    }
  }
  return __all_sync(0xFFFFFFFFu, ok);
}

// warp-uniform bounded wait: every lane polls, the warp agrees on the outcome
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtl& wc) {
  const bool ok = mbar_wait(bar, parity, wc);
  return __all_sync(0xFFFFFFFFu, ok);
}

// ------------------------------------------------------------ greedy argmax
// A logit's 32-bit order key: for the logits the epilogue forms (never -0;
// a NaN only in the positive form the GPU's arithmetic produces) unsigned
// order of keys is the order of values and every NaN is above +Inf.  A
// candidate is key << 32 | ~n: the larger 64-bit word has the larger
// logit, and of equal logits the smaller row.
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t b = __float_as_uint(v);
  return b ^ ((uint32_t)((int32_t)b >> 31) | 0x80000000u);
}

// Order key of a logit for the top-k selection: unsigned order equals the
// float order, -0 counts as +0, a NaN sits above every number (positive
// NaNs) or below (negative).
__device__ __forceinline__ uint32_t logit_order(float v) {
  uint32_t b = __float_as_uint(v);
  if ((b & 0x7FFFFFFFu) == 0u) b = 0u;
  return b ^ ((uint32_t)((int32_t)b >> 31) | 0x80000000u);
}

// Per token of a 16-token chunk, the largest order key of the warp's 32
// rows (one group: the warp's rows start at a multiple of 32), into
// p.grp_max[token][group].  A butterfly over the lanes halves the tokens
// each lane keeps at every step (exchanging the half its partner keeps), so
// that lanes 2u and 2u + 1 end with token u's maximum: 16 shuffles and one
// store where a reduction per token would take 16 of each.
__device__ __forceinline__ void group_maxima(const GemmArgs& p, int64_t tc, int64_t live,
                                             const float (&val)[16], bool valid, uint32_t n_base,
                                             int lane) {
  uint32_t a[16];
#pragma unroll
  for (int t = 0; t < 16; ++t) a[t] = valid ? logit_order(val[t]) : 0u;
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1) {  // keep w of 2w tokens: lane bit 2w (as a mask) picks the half
    const bool upper = (lane & (2 * w)) != 0;
#pragma unroll
    for (int j = 0; j < w; ++j) {
      const uint32_t mine = upper ? a[j + w] : a[j];
      const uint32_t send = upper ? a[j] : a[j + w];
      a[j] = max(mine, __shfl_xor_sync(0xFFFFFFFFu, send, 2 * w));
    }
  }
  a[0] = max(a[0], __shfl_xor_sync(0xFFFFFFFFu, a[0], 1));
  const int t = (lane >> 1) & 15;
  if ((lane & 1) == 0 && t < live) {
    const int64_t G = (p.N + 31) >> 5;
    p.grp_max[(tc + t) * G + (n_base >> 5)] = a[0];
  }
}

// 16 consecutive floats of shared memory (16-byte aligned)
__device__ __forceinline__ void lds_f32x16(const float* src, float (&d)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 f = reinterpret_cast<const float4*>(src)[i];
    d[4 * i] = f.x;
    d[4 * i + 1] = f.y;
    d[4 * i + 2] = f.z;
    d[4 * i + 3] = f.w;
  }
}

__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// ------------------------------------------------------------ fused top-k
// Per token: a threshold key T (a lower bound of the token's k-th largest
// candidate key, so every one of its k largest logits reaches it), the
// largest candidate order key, a histogram of the candidate groups' largest
// order keys and the candidates themselves: the order key of a logit that
// reached T sits in slot n of the token's N slots (the row is the slot).  Per token and group
// of 32 rows that holds candidates, the warp that owns the group writes
// {largest candidate order key, bitmap of the slots it filled} and sets the
// group's bit in the token's group bitmap (cleared with the histogram by
// the prep kernel): groups without candidates are neither written nor read,
// and the selection skips every group below its final T.
// Histogram bins: all negative keys; positive keys below 2^-32; a
// sixteenth of an octave each from 2^-32 to 2^32 (exponent and top 4
// mantissa bits); 2^32 and above.  The largest candidate of each 32-row
// group with candidates adds one to its bin (one atomic add without a reply
// per group: the counted keys are distinct candidates, and leaving the
// others out only lowers the bin found; counting every candidate within a
// quarter exponent step of its group's largest cost the M = 2048 GEMM 1.48
// against 1.25 ms, for its atomics).  A threshold warp in
// every CTA keeps walking its tokens' bins down from the largest key's bin
// to the one that holds the k-th counted candidate and raises T to that
// bin's lower edge: at least k candidates of the token reach it (counts and
// the maximum only ever lag, which lowers the edge, never invalidates it).
constexpr int kHistBins = 1027;
constexpr int kHistWords = 1028;  // u32 of a token's histogram (whole 16-byte vectors)

// u32 per token of the histogram region: the histogram, then the group
// bitmap (one bit per 32 rows), padded to whole 16-byte vectors.
static inline int topk_hist_stride(int64_t N) {
  const int64_t words = ((N + 31) / 32 + 31) / 32;
  return kHistWords + (int)((words + 3) / 4 * 4);
}

__host__ __device__ __forceinline__ uint32_t topk_bin(uint32_t ok) {
  if (ok < 0x80000000u) return 0u;
  const uint32_t e = (ok >> 23) & 0xFFu;
  if (e < 96u) return 1u;
  if (e >= 160u) return (uint32_t)kHistBins - 1u;
  return 2u + ((e - 96u) << 4) + ((ok >> 19) & 15u);
}
__host__ __device__ __forceinline__ unsigned long long topk_edge(uint32_t bin) {
  uint32_t ok;
  if (bin == 0u) return 0ull;
  if (bin == 1u) ok = 0x80000000u;
  else if (bin == (uint32_t)kHistBins - 1u) ok = 0x80000000u | (160u << 23);
  else ok = 0x80000000u | ((96u + ((bin - 2u) >> 4)) << 23) | (((bin - 2u) & 15u) << 19);
  return (unsigned long long)ok << 32;
}

__device__ __forceinline__ unsigned long long* topk_thr(const GemmArgs& p, int64_t tok) {
  return p.am_keys + tok * kKeyStride;
}
__device__ __forceinline__ uint32_t* topk_max(const GemmArgs& p, int64_t tok) {
  return reinterpret_cast<uint32_t*>(p.am_keys + tok * kKeyStride + 2);
}

__device__ __forceinline__ void red_add_u32(uint32_t* a, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void red_or_u32(uint32_t* a, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.or.b32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void red_max_u32(uint32_t* a, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}

// Raise token `tok`'s threshold to the lower edge of the histogram bin that
// holds its k-th largest counted candidate (whole warp): 32 bins per step,
// downwards from the bin of the largest candidate key.
__device__ __forceinline__ void topk_raise(const GemmArgs& p, int64_t tok, int lane) {
  const uint32_t* h = p.tk_hist + tok * p.tk_hstride;
  int hi = (int)topk_bin(__ldcg(topk_max(p, tok)));
  uint32_t need = (uint32_t)p.tk_k;
#pragma unroll 1
  for (; hi >= 0; hi -= 32) {
    const int bin = hi - lane;
    const uint32_t c = bin >= 0 ? __ldcg(h + bin) : 0u;
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    const uint32_t hit = __ballot_sync(0xFFFFFFFFu, incl >= need);
    if (hit) {
      if (lane == 0) atomicMax(topk_thr(p, tok), topk_edge((uint32_t)(hi - (__ffs(hit) - 1))));
      return;
    }
    need -= __shfl_sync(0xFFFFFFFFu, incl, 31);
  }
}

// The threshold warp of a CTA: tokens blockIdx.x, + gridDim.x, ... (below
// M), one raise each per sweep, until the CTA's four epilogue warps have
// counted themselves out in *epi_done (or a time limit passes).
__device__ __forceinline__ void topk_threshold_role(const GemmArgs& p, volatile int32_t* epi_done,
                                                    int lane) {
  // the histograms, maxima and thresholds are cleared by the prep kernel,
  // which may still be running: nothing is read before it has finished
  grid_dependency_wait();
  if ((int64_t)blockIdx.x >= p.M) return;
  const uint64_t t0 = globaltimer_ns();
  while (*epi_done < 4) {
    for (int64_t tok = blockIdx.x; tok < p.M; tok += gridDim.x) topk_raise(p, tok, lane);
    if (globaltimer_ns() - t0 > 4 * kWaitLimitNs) return;
    __nanosleep(500);
  }
}

// One chunk of 16 tokens (token rows tc .. tc + 15) x the warp's 32 rows
// (n = n_base + lane): where some row reached its token's threshold, the
// candidates, their histogram counts and each token's maximum; then the
// group words (lane t < 16 owns token t's).  The epilogue shares its SM
// sub-partitions with the dequant warps, so what counts is instructions:
// one vote per token, and the rest only for the tokens that have
// candidates (a warp-uniform branch).
__device__ __forceinline__ void topk_chunk(const GemmArgs& p, int64_t tc, int64_t t_end,
                                           const float (&val)[16], const float (&thr)[16],
                                           bool valid, bool any, uint32_t n_base, int lane) {
  uint32_t my_bal = 0, my_mx = 0;
  if (any) {
    const uint32_t n = n_base + (uint32_t)lane;
    const int64_t live = t_end - tc;  // tokens of the chunk below t_end
    uint32_t b[16];
#pragma unroll
    for (int t = 0; t < 16; ++t)
      b[t] = __ballot_sync(0xFFFFFFFFu, valid && t < live && !(val[t] < thr[t]));
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      if (b[t] == 0u) continue;  // warp-uniform
      const bool mine = (b[t] >> lane) & 1u;
      const uint32_t ok = order_key(val[t]);
      const uint32_t mx = __reduce_max_sync(0xFFFFFFFFu, mine ? ok : 0u);
      if (lane == t) {
        my_bal = b[t];
        my_mx = mx;
      }
      // every in-range lane of an 8-row segment that holds a candidate
      // stores, 0 where it holds none (a slot the selection never reads):
      // the 32-byte sector is written whole, so L2 need not fetch the rest
      // of it from DRAM before writing it back
      if (valid && ((b[t] >> (lane & 24)) & 0xFFu) != 0u)
        p.tk_cand[(tc + t) * p.N + n] = mine ? ok : 0u;
    }
    if (my_bal) {  // lane t < 16, live tokens only: the group's largest candidate is counted
      red_max_u32(topk_max(p, tc + lane), my_mx);
      red_add_u32(p.tk_hist + (tc + lane) * p.tk_hstride + topk_bin(my_mx), 1u);
    }
  }
  // lane t < 16 holds token t's group word (my_bal != 0: live token with candidates)
  if (my_bal) {
    const int64_t my_tok = tc + lane;
    const uint32_t g = n_base >> 5;
    p.tk_grp[my_tok * p.tk_groups + g] = make_uint2(my_mx, my_bal);
    red_or_u32(p.tk_hist + my_tok * p.tk_hstride + kHistWords + (g >> 5), 1u << (g & 31));
  }
}

// The prep kernels' clearing of token m's argmax / top-k state (thread
// `tid` of `nthreads` working on the token): the line's maximum or
// threshold and the largest candidate key, and the top-k histogram and
// group bitmap (hstride u32, a multiple of 4).
__device__ __forceinline__ void token_state_clear(unsigned long long* am_keys, uint32_t* tk_hist,
                                                  int hstride, int64_t m, int tid, int nthreads) {
  if (am_keys && tid == 0) {
    am_keys[m * kKeyStride] = 0ull;
    am_keys[m * kKeyStride + 2] = 0ull;
  }
  if (tk_hist) {
    uint4* h = reinterpret_cast<uint4*>(tk_hist + m * hstride);
    for (int i = tid; i < hstride / 4; i += nthreads) h[i] = make_uint4(0, 0, 0, 0);
  }
}

// ------------------------------------------------------------ schedule
// A CTA's work is a list of pieces (a unit, or the part of a unit inside the
// CTA's tail range): first n_dp whole units in strided waves (so that at any
// time the CTAs stream neighbouring weight tiles and the same activation
// stages), then an even share of the remaining units' stages (stream-K).
// Every role walks the same list.
struct Piece {
  uint32_t u, kb0, kb1;
};

// First stage of CTA c's tail range, relative to the tail (c in [0, grid]):
// a split whose density falls linearly from (64 + a) / 64 of the mean at CTA
// 0 to (64 - a) / 64 at the last CTA (a = sc.tail_skew; 0: even), so that
// the CTAs that start later take fewer stages.
__host__ __device__ __forceinline__ uint64_t tail_bound(uint64_t tail_len, uint64_t grid,
                                                        uint64_t skew, uint64_t c) {
  return tail_len * (c * ((64 + skew) * grid - skew * c)) / (64 * grid * grid);
}

template <typename F>
__device__ __forceinline__ void for_each_piece(const Sched& sc, uint32_t n_kb, F&& body) {
  if (blockIdx.x >= sc.grid) return;
  for (uint32_t j = 0; j < sc.n_dp; ++j) {
    const uint32_t u = blockIdx.x + j * sc.grid;
    if (u >= sc.units_end) break;
    if (!body(Piece{u, 0u, n_kb})) return;
  }
  const uint64_t t0 = sc.tail_s0 + tail_bound(sc.tail_len, sc.grid, sc.tail_skew, blockIdx.x);
  const uint64_t t1 = sc.tail_s0 + tail_bound(sc.tail_len, sc.grid, sc.tail_skew, blockIdx.x + 1);
  for (uint64_t s = t0; s < t1;) {
    const uint32_t u = (uint32_t)(s / n_kb), kb0 = (uint32_t)(s - (uint64_t)u * n_kb);
    const uint32_t kb1 = (uint32_t)(((uint64_t)kb0 + (t1 - s) < n_kb) ? kb0 + (t1 - s) : n_kb);
    s += kb1 - kb0;
    if (!body(Piece{u, kb0, kb1})) return;
  }
}

template <typename F>
__device__ __forceinline__ void for_each_piece(const GemmArgs& p, F&& body) {
  for_each_piece(plain_sched(p), (uint32_t)p.n_kb, body);
}

__device__ __forceinline__ uint32_t cta_stages(const Sched& sc, uint32_t n_kb) {
  if (blockIdx.x >= sc.grid) return 0;
  const uint32_t waves =
      sc.units_end > blockIdx.x ? min(sc.n_dp, (sc.units_end - blockIdx.x + sc.grid - 1) / sc.grid) : 0u;
  const uint64_t t0 = tail_bound(sc.tail_len, sc.grid, sc.tail_skew, blockIdx.x);
  const uint64_t t1 = tail_bound(sc.tail_len, sc.grid, sc.tail_skew, blockIdx.x + 1);
  return (uint32_t)((uint64_t)waves * n_kb + (t1 - t0));
}

// ------------------------------------------------------------ epilogue
// The epilogue role: four warps, warp % 4 = the TMEM lane quadrant it may
// read, one thread per vocabulary row of the unit.  Per piece: the token
// multipliers (and argmax thresholds) are fetched before the accumulator is
// ready; then 16 tokens at a time are drained from TMEM, combined with the
// other CTA's partial where a unit was split, scaled (token multiplier, then
// the row's own scale for fp8 weights) and stored, or reduced to per-token
// candidates (argmax, top-k).  `epi` is the warp's index among the four.
// kTokStride: floats per epilogue warp in s_tok / s_thr (>= the token tile)
template <int kOut, bool kRowScale, bool kGrouped = false, int kTokStride = kMaxBN>
__device__ __forceinline__ void epilogue_role(const GemmArgs& p, const Sched& sc, int warp, int epi,
                                              int lane, uint32_t tmem_base, uint64_t* d_full,
                                              uint64_t* d_empty, const WaitCtl& wc,
                                              float* s_tok, float* s_thr) {
  grid_dependency_wait();  // token multipliers and split flags come from the prep kernel
  const int BN = p.BN;
  const int n_kb = p.n_kb;
  const int q = warp & 3;
  const int row = q * 32 + lane;
  const uint32_t lane_off = (uint32_t)(q * 32) << 16;
  float* tok = s_tok + epi * kTokStride;
  float* wthr = s_thr + epi * kTokStride;
  int64_t i = 0;
  for_each_piece(sc, (uint32_t)n_kb, [&](const Piece& pc) {
    const uint32_t u = pc.u, kb0 = pc.kb0, kb1 = pc.kb1;
    const uint32_t buf = (uint32_t)(i & ((1 << p.dbuf_log2) - 1));
    const uint32_t dph = (uint32_t)((i >> p.dbuf_log2) & 1);
    ++i;
    const UnitGeom geo = unit_geom<kGrouped>(p, sc, u, (uint32_t)(i - 1));
    const int64_t n = geo.n0 + row;
    const int64_t t0 = geo.t0;
    const int64_t t_end = geo.t_end;
    // Before the accumulators are ready: this unit's token multipliers,
    // once per warp (written by the prep kernel, which may still have been
    // running when this kernel started, so read coherently from L2, not
    // the read-only path) and, for argmax, each token's current maximum
    // as a threshold (top-k: the value part of its threshold key; a stale
    // one is only lower; none yet: -Inf; tokens past M: +Inf, nothing
    // passes).
    for (int t = lane; t < BN; t += 32) {
      const bool live = t0 + t < t_end;
      tok[t] = live ? __ldcg(p.tok_scale + t0 + t) : 0.0f;
      if (kOut == kOutArgmax || kOut == kOutTopk) {
        const uint32_t kh =
            live ? __ldcg(reinterpret_cast<const uint32_t*>(p.am_keys + (t0 + t) * kKeyStride) + 1)
                 : 0u;
        wthr[t] = !live ? __int_as_float(0x7F800000)
                        : (kh ? key_value(kh) : __int_as_float(0xFF800000));
      }
    }
    // the vocabulary row's own scale (fp8 weights), written before this grid began
    const float rs = kRowScale ? (n < p.N ? __ldg(p.row_scale + n) : 0.0f) : 1.0f;
    __syncwarp();
    if (!warp_wait(&d_full[buf], dph, wc)) return false;
    tc_fence_after();
    if (kOut == kOutTopk && i <= 2) {
      // top-k thresholds rise fastest while the first units' accumulators
      // fill: for those, read them again
      for (int t = lane; t < BN; t += 32) {
        if (t0 + t < t_end) {
          const uint32_t kh = __ldcg(
              reinterpret_cast<const uint32_t*>(p.am_keys + (t0 + t) * kKeyStride) + 1);
          if (kh) wthr[t] = key_value(kh);
        }
      }
      __syncwarp();
    }
    // A tail unit cut by a range boundary: its two CTAs share slot `key`
    // (the CTA whose tail range starts inside the unit).  The first to get here parks
    // its fp32 partial; the second adds it to its own and stores logits.
    // fp32 addition is commutative, so the result does not depend on which
    // CTA comes second.
    const bool whole = kb0 == 0 && kb1 == (uint32_t)n_kb;
    bool finish = true;
    float* part = nullptr;
    uint32_t slot = 0;
    if (!whole) {
      const uint32_t key = kb0 == 0 ? blockIdx.x + 1 : blockIdx.x;
      slot = key * 4 + q;
      part = p.split_part + (size_t)slot * BN * 32;
      uint32_t first = 0;
      if (lane == 0) first = atomicAdd(p.split_cnt + slot, 1u) == 0u;
      finish = __shfl_sync(0xFFFFFFFFu, first, 0) == 0u;
      if (finish && !spin_until_set(p.split_ready + slot, wc)) finish = false;
    }
    for (int c = 0; c < BN; c += 16) {
      uint32_t v[16];
      tmem_ld16(tmem_base + lane_off + buf * BN + c, v);
      tc_wait_ld();
      if (!whole && !finish) {
        // park this partial: token-major, so a warp's 32 rows are one line
#pragma unroll
        for (int t = 0; t < 16; ++t) part[(c + t) * 32 + lane] = __uint_as_float(v[t]);
        continue;
      }
      if (!whole) {
        // the other CTA's partial for these 16 tokens: all loads first, so
        // they are in flight together (the logits stores below could alias)
        float other[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) other[t] = __ldcg(part + (c + t) * 32 + lane);
#pragma unroll
        for (int t = 0; t < 16; ++t)
          v[t] = __float_as_uint(__fadd_rn(__uint_as_float(v[t]), other[t]));
      }
      if (kOut == kOutTopk) {
        // the logits as for argmax; one vote per chunk on the thresholds,
        // then the bitmap words and the candidates
        const bool valid = n < p.N;
        float thr[16], mul[16], val[16];
        lds_f32x16(wthr + c, thr);
        lds_f32x16(tok + c, mul);
        bool pass = false;
#pragma unroll
        for (int t = 0; t < 16; t += 2) {
          float2 r = __ffma2_rn(make_float2(__uint_as_float(v[t]), __uint_as_float(v[t + 1])),
                                make_float2(mul[t], mul[t + 1]), make_float2(0.0f, 0.0f));
          if (kRowScale) r = __fmul2_rn(r, make_float2(rs, rs));
          val[t] = r.x;
          val[t + 1] = r.y;
          pass |= !(r.x < thr[t]);
          pass |= !(r.y < thr[t + 1]);
        }
        topk_chunk(p, t0 + c, t_end, val, thr, valid, __any_sync(0xFFFFFFFFu, valid && pass),
                   (uint32_t)(n - lane), lane);
      } else if (kOut == kOutArgmax) {
        // The logits as the plain product rounds them (the fma with +0
        // rounds like the multiply and turns an exact -0 into +0), then one
        // vote: does any row of this warp reach the threshold of its token
        // (>=, so that ties and NaN reach the exact comparison)?  Only then,
        // per such token, the warp finds its largest key and the lowest lane
        // holding it and merges that candidate with one atomic maximum.
        const bool valid = n < p.N;
        const uint32_t n_base = (uint32_t)(n - lane);
        float thr[16], mul[16], val[16];
        lds_f32x16(wthr + c, thr);
        lds_f32x16(tok + c, mul);
        bool pass = false;
#pragma unroll
        for (int t = 0; t < 16; t += 2) {
          float2 r = __ffma2_rn(make_float2(__uint_as_float(v[t]), __uint_as_float(v[t + 1])),
                                make_float2(mul[t], mul[t + 1]), make_float2(0.0f, 0.0f));
          if (kRowScale) r = __fmul2_rn(r, make_float2(rs, rs));
          val[t] = r.x;
          val[t + 1] = r.y;
          pass |= !(r.x < thr[t]);
          pass |= !(r.y < thr[t + 1]);
        }
        if (__any_sync(0xFFFFFFFFu, valid && pass)) {
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            if (__any_sync(0xFFFFFFFFu, valid && !(val[t] < thr[t]))) {
              const uint32_t kk = valid ? order_key(val[t]) : 0u;
              const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, kk);
              const uint32_t bal = __ballot_sync(0xFFFFFFFFu, valid && kk == m);
              if (lane == 0)
                atomicMax(p.am_keys + (t0 + c + t) * kKeyStride,
                          ((unsigned long long)m << 32) |
                              (uint32_t)~(n_base + (uint32_t)(__ffs(bal) - 1)));
            }
          }
        }
      } else if (kOut == kOutLogitsGroups) {
        // the fp32 logits as below, then the maxima of the warp's group
        const bool valid = n < p.N;
        float mul[16], val[16];
        lds_f32x16(tok + c, mul);
#pragma unroll
        for (int t = 0; t < 16; t += 2) {
          float2 r = __fmul2_rn(make_float2(__uint_as_float(v[t]), __uint_as_float(v[t + 1])),
                                make_float2(mul[t], mul[t + 1]));
          if (kRowScale) r = __fmul2_rn(r, make_float2(rs, rs));
          val[t] = r.x;
          val[t + 1] = r.y;
        }
        const int64_t tc = t0 + c;
        const int64_t live = t_end - tc;
        if (valid) {
          float* ptr = reinterpret_cast<float*>(p.out) + tc * p.N + n;
#pragma unroll
          for (int t = 0; t < 16; ++t, ptr += p.N)
            if (t < live) *ptr = val[t];
        }
        if (n - lane < p.N) group_maxima(p, tc, live, val, valid, (uint32_t)(n - lane), lane);
      } else if (n < p.N) {
        // token multipliers by vector loads, scaled in pairs (each lane of
        // the packed multiply rounds like the scalar one), one store per
        // token walking down the column; a full chunk needs no predicate
        float mul[16], val[16];
        lds_f32x16(tok + c, mul);
#pragma unroll
        for (int t = 0; t < 16; t += 2) {
          float2 r = __fmul2_rn(make_float2(__uint_as_float(v[t]), __uint_as_float(v[t + 1])),
                                make_float2(mul[t], mul[t + 1]));
          if (kRowScale) r = __fmul2_rn(r, make_float2(rs, rs));
          val[t] = r.x;
          val[t + 1] = r.y;
        }
        const int64_t tc = t0 + c;
        const int64_t live = t_end - tc;  // tokens of this chunk inside the group
        using OutT = typename std::conditional<kOut == NVFP4_OUT_BF16, __nv_bfloat16, float>::type;
        OutT* ptr = reinterpret_cast<OutT*>(p.out) + tc * p.N + n;
        if (live >= 16) {
#pragma unroll
          for (int t = 0; t < 16; ++t, ptr += p.N) {
            if constexpr (kOut == NVFP4_OUT_BF16) *ptr = __float2bfloat16_rn(val[t]);
            else *ptr = val[t];
          }
        } else {
#pragma unroll
          for (int t = 0; t < 16; ++t, ptr += p.N) {
            if (t < live) {
              if constexpr (kOut == NVFP4_OUT_BF16) *ptr = __float2bfloat16_rn(val[t]);
              else *ptr = val[t];
            }
          }
        }
      }
    }
    if (!whole && !finish) {
      __threadfence();  // the partial is visible before the flag
      __syncwarp();
      if (lane == 0) atomicExch(p.split_ready + slot, 1u);
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&d_empty[buf]);
    return true;
  });
}

// After every role of the CTA is done (call from all threads, after the
// block barrier that follows the roles): the last CTA to finish turns the
// per-token maxima into rows and values.
__device__ __forceinline__ void argmax_finish(const GemmArgs& p, int first_epi_thread,
                                              int32_t* s_last) {
  // Every candidate of this CTA has been merged (the atomics precede the
  // caller's barrier); the release-acquire counter orders the other CTAs'
  // atomics before the last CTA's reads.
  if ((int)threadIdx.x == first_epi_thread) {
    uint32_t old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;"
                 : "=r"(old) : "l"(p.am_done) : "memory");
    *s_last = old == gridDim.x - 1 ? 1 : 0;
  }
  __syncthreads();
  if (*s_last) {
    for (int64_t t = threadIdx.x; t < p.M; t += blockDim.x) {
      const unsigned long long k = __ldcg(p.am_keys + t * kKeyStride);
      p.am_idx[t] = k != 0ull ? (int64_t)(uint32_t)~(uint32_t)k : (int64_t)-1;
      if (p.am_val) p.am_val[t] = key_value((uint32_t)(k >> 32));
    }
  }
}

// ------------------------------------------------------------ host side
// Raise a kernel's dynamic shared memory limit on the current device, once
// per device (the attribute belongs to the device's context).  `done` is the
// launch site's own record of the devices already set.
static inline cudaError_t smem_limit_once(std::atomic<uint64_t>& done, const void* kern,
                                          size_t bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? 1ull << dev : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

static inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

static inline bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base,
                             uint64_t inner, uint64_t outer, uint64_t row_bytes,
                             uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static inline int lm_head_token_tile(int64_t M) {
  if (M >= kMaxBN) return kMaxBN;
  return (int)((M + 15) / 16 * 16);
}

static inline int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

// How a product's activations sit in its workspace (the first region after
// the status header): fp16 [m_pad, K] (W4A16), e4m3 [m_pad, K] (W8A8), or
// e2m1 codes [m_pad, row stride] followed by their 128x4-interleaved block
// scales (W4A4).  K % 16 == 0 in all three.
enum class ActFormat { kF16, kE4M3, kE2M1 };

// Row stride of the W4A4 x codes in the workspace: K/2 bytes rounded up to
// the 16-byte multiple a TMA row stride needs.
static inline int64_t e2m1_code_stride(int64_t K) { return (K / 2 + 15) / 16 * 16; }

// Columns of a 128x4-interleaved block-scale matrix: K/16 rounded up to 4.
static inline int64_t interleaved_sf_cols(int64_t K) { return (K / 16 + 3) / 4 * 4; }

static inline size_t act_region_bytes(ActFormat f, int64_t m_pad, int64_t M, int64_t K) {
  switch (f) {
    case ActFormat::kF16: return (size_t)m_pad * K * 2;
    case ActFormat::kE4M3: return (size_t)m_pad * K;
    case ActFormat::kE2M1:
      return align_up((size_t)m_pad * e2m1_code_stride(K), 256) +
             (size_t)((M + 127) / 128 * 128) * interleaved_sf_cols(K);
  }
  return 0;
}

// Workspace layout of one call: [status header][activations as the MMA
// reads them (ActFormat)]
// [token multipliers, m_pad][split counters, grid x 4][split ready flags,
// grid x 4] and, for argmax and top-k, [CTAs done, 1]; these are zeroed by
// the prep kernel's first CTA.  Then [split partials, grid x 4 x BN x 32
// fp32] and, for argmax and top-k, [per-token state, m_pad x 128 bytes: the
// maximum or the threshold key in word 0, the largest top-k candidate order
// key in word 2], both words zeroed by the prep CTA of the token.  Top-k
// only: [histograms and group bitmaps, m_pad x topk_hist_stride(N) u32,
// zeroed the same way][candidate groups, M x ceil(N / 32) x 8 bytes, written
// by the GEMM only where its bitmap bit is set][candidates, M x N u32 order
// keys, read only where the group words say].
struct WsLayout {
  size_t x16, tok, cnt, ready, done, keys, part, hist, grp, cand, total;
  int grid;
};


// bn: the call's token tile when it is not lm_head_token_tile(M)
static inline WsLayout ws_layout(int64_t M, int64_t N, int64_t K, int sms, bool argmax,
                                 ActFormat act, int topk_k = 0, int bn = 0) {
  WsLayout l;
  const bool keys = argmax || topk_k > 0;
  const int BN = bn > 0 ? bn : lm_head_token_tile(M);
  const int64_t m_pad = (M + BN - 1) / BN * BN;
  const int64_t n_units = ((N + kRows - 1) / kRows) * ((M + BN - 1) / BN);
  l.grid = (int)std::max<int64_t>(1, std::min<int64_t>(sms, n_units));
  l.x16 = kWsHeader;
  l.tok = l.x16 + align_up(act_region_bytes(act, m_pad, M, K), 1024);
  l.cnt = l.tok + align_up((size_t)m_pad * 4, 256);
  l.ready = l.cnt + align_up((size_t)l.grid * 4 * 4, 256);
  l.done = l.ready + align_up((size_t)l.grid * 4 * 4, 256);
  l.part = l.done + (keys ? 256 : 0);
  l.keys = l.part + align_up((size_t)l.grid * 4 * BN * 32 * 4, 256);
  l.hist = l.keys + (keys ? (size_t)m_pad * kKeyStride * 8 : 0);
  l.grp = l.hist + (topk_k > 0 ? (size_t)m_pad * topk_hist_stride(N) * 4 : 0);
  l.cand = l.grp + (topk_k > 0 ? align_up((size_t)M * ((N + 31) / 32) * 8, 256) : 0);
  l.total = l.cand + (topk_k > 0 ? (size_t)M * N * 4 : 0);
  return l;
}

// Weight rows whose byte length is not a 16-byte multiple cannot be read by
// TMA in place (a tensor map's row stride must be one): such a matrix is
// copied, row for row, into the workspace with the stride rounded up, and
// the TMA zero-fills everything past the row's real length.  NVFP4 codes
// [rows, K/2] need the copy when K % 32 != 0, block scales [rows, K/16] when
// K % 256 != 0.  `off` is where the copies start (after the call's other
// regions); a copy absent for this K has size 0.
struct WeightStage {
  size_t packed_off, packed_stride, scales_off, scales_stride, total;
  bool packed, scales;
};

static inline int64_t round_up16(int64_t v) { return (v + 15) / 16 * 16; }

static inline WeightStage weight_stage(int64_t rows, int64_t K, size_t off, bool with_scales) {
  WeightStage w;
  w.packed = (K / 2) % 16 != 0;
  w.scales = with_scales && (K / 16) % 16 != 0;
  w.packed_stride = (size_t)round_up16(K / 2);
  w.scales_stride = (size_t)round_up16(K / 16);
  w.packed_off = align_up(off, 256);
  const size_t after_packed = w.packed_off + (w.packed ? align_up(rows * w.packed_stride, 256) : 0);
  w.scales_off = after_packed;
  w.total = w.scales_off + (w.scales ? align_up(rows * w.scales_stride, 256) : 0);
  return w;
}

// Launch the row copy (lm_head.cu) as a programmatic dependent of the
// previous kernel in the stream: `rows` rows of `row_bytes` bytes, read back
// to back from `src`, written `dst_stride` bytes apart (a 16-byte multiple).
cudaError_t stage_rows_launch(const uint8_t* src, int64_t rows, int64_t row_bytes, uint8_t* dst,
                              int64_t dst_stride, cudaStream_t stream);

// Up to this many tokens a top-k call writes the fp32 logits (at most
// 256 x N x 4 bytes, under half the weight bytes of a 4096-wide head) and
// the per-token maxima of every 32 rows, and selects from them (topk.cu,
// topk_logits_launch); beyond, the GEMM keeps thresholded candidates in its
// epilogue and topk_select_launch picks from those, so that a prefill never
// writes its logits.  (Same-box, k = 50 over 128256 rows: the candidate
// route took 104 / 123 / 149 / 243 us at 65 / 96 / 128 / 256 tokens
// against 73 / 81 / 96 / 171 us for the fp32 logits alone.)
constexpr int64_t kTopkLogitsMaxM = 256;
// The selecting CTA holds a token's group maxima in registers: vocabularies
// up to this many rows take the logits route.
constexpr int64_t kTopkLogitsMaxN = 32 * 8192;

// Workspace of the logits route after a call's own layout ending at `base`:
// [fp32 logits, M x N][u32 group maxima, M x ceil(N / 32)].
struct TopkLogitsLayout {
  size_t logits, gmax, total;
};
static inline TopkLogitsLayout topk_logits_layout(size_t base, int64_t M, int64_t N) {
  TopkLogitsLayout t;
  t.logits = align_up(base, 256);
  t.gmax = align_up(t.logits + (size_t)M * N * 4, 256);
  t.total = t.gmax + (size_t)M * ((N + 31) / 32) * 4;
  return t;
}

cudaError_t topk_logits_launch(const float* logits, const uint32_t* gmax, int64_t M, int64_t N,
                               int k, int64_t* ids, float* vals, cudaStream_t stream);
static inline bool topk_logits_fits(int64_t N) { return N <= kTopkLogitsMaxN; }

// The top-k selection kernel (topk.cu), launched after a top-k GEMM.
cudaError_t topk_select_launch(const unsigned long long* lines, const uint2* grp,
                               const uint32_t* cand, const uint32_t* hist, int hstride, int64_t M,
                               int64_t N, int k, int64_t* ids, float* vals, cudaStream_t stream);

// The top-k arguments of a GEMM whose workspace follows layout L.
static inline void topk_args(GemmArgs& a, uint8_t* ws, const WsLayout& L, int k, int64_t N) {
  a.tk_cand = reinterpret_cast<uint32_t*>(ws + L.cand);
  a.tk_hist = reinterpret_cast<uint32_t*>(ws + L.hist);
  a.tk_grp = reinterpret_cast<uint2*>(ws + L.grp);
  a.tk_groups = (N + 31) / 32;
  a.tk_hstride = topk_hist_stride(N);
  a.tk_k = k;
}

// Split the units of a call into strided whole-unit waves and a stream-K
// tail: all but the last one to two waves run whole; the rest is split
// evenly, so every CTA's tail range holds at least one unit's stages and a
// unit is cut at most once.
static inline void schedule_units(GemmArgs& a, int64_t grid, uint32_t max_skew = 0) {
  const int64_t dp_waves = a.n_units >= 2 * grid ? a.n_units / grid - 1 : 0;
  a.n_dp = (uint32_t)dp_waves;
  a.tail_s0 = (uint64_t)(dp_waves * grid) * a.n_kb;
  a.tail_len = (uint64_t)(a.n_units - dp_waves * grid) * a.n_kb;
  // the largest skew up to max_skew that leaves every CTA's tail range at
  // least one unit long (so that a unit is still cut at most once)
  a.tail_skew = 0;
  for (uint32_t s = max_skew; s > 0; --s) {
    bool ok = true;
    for (int64_t c = 0; c < grid && ok; ++c)
      ok = tail_bound(a.tail_len, grid, s, c + 1) - tail_bound(a.tail_len, grid, s, c) >=
           (uint64_t)a.n_kb;
    if (ok) {
      a.tail_skew = s;
      break;
    }
  }
}

// Launch configuration of a programmatic dependent launch.
struct PdlLaunch {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg;
  PdlLaunch(dim3 grid, dim3 block, size_t smem, cudaStream_t stream) : cfg{} {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
};

}  // namespace nvfp4
