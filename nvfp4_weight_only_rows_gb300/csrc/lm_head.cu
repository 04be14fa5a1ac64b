// lm_head.cu -- the weight-only W4A16 lm_head product on sm_103a tensor cores.
//
// logits[m, n] = global * sum_k x[m, k] * e2m1(code[n, k]) * f32(scale[n, k/16])
// (`CompressedTensorsW4A16Fp4.apply_weights` on the page
// "vllm.model_executor.layers.quantization.compressed_tensors.schemes", with
// the checkpoint layout `_quantize_nvfp4` writes on the page
// "vllm.model_executor.layers.quantization.online.lm_head").
//
// Two kernels per call (the second launched as a programmatic dependent of
// the first, so it streams weights while the first finishes):
//  1. w4a16_prep_x_kernel: each token row of x (bf16) is rescaled by an
//     exact power of two 2^e so that its largest magnitude lands in
//     [2^14, 2^15), and stored as fp16 in the workspace; the token's output
//     multiplier global * 2^-e is stored beside it.  fp16 holds every bf16
//     value of that row exactly down to 2^-28 of the row maximum.
//  2. w4a16_tc_kernel: a persistent, warp-specialized tcgen05 GEMM in the
//     swapped orientation D[vocab row, token] = A . B^T:
//       A = dequantized weights, 128 vocabulary rows x 256 k per stage, held
//           in TENSOR MEMORY (the "ts" MMA form), written by eight dequant
//           warps with one thread per row and half a stage per warp: e2m1
//           pairs -> fp16 pairs with the hardware cvt, times the E4M3 block
//           scale (fp16, exact);
//       B = the fp16 activations, four TMA boxes [BN tokens x 64 k] per
//           stage in shared memory with the 128-byte swizzle;
//       D = fp32 accumulators in tensor memory, double buffered, drained by
//           four epilogue warps (tcgen05.ld, x token multiplier, store).
//     Packed codes and scales arrive by TMA in 256-k stages; every product
//     x * w is exact in fp32, so the only rounding is the fp32 summation.
//
// Warp roles (480 threads): 0 packed/scale TMA producer, 1 activation TMA
// producer, 2 MMA issuer (and TMEM owner), 3-10 dequant (two warps per TMEM
// lane quadrant taking 256-k stages in turn), 11-14 epilogue.  The producer
// and MMA warps run warp-uniform loops and issue from one elected lane.
// Every pipeline wait is bounded in time; on expiry the CTA raises
// NVFP4_ERR_TIMEOUT in the workspace status word, drains what it issued and
// returns.
#include <cuda_fp16.h>

#include "gemm_common.cuh"

namespace nvfp4 {

constexpr int kKS = 256;            // k per packed/scale stage
constexpr int kFirstDqWarp = 3;

// Ring depths and the number of dequant warps per TMEM lane quadrant are
// template parameters of the GEMM:
//   token tiles of up to 64 (decode): 3 A/activation stages, 6 packed
//     stages, 3 warps per quadrant (TMEM: 2 x 64 accumulator columns +
//     3 x 128 A columns = 512);
//   token tiles of 128 (prefill): 2 A/activation stages, 4 packed stages,
//     2 warps per quadrant.
// A dequant warp takes every kDq-th stage.  An mbarrier parity wait for
// phase j is only sound once phase j-1 has completed; the warp itself has
// checked that for the slot's previous use only if that use was one of its
// own stages, i.e. if kDq divides the ring depth.
template <int kStages, int kPStages, int kDq>
struct GemmShape {
  static_assert(kStages % kDq == 0 && kPStages % kDq == 0,
                "dequant warps per quadrant must divide every ring depth they wait on");
  static constexpr int kDqWarps = 4 * kDq;
  static constexpr int kFirstEpiWarp = kFirstDqWarp + kDqWarps;
  static constexpr int kThreads = 32 * (kFirstEpiWarp + 4);
};
constexpr uint32_t kPackedStageBytes = kRows * (kKS / 2);   // 16384
constexpr uint32_t kScaleStageBytes = kRows * (kKS / 16);   // 2048


// The plain product's stream-K tail gives the CTAs of higher index (which
// enter later: the first MMA of a decode call comes 2.8 to 5.6 us after the
// first CTA's entry, correlated 0.8 with the index at M = 64) fewer stages,
// up to 4/64 of the mean less (the skew bound passed to schedule_units).
// Same box, the four decode calls M = 1, 8, 32, 64: 224.4 -> 223.5 us; M = 8
// alone 52.8 -> 51.7 us; a skew of 8 gave 224.6 us, of 12 227.1 us.
constexpr uint32_t kDecodeTailSkew = 4;

// ------------------------------------------------------------ activations
// kWarpsPerRow warps per token row (4, with a 128-thread CTA per row, for
// few rows, where the latency of one row is what counts and the CTA must
// fit beside a GEMM CTA on its SM; 1: a warp per row, 8 rows per 256-thread
// CTA, for many rows); rows m_rows and beyond do not exist, rows
// M .. m_rows-1 are zero padding.
template <int kWarpsPerRow>
__global__ void __launch_bounds__(256) w4a16_prep_x_kernel(const uint16_t* __restrict__ x,
                                                           int64_t M, int64_t K, int64_t m_rows,
                                                           const float* __restrict__ global,
                                                           __half* __restrict__ x16,
                                                           float* __restrict__ tok_scale,
                                                           int32_t* __restrict__ status,
                                                           uint32_t* __restrict__ split_flags,
                                                           int n_split_flags,
                                                           unsigned long long* __restrict__ am_keys,
                                                           uint32_t* __restrict__ tk_hist,
                                                           int tk_hstride,
                                                           const int32_t* __restrict__ grp_off,
                                                           const float* __restrict__ grp_global,
                                                           int n_groups) {
  // launched as a programmatic dependent of whatever ran before it: wait for
  // that kernel's results before touching memory (the previous call's GEMM
  // may still be reading this workspace)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the GEMM may launch now: it waits for this grid's results (griddepcontrol.wait)
  // only where it reads them, and streams the weights meanwhile
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (blockIdx.x == 0) {  // a fresh call: clear the status word and the split-K flags
    if (threadIdx.x == 0) *status = NVFP4_OK;
    for (int i = threadIdx.x; i < n_split_flags; i += blockDim.x) split_flags[i] = 0;
  }
  __shared__ int32_t s_grp[kMaxGroups + 1];
  if (grp_off) {  // grouped: the group offsets, loaded by the whole block
    for (int e = threadIdx.x; e <= n_groups; e += blockDim.x) s_grp[e] = grp_off[e];
    __syncthreads();
  }
  constexpr int kT = 32 * kWarpsPerRow;  // threads of one row
  const int lane = threadIdx.x % kT;
  const int64_t m = (int64_t)blockIdx.x * (blockDim.x / kT) + threadIdx.x / kT;
  if (m >= m_rows) return;  // uniform over the row's threads
  token_state_clear(am_keys, tk_hist, tk_hstride, m, lane, kT);  // argmax / top-k: nothing seen yet
  uint4* d4 = reinterpret_cast<uint4*>(x16 + m * K);
  const int64_t nv = K / 8;
  if (m >= M) {  // padding rows of the last token tile
    for (int64_t i = lane; i < nv; i += kT) d4[i] = make_uint4(0, 0, 0, 0);
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(x + m * K);
  uint32_t mx = 0;
  for (int64_t i = lane; i < nv; i += kT) {
    const uint4 v = src[i];
    const uint32_t k = 0x7FFF7FFFu;
    mx = __vmaxu2(mx, v.x & k);
    mx = __vmaxu2(mx, v.y & k);
    mx = __vmaxu2(mx, v.z & k);
    mx = __vmaxu2(mx, v.w & k);
  }
  mx = max(mx & 0xFFFFu, mx >> 16);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  if constexpr (kWarpsPerRow > 1) {  // the CTA is one row: combine its warps
    __shared__ uint32_t red[kWarpsPerRow];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = 0;
    for (int w = 0; w < kWarpsPerRow; ++w) mx = max(mx, red[w]);
  }
  int e = 0;
  if (mx != 0 && mx < 0x7F80u) {
    const int E = ilogbf(__uint_as_float(mx << 16));  // floor(log2(max|x|))
    e = min(max(14 - E, -126), 126);
  }
  if (lane == 0) {
    float gw;
    if (grp_off) {  // grouped: the global of the group holding token row m
      int lo = 0, hi = n_groups;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_grp[mid] <= m) lo = mid; else hi = mid;
      }
      gw = (s_grp[lo] <= m && m < s_grp[lo + 1]) ? grp_global[lo] : 0.0f;
    } else {
      gw = *global;
    }
    tok_scale[m] = __fmul_rn(gw, __int_as_float((127 - e) << 23));
  }
  const float p2 = __int_as_float((127 + e) << 23);
  for (int64_t i = lane; i < nv; i += kT) {
    const uint4 v = src[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = __fmul_rn(__uint_as_float(w[j] << 16), p2);
      const float hi = __fmul_rn(__uint_as_float(w[j] & 0xFFFF0000u), p2);
      __half2 h = __floats2half2_rn(lo, hi);
      o[j] = *reinterpret_cast<uint32_t*>(&h);
    }
    d4[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// ------------------------------------------------------------ weight rows
// Row copy into a TMA-readable stride (see WeightStage): one warp per row,
// in units of T (8 bytes for NVFP4 code rows, which K % 16 makes 8-byte
// multiples; 1 byte for block-scale rows).  Launched as a programmatic
// dependent: the weights may have been written by the kernel before it.
template <typename T>
__global__ void __launch_bounds__(256) stage_rows_kernel(const T* __restrict__ src, int64_t rows,
                                                         int64_t row_elems, T* __restrict__ dst,
                                                         int64_t dst_stride_elems) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows;
       r += warps) {
    const T* s = src + r * row_elems;
    T* d = dst + r * dst_stride_elems;
    for (int64_t j = lane; j < row_elems; j += 32) d[j] = s[j];
  }
}

cudaError_t stage_rows_launch(const uint8_t* src, int64_t rows, int64_t row_bytes, uint8_t* dst,
                              int64_t dst_stride, cudaStream_t stream) {
  const int sms = std::max(sm_count(), 1);
  const int64_t blocks = std::min<int64_t>((rows + 7) / 8, (int64_t)sms * 8);
  PdlLaunch l(dim3((unsigned)std::max<int64_t>(blocks, 1)), dim3(256), 0, stream);
  if (row_bytes % 8 == 0)
    return cudaLaunchKernelEx(&l.cfg, stage_rows_kernel<uint2>,
                              reinterpret_cast<const uint2*>(src), rows, row_bytes / 8,
                              reinterpret_cast<uint2*>(dst), dst_stride / 8);
  return cudaLaunchKernelEx(&l.cfg, stage_rows_kernel<uint8_t>, src, rows, row_bytes, dst,
                            dst_stride);
}

// Stage the weight rows that TMA cannot read in place (both copies are
// no-ops for K % 256 == 0, the usual lm_head width).
static cudaError_t stage_weights(const WeightStage& w, const uint8_t* packed,
                                 const uint8_t* scales, int64_t rows, int64_t K, uint8_t* ws,
                                 cudaStream_t stream) {
  cudaError_t e = cudaSuccess;
  if (w.packed)
    e = stage_rows_launch(packed, rows, K / 2, ws + w.packed_off, (int64_t)w.packed_stride, stream);
  if (e == cudaSuccess && w.scales)
    e = stage_rows_launch(scales, rows, K / 16, ws + w.scales_off, (int64_t)w.scales_stride,
                          stream);
  return e;
}

// Up to this many token rows the prep kernel gives each row a whole CTA.
constexpr int64_t kPrepWideRows = 256;

// ------------------------------------------------------------ dequant helpers
// 8 e2m1 codes (one word; byte j = codes 2j | 2j+1 << 4) -> 4 fp16 pairs,
// element 2j in the low half, each multiplied by the block scale pair sf2.
__device__ __forceinline__ void dequant8(uint32_t w, uint32_t sf2, uint32_t* out) {
  uint32_t h0, h1, h2, h3;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
      : "r"(w));
  asm("mul.rn.f16x2 %0, %0, %4;\n\t"
      "mul.rn.f16x2 %1, %1, %4;\n\t"
      "mul.rn.f16x2 %2, %2, %4;\n\t"
      "mul.rn.f16x2 %3, %3, %4;"
      : "+r"(h0), "+r"(h1), "+r"(h2), "+r"(h3)
      : "r"(sf2));
  out[0] = h0;
  out[1] = h1;
  out[2] = h2;
  out[3] = h3;
}

// 4 E4M3 scale bytes -> two fp16 pairs (s0, s1) and (s2, s3)
__device__ __forceinline__ void scales4_to_f16(uint32_t s, uint32_t& s01, uint32_t& s23) {
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "mov.b32 {lo, hi}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
      : "=r"(s01), "=r"(s23)
      : "r"(s));
}

__device__ __forceinline__ uint32_t dup_lo(uint32_t v) { return __byte_perm(v, 0, 0x1010); }
__device__ __forceinline__ uint32_t dup_hi(uint32_t v) { return __byte_perm(v, 0, 0x3232); }

// ------------------------------------------------------------ the GEMM
// kOut: NVFP4_OUT_F32 / NVFP4_OUT_BF16 store the logits; kOutArgmax keeps
// only each token's largest logit and its vocabulary row; kOutTopk appends
// the candidates for each token's k largest (topk.cu selects them).
// kGrouped: the grouped (experts) product: weight rows e * N + n, token rows
// grouped by the offsets in p.grp_off, one global scale per group.
// Threads of one CTA: the shape's roles, plus the threshold warp in top-k mode.
template <int kOut, int kStages, int kPStages, int kDq>
constexpr int gemm_threads() {
  return GemmShape<kStages, kPStages, kDq>::kThreads + (kOut == kOutTopk ? 32 : 0);
}

template <int kOut, int kStages, int kPStages, int kDqPerQuad, bool kGrouped = false>
__global__ void __launch_bounds__((gemm_threads<kOut, kStages, kPStages, kDqPerQuad>()), 1)
    w4a16_tc_kernel(const __grid_constant__ CUtensorMap tm_packed,
                    const __grid_constant__ CUtensorMap tm_scales,
                    const __grid_constant__ CUtensorMap tm_x, const GemmArgs p) {
  using Shape = GemmShape<kStages, kPStages, kDqPerQuad>;
  constexpr int kFirstEpiWarp = Shape::kFirstEpiWarp;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int BN = p.BN;
  const uint32_t x_box_bytes = (uint32_t)BN * 128;  // one 64-k TMA box of the activations
  const uint32_t x_stage_bytes = (kKB / 64) * x_box_bytes;
  uint8_t* s_packed = smem;                                        // kPStages x 16 KB
  uint8_t* s_scales = s_packed + kPStages * kPackedStageBytes;     // kPStages x 2 KB
  uint8_t* s_x = s_scales + kPStages * kScaleStageBytes;           // kStages x BN*512
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_x + kStages * x_stage_bytes);
  uint64_t* p_full = bars;                 // packed/scale stage landed (TMA)
  uint64_t* p_empty = p_full + kPStages;   // packed/scale stage read by its 4 dequant warps
  uint64_t* s_full = p_empty + kPStages;   // A stage in TMEM (4 warps) + activation TMA landed
  uint64_t* s_empty = s_full + kStages;    // the MMAs reading stage s completed
  uint64_t* d_full = s_empty + kStages;   // accumulator buffer b holds a finished unit
  uint64_t* d_empty = d_full + 4;         // the epilogue has drained buffer b
  uint64_t* done_bar = d_empty + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(tmem_slot + 1);
  float* s_tok = reinterpret_cast<float*>(bars + 32);  // 4 epilogue warps x kMaxBN multipliers
  // argmax: the "last CTA" flag, then per epilogue warp the thresholds of
  // its current unit's tokens (lower bounds of each token's largest logit)
  int32_t* s_last = reinterpret_cast<int32_t*>(s_tok + 4 * kMaxBN);
  float* s_thr = reinterpret_cast<float*>(s_last + 4);
  // grouped: the schedule derived from the group offsets
  Sched* s_sched = reinterpret_cast<Sched*>(s_thr + 4 * kMaxBN);
  uint32_t* s_unit_pre = reinterpret_cast<uint32_t*>(s_sched + 1);
  int32_t* s_off = reinterpret_cast<int32_t*>(s_unit_pre + kMaxGroups + 1);
  uint2* s_grp_tab = reinterpret_cast<uint2*>(s_off + kMaxGroups + 1);  // 8-byte aligned

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if constexpr (kGrouped) {
    grouped_offsets_load(p, s_off);
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kPStages; ++i) {
      mbar_init(&p_full[i], 1);
      mbar_init(&p_empty[i], 4);
    }
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s_full[i], 4 + 1);
      mbar_init(&s_empty[i], 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&d_full[i], 1);
      mbar_init(&d_empty[i], 4);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    if (kOut == kOutTopk) s_last[1] = 0;  // epilogue warps done (the region exists in this mode)
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if constexpr (kGrouped)
    if (warp == 0)
      grouped_sched_build(p, s_sched, s_unit_pre, s_off, s_grp_tab, (uint32_t)p.n_kb, lane);
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_packed);
    tma_prefetch_desc(&tm_scales);
    tma_prefetch_desc(&tm_x);
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, p.tmem_cols);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  // warp-uniform copy of the TMEM base (lets the compiler keep it uniform)
  const uint32_t tmem_base = __shfl_sync(0xFFFFFFFFu, *tmem_slot, 0);
  const uint32_t tmem_a = tmem_base + ((uint32_t)BN << p.dbuf_log2);  // A ring after the D buffers

  WaitCtl wc{p.status, abort_flag, kWaitLimitNs};
  Sched sc;
  if constexpr (kGrouped) sc = *s_sched; else sc = plain_sched(p);
  const uint32_t n_kb_u = (uint32_t)p.n_kb;
  // the producer and MMA loops below are warp-uniform; one elected lane
  // issues each TMA / tcgen05 instruction

  if (warp == 0) {
    // ---------------- packed codes + scales producer
    // a weight tile read once (one token tile) is not kept in L2; one read
    // by several token tiles in a row is
    const uint64_t pol_once = policy_evict_first(), pol_reused = policy_evict_last();
    uint32_t issued = 0, piece = 0;
    for_each_piece(sc, n_kb_u, [&](const Piece& pc) {
      const UnitGeom geo = unit_geom<kGrouped>(p, sc, pc.u, piece++);
      const int32_t n0 = (int32_t)geo.w_row;
      const uint64_t pol = geo.reused ? pol_reused : pol_once;  // packed codes
      for (uint32_t kb = pc.kb0; kb < pc.kb1; ++kb, ++issued) {
        const uint32_t st = issued % kPStages, ph = (issued / kPStages) & 1;
        if (!warp_wait(&p_empty[st], ph ^ 1, wc)) return false;
        if (elect_one()) {
          mbar_arrive_expect_tx(&p_full[st], kPackedStageBytes + kScaleStageBytes);
          tma_load_2d_hint(s_packed + st * kPackedStageBytes, &tm_packed, kb * (kKS / 2), n0,
                           &p_full[st], pol);
          // a stage takes 16 bytes of each 32-byte scale sector, the next
          // stage the other 16: scales read once keep the default policy
          // (evict-first would drop the sector before its second half is read)
          if (geo.reused)
            tma_load_2d_hint(s_scales + st * kScaleStageBytes, &tm_scales, kb * (kKS / 16), n0,
                             &p_full[st], pol_reused);
          else
            tma_load_2d(s_scales + st * kScaleStageBytes, &tm_scales, kb * (kKS / 16), n0,
                        &p_full[st]);
        }
        __syncwarp();
      }
      return true;
    });
    drain_loads(p_full, kPStages, issued, 1, p.status);
  } else if (warp == 1) {
    // ---------------- activation producer (four 64-k boxes per stage)
    grid_dependency_wait();  // the rescaled activations come from the prep kernel
    const uint64_t pol = policy_evict_last();
    uint32_t issued = 0, piece = 0;
    for_each_piece(sc, n_kb_u, [&](const Piece& pc) {
      const int32_t t0 = (int32_t)unit_geom<kGrouped>(p, sc, pc.u, piece++).t0;
      for (uint32_t kb = pc.kb0; kb < pc.kb1; ++kb, ++issued) {
        const uint32_t st = issued % kStages, ph = (issued / kStages) & 1;
        if (!warp_wait(&s_empty[st], ph ^ 1, wc)) return false;
        if (elect_one()) {
          mbar_arrive_expect_tx(&s_full[st], x_stage_bytes);
          uint8_t* dst = s_x + st * x_stage_bytes;
#pragma unroll
          for (int b = 0; b < kKB / 64; ++b)
            tma_load_2d_hint(dst + b * x_box_bytes, &tm_x, kb * kKB + 64 * b, t0, &s_full[st],
                             pol);
        }
        __syncwarp();
      }
      return true;
    });
    drain_loads(s_full, kStages, issued, 5, p.status);
  } else if (warp == 2) {
    // ---------------- MMA issuer (whole warp; one elected lane issues).
    // One accumulator per piece, double buffered.
    const uint32_t idesc = idesc_f16_f32((uint32_t)BN);
    const uint64_t xdesc0 = smem_desc_sw128(smem_u32(s_x));
    const uint32_t box_desc = x_box_bytes >> 4;
    uint32_t g = 0;
    int64_t i = 0;
    for_each_piece(sc, n_kb_u, [&](const Piece& pc) {
      const uint32_t buf = (uint32_t)(i & ((1 << p.dbuf_log2) - 1));
      const uint32_t dph = (uint32_t)((i >> p.dbuf_log2) & 1);
      ++i;
      // grouped 128-token tiles: a group's last, partly filled tile takes MMAs
      // only as wide as its tokens, in 16-token steps (same box, 2048 tokens:
      // w13 134.9 -> 132.5 us, w2 89.2 -> 88.7 us; smaller tiles keep BN)
      uint32_t id = idesc;
      if constexpr (kGrouped) {
        if (BN == kMaxBN) {
          const UnitGeom geo = unit_geom<kGrouped>(p, sc, pc.u, (uint32_t)(i - 1));
          const int64_t live = geo.t_end - geo.t0;
          if (live < BN) id = idesc_f16_f32(live > 0 ? (uint32_t)((live + 15) / 16 * 16) : 16u);
        }
      }
      if (!warp_wait(&d_empty[buf], dph ^ 1, wc)) return false;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + buf * BN;
      for (uint32_t kb = pc.kb0; kb < pc.kb1; ++kb, ++g) {
        const uint32_t st = g % kStages, ph = (g / kStages) & 1;
        if (!warp_wait(&s_full[st], ph, wc)) return false;
        tc_fence_after();
        const uint64_t bdesc = xdesc0 + ((st * x_stage_bytes) >> 4);
        const uint32_t a_t = tmem_a + st * (kKB / 2);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kKB / 16; ++kk)
            tc_mma_ts(d_tmem, a_t + kk * 8, bdesc + (kk >> 2) * box_desc + 2 * (kk & 3), id,
                      (kb != pc.kb0) || (kk != 0));
          tc_commit(&s_empty[st]);
        }
        __syncwarp();
      }
      if (elect_one()) tc_commit(&d_full[buf]);
      __syncwarp();
      return true;
    });
    // this CTA has issued its last MMA: the next kernel in the stream may be
    // launched (it waits for this grid's completion before touching memory)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // every MMA issued above has completed once done_bar flips
    if (elect_one()) tc_commit(done_bar);
    __syncwarp();
    WaitCtl drain{p.status, abort_flag, 100000000ull};
    volatile int32_t zero = 0;
    drain.abort = &zero;
    mbar_wait(done_bar, 0, drain);
  } else if (warp < kFirstEpiWarp) {
    // ---------------- dequant: one thread per vocabulary row.  The kDqPerQuad
    // warps of a TMEM lane quadrant take the 256-k stages in turn: wait for
    // the packed stage, convert 64 k at a time into 32 registers and store
    // them to the stage's TMEM columns, then signal the MMA warp.
    const int q = warp & 3;
    const int r = (warp - kFirstDqWarp) >> 2;
    const int row = q * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const int sw = row & 7;
    // this warp's stages are g = r, r + kDqPerQuad, ... of the CTA's sequence
    const uint32_t total = cta_stages(sc, n_kb_u);
    // NaN block scales (E4M3 S.1111.111: the "never loaded" sentinel of
    // `KNvfp4Static.process` on the page
    // "vllm/model_executor/layers/quantization/modelopt.py"): per byte,
    // (b & 0x7F) + 1 carries into bit 7 only for 0x7F / 0xFF, and never into
    // the next byte; the OR over the CTA's stages is tested once at the end
    uint32_t nan_seen = 0;
    bool ok = true;
    for (uint32_t g = (uint32_t)r; ok && g < total; g += kDqPerQuad) {
      const uint32_t ps = g % kPStages, pph = (g / kPStages) & 1;
      const uint32_t st = g % kStages, ph = (g / kStages) & 1;
      if (!warp_wait(&p_full[ps], pph, wc)) { ok = false; break; }
      const uint8_t* prow = s_packed + ps * kPackedStageBytes + row * (kKS / 2);
      const uint4 sc = *reinterpret_cast<const uint4*>(s_scales + ps * kScaleStageBytes +
                                                       row * (kKS / 16));
      const uint32_t scw[4] = {sc.x, sc.y, sc.z, sc.w};
      nan_seen |= ((sc.x & 0x7F7F7F7Fu) + 0x01010101u) | ((sc.y & 0x7F7F7F7Fu) + 0x01010101u) |
                  ((sc.z & 0x7F7F7F7Fu) + 0x01010101u) | ((sc.w & 0x7F7F7F7Fu) + 0x01010101u);
      const uint32_t ta = tmem_a + lane_off + st * (kKB / 2);
#pragma unroll
      for (int c4 = 0; c4 < kKB / 64; ++c4) {
        const uint4 c0 = *reinterpret_cast<const uint4*>(prow + (((2 * c4) ^ sw) << 4));
        const uint4 c1 = *reinterpret_cast<const uint4*>(prow + (((2 * c4 + 1) ^ sw) << 4));
        uint32_t s01, s23;
        scales4_to_f16(scw[c4], s01, s23);
        const uint32_t f0 = dup_lo(s01), f1 = dup_hi(s01), f2 = dup_lo(s23), f3 = dup_hi(s23);
        uint32_t v[32];
        dequant8(c0.x, f0, v + 0);
        dequant8(c0.y, f0, v + 4);
        dequant8(c0.z, f1, v + 8);
        dequant8(c0.w, f1, v + 12);
        dequant8(c1.x, f2, v + 16);
        dequant8(c1.y, f2, v + 20);
        dequant8(c1.z, f3, v + 24);
        dequant8(c1.w, f3, v + 28);
        if (c4 == 0 && !warp_wait(&s_empty[st], ph ^ 1, wc)) { ok = false; break; }
        tmem_st32(ta + c4 * 32, v);
      }
      if (!ok) break;
      // the packed stage has been read; the A stage is complete once the
      // TMEM stores land
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_empty[ps]);
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_full[st]);
    }
    if (__any_sync(0xFFFFFFFFu, (nan_seen & 0x80808080u) != 0u) && lane == 0)
      raise_status(p.status, NVFP4_ERR_NONFINITE);
  } else if (warp < kFirstEpiWarp + 4) {
    // ---------------- epilogue: one thread per vocabulary row, BN tokens
    epilogue_role<kOut, false, kGrouped>(p, sc, warp, warp - kFirstEpiWarp, lane, tmem_base,
                                         d_full, d_empty, wc, s_tok, s_thr);
    if (kOut == kOutTopk && lane == 0) atomicAdd(s_last + 1, 1);  // this warp is done
  } else {
    // ---------------- top-k thresholds (only launched in top-k mode)
    topk_threshold_role(p, s_last + 1, lane);
  }

  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
  if constexpr (kOut == kOutArgmax) argmax_finish(p, 32 * kFirstEpiWarp, s_last);
}

// ------------------------------------------------------------ host side
static size_t gemm_smem_bytes(int BN, int stages, int pstages, bool argmax, bool grouped = false) {
  // ring buffers, then 256 B of barriers and flags, then the epilogue's
  // per-warp token multipliers (and, for argmax, a flag and per-warp
  // token thresholds; for the grouped product, after that region, its
  // schedule and the per-group unit prefix and token offsets)
  return 1024 + pstages * (size_t)(kPackedStageBytes + kScaleStageBytes) +
         stages * (size_t)BN * kKB * 2 + 256 + 4 * kMaxBN * sizeof(float) +
         (argmax || grouped ? 16 + 4 * kMaxBN * sizeof(float) : 0) +
         (grouped ? sizeof(Sched) + 2 * (kMaxGroups + 1) * sizeof(uint32_t) +
                        kGrpTab * sizeof(uint2) : 0);
}

size_t lm_head_workspace_bytes(int64_t M, int64_t N, int64_t K, bool argmax) {
  const WsLayout L = ws_layout(M, N, K, std::max(sm_count(), 1), argmax, ActFormat::kF16);
  return weight_stage(N, K, L.total, true).total;
}

// Launch one instantiation (programmatic dependent of the prep kernel).
template <int kOut, int kStages, int kPStages, int kDq, bool kGrouped = false>
static cudaError_t launch_gemm(const CUtensorMap& tm_packed, const CUtensorMap& tm_scales,
                               const CUtensorMap& tm_x, const GemmArgs& a, int grid,
                               cudaStream_t stream) {
  auto kern = w4a16_tc_kernel<kOut, kStages, kPStages, kDq, kGrouped>;
  constexpr bool kArgmax = kOut == kOutArgmax || kOut == kOutTopk;  // per-warp thresholds
  const size_t smem = gemm_smem_bytes(a.BN, kStages, kPStages, kArgmax, kGrouped);
  // the 3-stage shape only serves token tiles of up to 64
  constexpr int kMaxTileBN = kStages >= 3 ? 64 : kMaxBN;
  static std::atomic<uint64_t> limit_set{0};
  const cudaError_t attr_err =
      smem_limit_once(limit_set, reinterpret_cast<const void*>(kern),
                      gemm_smem_bytes(kMaxTileBN, kStages, kPStages, kArgmax, kGrouped));
  if (attr_err != cudaSuccess) return attr_err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(gemm_threads<kOut, kStages, kPStages, kDq>());
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tm_packed, tm_scales, tm_x, a);
}

// Tensor maps of the packed codes and block scales of `rows` weight rows:
// in place where the row length is a 16-byte multiple, else over the
// staged copy.  The map's extent is the real row length, so the TMA fills
// the k past K with zeros (code 0, scale 0: the weight is 0 there).
static bool encode_weight_maps(CUtensorMap* tm_packed, CUtensorMap* tm_scales,
                               const WeightStage& w, const uint8_t* packed, const uint8_t* scales,
                               int64_t rows, int64_t K, uint8_t* ws) {
  return encode_2d(tm_packed, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.packed ? ws + w.packed_off : packed,
                   (uint64_t)K / 2, (uint64_t)rows, w.packed ? w.packed_stride : (uint64_t)K / 2,
                   kKS / 2, kRows, CU_TENSOR_MAP_SWIZZLE_128B) &&
         encode_2d(tm_scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.scales ? ws + w.scales_off : scales,
                   (uint64_t)K / 16, (uint64_t)rows, w.scales ? w.scales_stride : (uint64_t)K / 16,
                   kKS / 16, kRows, CU_TENSOR_MAP_SWIZZLE_NONE);
}

size_t lm_head_topk_workspace_bytes(int64_t M, int64_t N, int64_t K, int k) {
  const int sms = std::max(sm_count(), 1);
  if (M <= kTopkLogitsMaxM && topk_logits_fits(N)) {  // fp32 logits, then the selection
    const WsLayout L = ws_layout(M, N, K, sms, false, ActFormat::kF16);
    return weight_stage(N, K, topk_logits_layout(L.total, M, N).total, true).total;
  }
  const WsLayout L = ws_layout(M, N, K, sms, false, ActFormat::kF16, k);
  return weight_stage(N, K, L.total, true).total;
}

// out_mode: NVFP4_OUT_F32 / NVFP4_OUT_BF16 write logits[M, N] to `logits`;
// kOutArgmax writes token_ids[M] (and max_logits[M] unless null) instead;
// kOutTopk (topk_k > 0) writes token_ids[M, k] (and max_logits[M, k]).
static nvfp4_status lm_head_run(const void* x, int64_t M, int64_t K, const uint8_t* packed,
                                const uint8_t* scales, const float* global_scale, int64_t N,
                                void* logits, int out_mode, int64_t* token_ids,
                                float* max_logits, int topk_k, void* workspace,
                                cudaStream_t stream) {
  const int sms = sm_count();
  if (sms <= 0) return NVFP4_ERR_CUDA;
  const bool argmax = out_mode == kOutArgmax;
  // top-k of a few tokens: the fp32 logits are written and selected from;
  // of many tokens: thresholded candidates in the epilogue
  const bool topk_logits =
      out_mode == kOutTopk && M <= kTopkLogitsMaxM && topk_logits_fits(N);
  const bool topk = out_mode == kOutTopk && !topk_logits;
  const bool keys = argmax || topk;  // per-token lines the prep kernel clears
  const int BN = lm_head_token_tile(M);
  const int n_ttiles = (int)((M + BN - 1) / BN);
  const int64_t m_pad = (int64_t)n_ttiles * BN;
  const WsLayout L = ws_layout(M, N, K, sms, argmax, ActFormat::kF16, topk ? topk_k : 0);
  const TopkLogitsLayout TL = topk_logits_layout(L.total, M, N);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* status = reinterpret_cast<int32_t*>(ws);
  __half* x16 = reinterpret_cast<__half*>(ws + L.x16);
  float* tok_scale = reinterpret_cast<float*>(ws + L.tok);
  uint32_t* split_cnt = reinterpret_cast<uint32_t*>(ws + L.cnt);
  uint32_t* split_ready = reinterpret_cast<uint32_t*>(ws + L.ready);
  float* split_part = reinterpret_cast<float*>(ws + L.part);
  const WeightStage wst = weight_stage(N, K, topk_logits ? TL.total : L.total, true);
  if (topk_logits) {
    out_mode = NVFP4_OUT_F32;
    logits = ws + TL.logits;
  }

  CUtensorMap tm_packed, tm_scales, tm_x;
  if (!encode_weight_maps(&tm_packed, &tm_scales, wst, packed, scales, N, K, ws) ||
      !encode_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x16, (uint64_t)K, (uint64_t)m_pad,
                 (uint64_t)K * 2, 64, (uint32_t)BN, CU_TENSOR_MAP_SWIZZLE_128B))
    return NVFP4_ERR_CUDA;
  if (stage_weights(wst, packed, scales, N, K, ws, stream) != cudaSuccess) return NVFP4_ERR_CUDA;

  // the counters, ready flags and the argmax counter are adjacent: the
  // prep kernel clears them all
  {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    // few rows: a CTA per row (latency); many rows: a warp per row.  The
    // activation map covers whole token tiles and the prep kernel writes
    // the padding rows of the last one as zeros: a box mostly past the
    // map's last row (a single token in a 16-row tile) made every
    // activation load of the GEMM markedly slower than a box of rows
    // that exist (7 µs of a 59 µs call at M = 1)
    const bool wide = M <= kPrepWideRows;
    cfg.gridDim = dim3((unsigned)(wide ? m_pad : (m_pad + 7) / 8));
    cfg.blockDim = dim3(wide ? 128 : 256);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, wide ? w4a16_prep_x_kernel<4> : w4a16_prep_x_kernel<1>,
                           static_cast<const uint16_t*>(x), M, K, m_pad,
                           global_scale, x16, tok_scale, status, split_cnt,
                           (int)((L.part - L.cnt) / 4),
                           keys ? reinterpret_cast<unsigned long long*>(ws + L.keys) : nullptr,
                           topk ? reinterpret_cast<uint32_t*>(ws + L.hist) : nullptr,
                           topk ? topk_hist_stride(N) : 0, nullptr, nullptr, 0) != cudaSuccess)
      return NVFP4_ERR_CUDA;
  }

  GemmArgs a = {};
  a.M = M;
  a.N = N;
  a.K = K;
  a.BN = BN;
  a.n_ttiles = n_ttiles;
  a.n_units = ((N + kRows - 1) / kRows) * n_ttiles;
  a.n_kb = (int)((K + kKB - 1) / kKB);  // the last stage's k past K reads zeros
  schedule_units(a, L.grid, kDecodeTailSkew);
  a.split_cnt = split_cnt;
  a.split_ready = split_ready;
  a.split_part = split_part;
  a.am_keys = keys ? reinterpret_cast<unsigned long long*>(ws + L.keys) : nullptr;
  a.am_done = argmax ? reinterpret_cast<uint32_t*>(ws + L.done) : nullptr;
  a.am_idx = token_ids;
  a.am_val = max_logits;
  if (topk) topk_args(a, ws, L, topk_k, N);
  a.row_scale = nullptr;
  a.grp_max = topk_logits ? reinterpret_cast<uint32_t*>(ws + TL.gmax) : nullptr;
  // decode-sized token tiles get a third A stage, six packed stages and a
  // third dequant warp per quadrant; 128-token tiles leave TMEM room for two
  // A stages only
  const bool deep = BN <= 64;
  const int stages = deep ? 3 : 2;

  // four accumulator buffers where TMEM has room for them (small token
  // tiles: short units then overlap their epilogues), else two
  a.dbuf_log2 = (4 * BN + stages * (kKB / 2) <= 512) ? 2u : 1u;
  a.tmem_cols = ((BN << a.dbuf_log2) + stages * (kKB / 2) <= 256) ? 256u : 512u;
  a.tok_scale = tok_scale;
  a.out = logits;
  a.status = status;
  const int grid = L.grid;  // min(SMs, units): every CTA's range spans >= one unit
  // programmatic dependent launch: the GEMM starts streaming weights while
  // the prep kernel is still running
  cudaError_t err;
  if (topk_logits)
    err = deep ? launch_gemm<kOutLogitsGroups, 3, 6, 3>(tm_packed, tm_scales, tm_x, a, grid, stream)
               : launch_gemm<kOutLogitsGroups, 2, 4, 2>(tm_packed, tm_scales, tm_x, a, grid, stream);
  else if (argmax)
    err = deep ? launch_gemm<kOutArgmax, 3, 6, 3>(tm_packed, tm_scales, tm_x, a, grid, stream)
               : launch_gemm<kOutArgmax, 2, 4, 2>(tm_packed, tm_scales, tm_x, a, grid, stream);
  else if (topk) {
    err = deep ? launch_gemm<kOutTopk, 3, 6, 3>(tm_packed, tm_scales, tm_x, a, grid, stream)
               : launch_gemm<kOutTopk, 2, 4, 2>(tm_packed, tm_scales, tm_x, a, grid, stream);
    if (err == cudaSuccess)
      err = topk_select_launch(a.am_keys, a.tk_grp, a.tk_cand, a.tk_hist, a.tk_hstride, M, N,
                               topk_k, token_ids, max_logits, stream);
  } else if (out_mode == NVFP4_OUT_BF16)
    err = deep ? launch_gemm<NVFP4_OUT_BF16, 3, 6, 3>(tm_packed, tm_scales, tm_x, a, grid, stream)
               : launch_gemm<NVFP4_OUT_BF16, 2, 4, 2>(tm_packed, tm_scales, tm_x, a, grid, stream);
  else
    err = deep ? launch_gemm<NVFP4_OUT_F32, 3, 6, 3>(tm_packed, tm_scales, tm_x, a, grid, stream)
               : launch_gemm<NVFP4_OUT_F32, 2, 4, 2>(tm_packed, tm_scales, tm_x, a, grid, stream);
  if (err == cudaSuccess && topk_logits)
    err = topk_logits_launch(reinterpret_cast<const float*>(ws + TL.logits), a.grp_max, M, N,
                             topk_k, token_ids, max_logits, stream);
  if (err != cudaSuccess || cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
  return NVFP4_OK;
}

nvfp4_status lm_head_launch(const void* x, int64_t M, int64_t K, const uint8_t* packed,
                            const uint8_t* scales, const float* global_scale, int64_t N,
                            void* logits, int out_mode, int64_t* token_ids, float* max_logits,
                            void* workspace, cudaStream_t stream) {
  return lm_head_run(x, M, K, packed, scales, global_scale, N, logits, out_mode, token_ids,
                     max_logits, 0, workspace, stream);
}

nvfp4_status lm_head_topk_launch(const void* x, int64_t M, int64_t K, const uint8_t* packed,
                                 const uint8_t* scales, const float* global_scale, int64_t N,
                                 int k, int64_t* token_ids, float* values, void* workspace,
                                 cudaStream_t stream) {
  return lm_head_run(x, M, K, packed, scales, global_scale, N, nullptr, kOutTopk, token_ids,
                     values, k, workspace, stream);
}

// ------------------------------------------------------------ grouped product
// Token tile of a grouped call: from the mean rows per group.
static int grouped_token_tile(int64_t M, int64_t n_groups) {
  const int64_t mean = std::max<int64_t>(1, (M + n_groups - 1) / n_groups);
  int bn = 16;  // a power of two (the device divides by shifting)
  while (bn < kMaxBN && bn < mean) bn *= 2;
  return bn;
}

// Units of a grouped call are at most weight tiles x (token tiles of M + one
// partial tile per group); the split-K arrays are sized for that grid.
static int64_t grouped_units_bound(int64_t M, int64_t N, int64_t n_groups, int BN) {
  return ((N + kRows - 1) / kRows) * ((M + BN - 1) / BN + n_groups);
}

size_t grouped_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t n_groups) {
  const int BN = grouped_token_tile(M, n_groups);
  const int sms = std::max(sm_count(), 1);
  const int64_t units = grouped_units_bound(M, N, n_groups, BN);
  // the plain product's layout for M token rows and a grid of at most
  // min(SMs, unit bound); its token tile is never below the grouped one, so
  // the split-K partials fit
  const WsLayout L = ws_layout(M, units * kRows, K, sms, false, ActFormat::kF16);
  return weight_stage(n_groups * N, K, L.total, true).total;
}

nvfp4_status grouped_launch(const void* x, int64_t M, int64_t K, const int32_t* grp_off,
                            int64_t n_groups, const uint8_t* packed, const uint8_t* scales,
                            const float* grp_global, int64_t N, void* out, int out_dtype,
                            void* workspace, cudaStream_t stream) {
  const int sms = sm_count();
  if (sms <= 0) return NVFP4_ERR_CUDA;
  const int BN = grouped_token_tile(M, n_groups);
  const int64_t units = grouped_units_bound(M, N, n_groups, BN);
  // same byte layout as grouped_workspace_bytes: token rows M (TMA zero-fills
  // past them), grid min(SMs, unit bound)
  const WsLayout L = ws_layout(M, units * kRows, K, sms, false, ActFormat::kF16);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* status = reinterpret_cast<int32_t*>(ws);
  __half* x16 = reinterpret_cast<__half*>(ws + L.x16);
  float* tok_scale = reinterpret_cast<float*>(ws + L.tok);

  CUtensorMap tm_packed, tm_scales, tm_x;
  const int64_t rows = n_groups * N;
  const WeightStage wst = weight_stage(rows, K, L.total, true);
  if (!encode_weight_maps(&tm_packed, &tm_scales, wst, packed, scales, rows, K, ws) ||
      !encode_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x16, (uint64_t)K, (uint64_t)M,
                 (uint64_t)K * 2, 64, (uint32_t)BN, CU_TENSOR_MAP_SWIZZLE_128B))
    return NVFP4_ERR_CUDA;
  if (stage_weights(wst, packed, scales, rows, K, ws, stream) != cudaSuccess) return NVFP4_ERR_CUDA;
  {
    const bool wide = M <= kPrepWideRows;
    PdlLaunch l(dim3((unsigned)(wide ? M : (M + 7) / 8)), dim3(wide ? 128 : 256), 0, stream);
    if (cudaLaunchKernelEx(&l.cfg, wide ? w4a16_prep_x_kernel<4> : w4a16_prep_x_kernel<1>,
                           static_cast<const uint16_t*>(x), M, K, M,
                           (const float*)nullptr, x16, tok_scale, status,
                           reinterpret_cast<uint32_t*>(ws + L.cnt), (int)((L.part - L.cnt) / 4),
                           (unsigned long long*)nullptr, (uint32_t*)nullptr, 0,
                           grp_off, grp_global,
                           (int)n_groups) != cudaSuccess)
      return NVFP4_ERR_CUDA;
  }
  GemmArgs a = {};
  a.M = M;
  a.N = N;
  a.K = K;
  a.BN = BN;
  a.n_ttiles = 1;
  a.n_kb = (int)((K + kKB - 1) / kKB);
  a.split_cnt = reinterpret_cast<uint32_t*>(ws + L.cnt);
  a.split_ready = reinterpret_cast<uint32_t*>(ws + L.ready);
  a.split_part = reinterpret_cast<float*>(ws + L.part);
  a.tok_scale = tok_scale;
  a.out = out;
  a.status = status;
  a.grp_off = grp_off;
  a.grp_global = grp_global;
  a.n_groups = (int)n_groups;
  const bool deep = BN <= 64;
  const int stages = deep ? 3 : 2;
  // four accumulator buffers where TMEM has room for them (small token
  // tiles: short units then overlap their epilogues), else two
  a.dbuf_log2 = (4 * BN + stages * (kKB / 2) <= 512) ? 2u : 1u;
  a.tmem_cols = ((BN << a.dbuf_log2) + stages * (kKB / 2) <= 256) ? 256u : 512u;
  const int grid = L.grid;
  cudaError_t err;
  if (out_dtype == NVFP4_OUT_BF16)
    err = deep ? launch_gemm<NVFP4_OUT_BF16, 3, 6, 3, true>(tm_packed, tm_scales, tm_x, a, grid, stream)
               : launch_gemm<NVFP4_OUT_BF16, 2, 4, 2, true>(tm_packed, tm_scales, tm_x, a, grid, stream);
  else
    err = deep ? launch_gemm<NVFP4_OUT_F32, 3, 6, 3, true>(tm_packed, tm_scales, tm_x, a, grid, stream)
               : launch_gemm<NVFP4_OUT_F32, 2, 4, 2, true>(tm_packed, tm_scales, tm_x, a, grid, stream);
  if (err != cudaSuccess || cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
  return NVFP4_OK;
}

}  // namespace nvfp4
