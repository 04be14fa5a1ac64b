// fp8.cu -- the "fp8" lm_head copy on sm_103a: per-row E4M3 weights with an
// fp32 scale, per-token E4M3 activations, and the W8A8 product on
// kind::f8f6f4 tcgen05 MMAs.
//
// The copy is the "fp8" branch of `quantized_lm_head_copy` on the page
// "vllm.model_executor.layers.quantization.online.lm_head" (per-row weight
// and per-token activation scales on an FP8 linear kernel), i.e. the
// FP8_PER_CHANNEL_PER_TOKEN scheme of the page
// "vllm/model_executor/layers/quantization/modelopt.py".  The quantizer body
// is not printed; for a row v (a weight row, or a token of x):
//   s = max(fl32(amax|v| / 448), fl32(1e-12)),  r = fl32(1 / s),
//   q = e4m3(fl32(v * r)) with round-to-nearest-even and saturation to
//       +-448 (the hardware cvt.rn.satfinite), sign kept;
// logits[m, n] = fl32(fl32(acc[m, n] * s_x[m]) * s_w[n]) with acc the fp32
// tensor-core sum of e4m3(q_x) * e4m3(q_w) (each product exact).
//
// Kernels:
//  fp8_quantize_kernel  one CTA per weight row: the row is held in registers,
//                       reduced to amax, then encoded (one HBM read, one write);
//  w8a8_prep_x_kernel   the same per token of x, into the workspace, plus the
//                       per-call clearing the GEMM relies on;
//  w8a8_tc_kernel       persistent warp-specialised GEMM: warp 0 streams the
//                       e4m3 weights and warp 1 the e4m3 activations into a
//                       shared-memory ring by TMA (128-byte swizzle), warp 2
//                       issues 8 MMAs of K = 32 per 256-k stage with both
//                       operands read from shared memory, warps 3-6 run the
//                       shared epilogue (token scale, then row scale).
#include "gemm_common.cuh"

namespace nvfp4 {

constexpr int kFp8MaxVec = 8;  // 16-byte loads held per thread: 64 values

// ------------------------------------------------------------ row quantizer
// Quantize one bf16 row of K values (K % 8 == 0, K <= 8 * kFp8MaxVec *
// blockDim.x) with the whole block: returns the scale (also to thread 0's
// caller) and writes K e4m3 bytes to dst.  Non-finite input raises
// NVFP4_ERR_NONFINITE in *status.
__device__ __forceinline__ float fp8_quant_row(const uint16_t* __restrict__ src, int64_t K,
                                               uint8_t* __restrict__ dst, int32_t* status,
                                               uint32_t* red /* shared, >= 32 words */) {
  const int nv = (int)(K / 8);
  const int tid = threadIdx.x, nt = blockDim.x;
  uint4 v[kFp8MaxVec];
  uint32_t mx = 0;
#pragma unroll
  for (int j = 0; j < kFp8MaxVec; ++j) {
    const int i = tid + j * nt;
    v[j] = i < nv ? reinterpret_cast<const uint4*>(src)[i] : make_uint4(0, 0, 0, 0);
    const uint32_t k = 0x7FFF7FFFu;  // |x| as bf16 bits: unsigned order is value order
    mx = __vmaxu2(mx, v[j].x & k);
    mx = __vmaxu2(mx, v[j].y & k);
    mx = __vmaxu2(mx, v[j].z & k);
    mx = __vmaxu2(mx, v[j].w & k);
  }
  mx = max(mx & 0xFFFFu, mx >> 16);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  __syncthreads();  // `red` may still be read from the previous row
  if ((tid & 31) == 0) red[tid >> 5] = mx;
  __syncthreads();
  uint32_t a = 0;
  for (int w = 0; w < (nt >> 5); ++w) a = max(a, red[w]);
  if (a >= 0x7F80u && tid == 0) raise_status(status, NVFP4_ERR_NONFINITE);
  const float amax = __uint_as_float(a << 16);
  const float s = fmaxf(__fdiv_rn(amax, 448.0f), 1e-12f);
  const float r = __frcp_rn(s);
#pragma unroll
  for (int j = 0; j < kFp8MaxVec; ++j) {
    const int i = tid + j * nt;
    if (i >= nv) break;
    const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
    uint32_t o[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint16_t b[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const uint32_t ww = w[2 * h + e];
        const float lo = __fmul_rn(__uint_as_float(ww << 16), r);
        const float hi = __fmul_rn(__uint_as_float(ww & 0xFFFF0000u), r);
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(b[e]) : "f"(hi), "f"(lo));
      }
      o[h] = (uint32_t)b[0] | ((uint32_t)b[1] << 16);
    }
    reinterpret_cast<uint2*>(dst)[i] = make_uint2(o[0], o[1]);
  }
  return s;
}

__global__ void __launch_bounds__(1024) fp8_quantize_kernel(const uint16_t* __restrict__ W,
                                                            int64_t K, uint8_t* __restrict__ q,
                                                            float* __restrict__ row_scale,
                                                            int32_t* __restrict__ status) {
  __shared__ uint32_t red[32];
  const int64_t n = blockIdx.x;
  const float s = fp8_quant_row(W + n * K, K, q + n * K, status, red);
  if (threadIdx.x == 0) row_scale[n] = s;
}

// ------------------------------------------------------------ activations
__global__ void __launch_bounds__(256) w8a8_prep_x_kernel(const uint16_t* __restrict__ x,
                                                          int64_t M, int64_t K,
                                                          uint8_t* __restrict__ xq,
                                                          float* __restrict__ tok_scale,
                                                          int32_t* __restrict__ status,
                                                          uint32_t* __restrict__ split_flags,
                                                          int n_split_flags,
                                                          unsigned long long* __restrict__ am_keys,
                                                          uint32_t* __restrict__ tk_hist,
                                                          int tk_hstride) {
  // wait for the previous kernel in the stream (it may still read this
  // workspace), then let the GEMM launch: it streams the weights meanwhile
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ uint32_t red[32];
  if (blockIdx.x == 0) {
    if (threadIdx.x == 0) *status = NVFP4_OK;
    for (int i = threadIdx.x; i < n_split_flags; i += blockDim.x) split_flags[i] = 0;
  }
  const int64_t m = blockIdx.x;
  token_state_clear(am_keys, tk_hist, tk_hstride, m, threadIdx.x, blockDim.x);  // argmax / top-k
  uint8_t* dst = xq + m * K;
  if (m >= M) {  // padding tokens of the last tile
    for (int64_t i = threadIdx.x; i < K / 16; i += blockDim.x)
      reinterpret_cast<uint4*>(dst)[i] = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) tok_scale[m] = 0.0f;
    return;
  }
  const float s = fp8_quant_row(x + m * K, K, dst, status, red);
  if (threadIdx.x == 0) tok_scale[m] = s;
}

// ------------------------------------------------------------ the GEMM
constexpr int kW8FirstEpiWarp = 3;
constexpr int kW8Threads = 32 * (kW8FirstEpiWarp + 4);
// threads of one CTA: the roles above, plus the threshold warp in top-k mode
template <int kOut>
constexpr int w8a8_threads() { return kW8Threads + (kOut == kOutTopk ? 32 : 0); }

template <int kOut, int kStages, int kKS = kKB, int kTokStride = kMaxBN>
__global__ void __launch_bounds__(w8a8_threads<kOut>(), 1)
    w8a8_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                   const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  constexpr uint32_t kAStageBytes = kRows * kKS;     // 128 rows x kKS e4m3
  constexpr int kBoxes = kKS / 128;                   // 128-k TMA boxes per stage
  const int BN = p.BN;
  const uint32_t x_box_bytes = (uint32_t)BN * 128;  // one 128-k TMA box of activations
  const uint32_t x_stage_bytes = kBoxes * x_box_bytes;
  uint8_t* s_a = smem;                                // kStages x kAStageBytes weights
  uint8_t* s_x = s_a + kStages * kAStageBytes;        // kStages x BN x kKS activations
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_x + kStages * x_stage_bytes);
  uint64_t* s_full = bars;                 // both operands of stage s landed (2 producers)
  uint64_t* s_empty = s_full + kStages;    // the MMAs reading stage s completed
  uint64_t* d_full = s_empty + kStages;
  uint64_t* d_empty = d_full + 2;
  uint64_t* done_bar = d_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(tmem_slot + 1);
  float* s_tok = reinterpret_cast<float*>(bars + 32);  // 4 epilogue warps x kTokStride
  int32_t* s_last = reinterpret_cast<int32_t*>(s_tok + 4 * kTokStride);
  float* s_thr = reinterpret_cast<float*>(s_last + 4);  // argmax, top-k: 4 warps x kTokStride

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s_full[i], 2);
      mbar_init(&s_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&d_full[i], 1);
      mbar_init(&d_empty[i], 4);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    if (kOut == kOutTopk) s_last[1] = 0;  // epilogue warps done (the region exists in this mode)
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, p.tmem_cols);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = __shfl_sync(0xFFFFFFFFu, *tmem_slot, 0);
  WaitCtl wc{p.status, abort_flag, kWaitLimitNs};

  if (warp == 0) {
    // ---------------- weight producer: kBoxes 128-k boxes of 128 rows per stage
    const uint64_t pol = p.n_ttiles == 1 ? policy_evict_first() : policy_evict_last();
    uint32_t issued = 0;
    for_each_piece(p, [&](const Piece& pc) {
      const int32_t n0 = (int32_t)((pc.u / p.n_ttiles) * kRows);
      for (uint32_t kb = pc.kb0; kb < pc.kb1; ++kb, ++issued) {
        const uint32_t st = issued % kStages, ph = (issued / kStages) & 1;
        if (!warp_wait(&s_empty[st], ph ^ 1, wc)) return false;
        if (elect_one()) {
          mbar_arrive_expect_tx(&s_full[st], kAStageBytes);
          uint8_t* dst = s_a + st * kAStageBytes;
#pragma unroll
          for (int b = 0; b < kBoxes; ++b)
            tma_load_2d_hint(dst + b * (kRows * 128), &tm_w, kb * kKS + 128 * b, n0, &s_full[st],
                             pol);
        }
        __syncwarp();
      }
      return true;
    });
    drain_loads(s_full, kStages, issued, 2, p.status);
  } else if (warp == 1) {
    // ---------------- activation producer (after the prep kernel's results)
    grid_dependency_wait();
    const uint64_t pol = policy_evict_last();
    uint32_t issued = 0;
    for_each_piece(p, [&](const Piece& pc) {
      const int32_t t0 = (int32_t)((pc.u % p.n_ttiles) * BN);
      for (uint32_t kb = pc.kb0; kb < pc.kb1; ++kb, ++issued) {
        const uint32_t st = issued % kStages, ph = (issued / kStages) & 1;
        if (!warp_wait(&s_empty[st], ph ^ 1, wc)) return false;
        if (elect_one()) {
          mbar_arrive_expect_tx(&s_full[st], x_stage_bytes);
          uint8_t* dst = s_x + st * x_stage_bytes;
#pragma unroll
          for (int b = 0; b < kBoxes; ++b)
            tma_load_2d_hint(dst + b * x_box_bytes, &tm_x, kb * kKS + 128 * b, t0, &s_full[st],
                             pol);
        }
        __syncwarp();
      }
      return true;
    });
    drain_loads(s_full, kStages, issued, 2, p.status);
  } else if (warp == 2) {
    // ---------------- MMA issuer: kKS / 32 x (M 128, N BN, K 32) per stage
    const uint32_t idesc = idesc_e4m3_f32((uint32_t)BN);
    const uint64_t adesc0 = smem_desc_sw128(smem_u32(s_a));
    const uint64_t xdesc0 = smem_desc_sw128(smem_u32(s_x));
    const uint32_t a_box = (kRows * 128) >> 4, x_box = x_box_bytes >> 4;
    uint32_t g = 0;
    int64_t i = 0;
    for_each_piece(p, [&](const Piece& pc) {
      const uint32_t buf = (uint32_t)(i & 1), dph = (uint32_t)((i >> 1) & 1);
      ++i;
      if (!warp_wait(&d_empty[buf], dph ^ 1, wc)) return false;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + buf * BN;
      for (uint32_t kb = pc.kb0; kb < pc.kb1; ++kb, ++g) {
        const uint32_t st = g % kStages, ph = (g / kStages) & 1;
        if (!warp_wait(&s_full[st], ph, wc)) return false;
        tc_fence_after();
        const uint64_t ad = adesc0 + ((st * kAStageBytes) >> 4);
        const uint64_t xd = xdesc0 + ((st * x_stage_bytes) >> 4);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kKS / 32; ++kk)
            tc_mma_ss_f8(d_tmem, ad + (kk >> 2) * a_box + 2 * (kk & 3),
                         xd + (kk >> 2) * x_box + 2 * (kk & 3), idesc,
                         (kb != pc.kb0) || (kk != 0));
          tc_commit(&s_empty[st]);
        }
        __syncwarp();
      }
      if (elect_one()) tc_commit(&d_full[buf]);
      __syncwarp();
      return true;
    });
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (elect_one()) tc_commit(done_bar);
    __syncwarp();
    volatile int32_t zero = 0;
    WaitCtl drain{p.status, &zero, 100000000ull};
    mbar_wait(done_bar, 0, drain);
  } else if (warp < kW8FirstEpiWarp + 4) {
    // ---------------- epilogue: token scale, then the row's own scale
    epilogue_role<kOut, true, false, kTokStride>(p, plain_sched(p), warp, warp - kW8FirstEpiWarp,
                                                 lane, tmem_base, d_full, d_empty, wc, s_tok,
                                                 s_thr);
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
  if constexpr (kOut == kOutArgmax) argmax_finish(p, 32 * kW8FirstEpiWarp, s_last);
}

// ------------------------------------------------------------ host side
// A stage covers ks of K (256, or 128 for the wide token tile): 128 weight
// rows x ks e4m3 and BN token rows x ks, in 128-byte-wide TMA boxes.
static size_t w8a8_smem_bytes(int BN, int stages, bool argmax, int ks, int tok_stride) {
  return 1024 + stages * ((size_t)kRows * ks + (size_t)BN * ks) + 256 +
         4 * (size_t)tok_stride * sizeof(float) +
         (argmax ? 16 + 4 * (size_t)tok_stride * sizeof(float) : 0);
}

// Threads per row of the row quantizer: each holds at most kFp8MaxVec
// 16-byte loads.  0: K too large.
static int fp8_row_threads(int64_t K) {
  for (int t = 128; t <= 1024; t *= 2)
    if (K <= (int64_t)8 * kFp8MaxVec * t) return t;
  return 0;
}

int64_t fp8_max_k() { return (int64_t)8 * kFp8MaxVec * 1024; }

nvfp4_status fp8_quantize_launch(const void* W, int64_t N, int64_t K, uint8_t* q,
                                 float* row_scale, void* workspace, cudaStream_t stream) {
  const int threads = fp8_row_threads(K);
  if (threads == 0) return NVFP4_ERR_SHAPE;
  int32_t* status = static_cast<int32_t*>(workspace);
  if (cudaMemsetAsync(status, 0, sizeof(int32_t), stream) != cudaSuccess) return NVFP4_ERR_CUDA;
  fp8_quantize_kernel<<<(unsigned)N, threads, 0, stream>>>(static_cast<const uint16_t*>(W), K, q,
                                                          row_scale, status);
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

// Logits of 256 tokens or more take 256-token tiles: an MMA of N = 256 reads
// each weight byte from shared memory once per 256 tokens instead of 128,
// and the shared-memory port, not the fp8 tensor rate, bounds the 128-token
// tile (128 KB of TMA writes and MMA reads per 4.2 M MACs).  TMEM holds two
// such accumulators (the fp8 product keeps no scales there).  The logits,
// argmax and top-k products take the same tiles, so they add the same
// partial sums in the same order.
static bool w8a8_wide(int64_t M) { return M >= kWideBN; }

size_t w8a8_workspace_bytes(int64_t M, int64_t N, int64_t K, bool argmax) {
  return ws_layout(M, N, K, std::max(sm_count(), 1), argmax, ActFormat::kE4M3, 0,
                   w8a8_wide(M) ? kWideBN : 0)
      .total;
}

size_t w8a8_topk_workspace_bytes(int64_t M, int64_t N, int64_t K, int k) {
  const int sms = std::max(sm_count(), 1);
  if (M <= kTopkLogitsMaxM && topk_logits_fits(N))  // fp32 logits, then the selection
    return topk_logits_layout(ws_layout(M, N, K, sms, false, ActFormat::kE4M3).total, M, N).total;
  return ws_layout(M, N, K, sms, false, ActFormat::kE4M3, k, w8a8_wide(M) ? kWideBN : 0).total;
}

template <int kOut, int kStages, int kKS = kKB, int kTokStride = kMaxBN>
static cudaError_t launch_w8a8(const CUtensorMap& tm_w, const CUtensorMap& tm_x, const GemmArgs& a,
                               int grid, cudaStream_t stream) {
  auto kern = w8a8_tc_kernel<kOut, kStages, kKS, kTokStride>;
  constexpr bool kArgmax = kOut == kOutArgmax || kOut == kOutTopk;  // per-warp thresholds
  constexpr int kMaxTileBN = kTokStride > kMaxBN ? kTokStride : (kStages >= 4 ? 64 : kMaxBN);
  static std::atomic<uint64_t> limit_set{0};
  const cudaError_t attr_err =
      smem_limit_once(limit_set, reinterpret_cast<const void*>(kern),
                      w8a8_smem_bytes(kMaxTileBN, kStages, kArgmax, kKS, kTokStride));
  if (attr_err != cudaSuccess) return attr_err;
  PdlLaunch l(dim3((unsigned)grid), dim3(w8a8_threads<kOut>()),
              w8a8_smem_bytes(a.BN, kStages, kArgmax, kKS, kTokStride), stream);
  return cudaLaunchKernelEx(&l.cfg, kern, tm_w, tm_x, a);
}

// out_mode: NVFP4_OUT_F32 / NVFP4_OUT_BF16 write logits[M, N]; kOutArgmax
// writes token_ids[M] (and max_logits[M] unless null); kOutTopk (topk_k > 0)
// writes token_ids[M, k] (and max_logits[M, k]).
static nvfp4_status w8a8_run(const void* x, int64_t M, int64_t K, const uint8_t* wq,
                             const float* w_scale, int64_t N, void* logits, int out_mode,
                             int64_t* token_ids, float* max_logits, int topk_k, void* workspace,
                             cudaStream_t stream) {
  const int sms = sm_count();
  if (sms <= 0) return NVFP4_ERR_CUDA;
  const bool argmax = out_mode == kOutArgmax;
  // top-k of a few tokens: the fp32 logits are written and selected from;
  // of many tokens: thresholded candidates in the epilogue
  const bool topk_logits =
      out_mode == kOutTopk && M <= kTopkLogitsMaxM && topk_logits_fits(N);
  const bool topk = out_mode == kOutTopk && !topk_logits;
  const bool wide = !topk_logits && w8a8_wide(M);
  const int BN = wide ? kWideBN : lm_head_token_tile(M);
  const int ks = wide ? 128 : kKB;  // K per stage
  const int n_ttiles = (int)((M + BN - 1) / BN);
  const int64_t m_pad = (int64_t)n_ttiles * BN;
  const WsLayout L = ws_layout(M, N, K, sms, argmax, ActFormat::kE4M3, topk ? topk_k : 0,
                               wide ? kWideBN : 0);
  const TopkLogitsLayout TL = topk_logits_layout(L.total, M, N);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (topk_logits) {
    out_mode = NVFP4_OUT_F32;
    logits = ws + TL.logits;
  }
  int32_t* status = reinterpret_cast<int32_t*>(ws);
  uint8_t* xq = ws + L.x16;
  float* tok_scale = reinterpret_cast<float*>(ws + L.tok);
  unsigned long long* keys =
      argmax || topk ? reinterpret_cast<unsigned long long*>(ws + L.keys) : nullptr;

  CUtensorMap tm_w, tm_x;
  if (!encode_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, (uint64_t)K, (uint64_t)N, (uint64_t)K,
                 128, kRows, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, (uint64_t)K, (uint64_t)m_pad,
                 (uint64_t)K, 128, (uint32_t)BN, CU_TENSOR_MAP_SWIZZLE_128B))
    return NVFP4_ERR_CUDA;

  {
    PdlLaunch l(dim3((unsigned)m_pad), dim3(256), 0, stream);
    if (cudaLaunchKernelEx(&l.cfg, w8a8_prep_x_kernel, static_cast<const uint16_t*>(x), M, K, xq,
                           tok_scale, status, reinterpret_cast<uint32_t*>(ws + L.cnt),
                           (int)((L.part - L.cnt) / 4), keys,
                           topk ? reinterpret_cast<uint32_t*>(ws + L.hist) : nullptr,
                           topk ? topk_hist_stride(N) : 0) != cudaSuccess)
      return NVFP4_ERR_CUDA;
  }

  GemmArgs a = {};
  a.M = M;
  a.N = N;
  a.K = K;
  a.BN = BN;
  a.n_ttiles = n_ttiles;
  a.n_units = ((N + kRows - 1) / kRows) * n_ttiles;
  // K % 16: the last stage's k past K reads zeros (the weight and activation
  // maps end at K; a TMA box past the end is filled with zeros)
  a.n_kb = (int)((K + ks - 1) / ks);
  schedule_units(a, L.grid);
  uint32_t cols = 32;
  while (cols < 2u * BN) cols *= 2;
  a.tmem_cols = cols;
  a.dbuf_log2 = 1;  // two accumulator buffers
  a.tok_scale = tok_scale;
  a.out = logits;
  a.status = status;
  a.split_cnt = reinterpret_cast<uint32_t*>(ws + L.cnt);
  a.split_ready = reinterpret_cast<uint32_t*>(ws + L.ready);
  a.split_part = reinterpret_cast<float*>(ws + L.part);
  a.am_keys = keys;
  a.am_done = argmax ? reinterpret_cast<uint32_t*>(ws + L.done) : nullptr;
  a.am_idx = token_ids;
  a.am_val = max_logits;
  a.row_scale = w_scale;
  a.grp_max = topk_logits ? reinterpret_cast<uint32_t*>(ws + TL.gmax) : nullptr;
  if (topk) topk_args(a, ws, L, topk_k, N);
  const int grid = L.grid;
  const bool small = BN <= 64;
  cudaError_t err;
  if (topk_logits)
    err = small ? launch_w8a8<kOutLogitsGroups, 4>(tm_w, tm_x, a, grid, stream)
                : launch_w8a8<kOutLogitsGroups, 3>(tm_w, tm_x, a, grid, stream);
  else if (argmax && wide)
    err = launch_w8a8<kOutArgmax, 4, 128, kWideBN>(tm_w, tm_x, a, grid, stream);
  else if (argmax)
    err = small ? launch_w8a8<kOutArgmax, 4>(tm_w, tm_x, a, grid, stream)
                : launch_w8a8<kOutArgmax, 3>(tm_w, tm_x, a, grid, stream);
  else if (topk) {
    err = wide ? launch_w8a8<kOutTopk, 4, 128, kWideBN>(tm_w, tm_x, a, grid, stream)
               : (small ? launch_w8a8<kOutTopk, 4>(tm_w, tm_x, a, grid, stream)
                        : launch_w8a8<kOutTopk, 3>(tm_w, tm_x, a, grid, stream));
    if (err == cudaSuccess)
      err = topk_select_launch(a.am_keys, a.tk_grp, a.tk_cand, a.tk_hist, a.tk_hstride, M, N,
                               topk_k, token_ids, max_logits, stream);
  } else if (wide && out_mode == NVFP4_OUT_BF16)
    err = launch_w8a8<NVFP4_OUT_BF16, 4, 128, kWideBN>(tm_w, tm_x, a, grid, stream);
  else if (wide)
    err = launch_w8a8<NVFP4_OUT_F32, 4, 128, kWideBN>(tm_w, tm_x, a, grid, stream);
  else if (out_mode == NVFP4_OUT_BF16)
    err = small ? launch_w8a8<NVFP4_OUT_BF16, 4>(tm_w, tm_x, a, grid, stream)
                : launch_w8a8<NVFP4_OUT_BF16, 3>(tm_w, tm_x, a, grid, stream);
  else
    err = small ? launch_w8a8<NVFP4_OUT_F32, 4>(tm_w, tm_x, a, grid, stream)
                : launch_w8a8<NVFP4_OUT_F32, 3>(tm_w, tm_x, a, grid, stream);
  if (err == cudaSuccess && topk_logits)
    err = topk_logits_launch(reinterpret_cast<const float*>(ws + TL.logits), a.grp_max, M, N,
                             topk_k, token_ids, max_logits, stream);
  if (err != cudaSuccess || cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
  return NVFP4_OK;
}

nvfp4_status w8a8_launch(const void* x, int64_t M, int64_t K, const uint8_t* wq,
                         const float* w_scale, int64_t N, void* logits, int out_mode,
                         int64_t* token_ids, float* max_logits, void* workspace,
                         cudaStream_t stream) {
  return w8a8_run(x, M, K, wq, w_scale, N, logits, out_mode, token_ids, max_logits, 0, workspace,
                  stream);
}

nvfp4_status w8a8_topk_launch(const void* x, int64_t M, int64_t K, const uint8_t* wq,
                              const float* w_scale, int64_t N, int k, int64_t* token_ids,
                              float* values, void* workspace, cudaStream_t stream) {
  return w8a8_run(x, M, K, wq, w_scale, N, nullptr, kOutTopk, token_ids, values, k, workspace,
                  stream);
}

}  // namespace nvfp4
