// w4a4.cu -- the W4A4 NVFP4 product on sm_103a: activations quantized to
// NVFP4 in the call, both operands multiplied at the FP4 tensor-core rate
// with block-scaled tcgen05 MMAs (kind::mxf4nvf4, one UE4M3 scale per 16
// values of K).
//
// Follows `CompressedTensorsW4A4Fp4.apply_weights` and `swizzle_blockscale`
// on the page "vllm.model_executor.layers.quantization.compressed_tensors.
// schemes" and `maybe_fuse_global_scales` / `KNvfp4Dynamic` on the page
// "vllm/model_executor/layers/quantization/modelopt.py":
//  - the weight is the NVFP4 checkpoint layout (codes, row-major E4M3 block
//    scales, global = amax/2688), its block scales re-laid once into the
//    128x4-interleaved order the tensor cores read (`swizzle_blockscale`);
//  - x is quantized per 16 values with the same rule as the weight, against a
//    per-tensor input global scale (a dequant multiplier, amax_x/2688 for a
//    calibrated amax), its scales written in the interleaved order;
//  - logits = fl32(acc * alpha), alpha = fl32(g_x * g_w), acc the fp32 sum of
//    the block-scaled products (each e2m1 * e2m1 * e4m3 * e4m3 exact).
//
// Kernels:
//  nvfp4_swizzle_scales_kernel  row-major [N, K/16] -> interleaved
//                               [N_pad128 / 128][ceil(K/64)][32][4][4] bytes
//                               (rows padded to 128, columns to 4, with zeros);
//  w4a4_prep_x_kernel           one CTA per token (padded to 128): codes,
//                               interleaved scales, alpha; per-call clearing;
//  w4a4_tc_kernel               persistent GEMM: warp 0 streams weight codes
//                               (TMA, 128-byte swizzle) and their scale atoms
//                               (bulk copy), warp 1 the same for x, warp 2
//                               copies the atoms into TMEM (tcgen05.cp) and
//                               issues 4 MMAs of K = 64 per 256-k stage,
//                               warps 3-6 run the shared epilogue.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "gemm_common.cuh"

namespace nvfp4 {

// Byte offset of scale (row r, k-block c) in the 128x4-interleaved layout of
// a matrix with kb scale columns after padding (kb % 4 == 0): 512-byte atoms
// of 128 rows x 4 columns, ordered [row / 128][c / 4]; inside an atom row
// 32 a + b, column d sits at b * 16 + a * 4 + d.
__host__ __device__ __forceinline__ int64_t sf_offset(int64_t r, int64_t c, int64_t kb) {
  const int64_t rr = r & 127, a = rr >> 5, b = rr & 31;
  return (((r >> 7) * (kb >> 2) + (c >> 2)) << 9) + b * 16 + a * 4 + (c & 3);
}

// ------------------------------------------------------------ scale layout
// One thread per 4 output bytes (one row's 4 consecutive k-blocks).  kb:
// the source's scale columns (K/16); kbp: kb rounded up to 4.  Rows past N
// and columns past kb are written as zero.
__global__ void __launch_bounds__(256) nvfp4_swizzle_scales_kernel(
    const uint8_t* __restrict__ scales, int64_t N, int64_t kb, int64_t kbp,
    uint8_t* __restrict__ out, int64_t n_words) {
  const int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (w >= n_words) return;
  // word w of the output: atom w / 128, inside it b = (w % 128) / 4, a = w % 4
  const int64_t atom = w >> 7, b = (w >> 2) & 31, a = w & 3;
  const int64_t c4 = atom % (kbp >> 2), rt = atom / (kbp >> 2);
  const int64_t r = rt * 128 + a * 32 + b;
  uint32_t v = 0;
  if (r < N) {
    const uint8_t* src = scales + r * kb + c4 * 4;
    if (kb % 4 == 0) {  // whole, 4-byte aligned words
      v = *reinterpret_cast<const uint32_t*>(src);
    } else {
      for (int d = 0; d < 4; ++d)
        if (c4 * 4 + d < kb) v |= (uint32_t)src[d] << (8 * d);
    }
  }
  reinterpret_cast<uint32_t*>(out)[w] = v;
}

// ------------------------------------------------------------ activations
__global__ void __launch_bounds__(256) w4a4_prep_x_kernel(
    const uint16_t* __restrict__ x, int64_t M, int64_t K, int64_t m_pad,
    const float* __restrict__ g_in, const float* __restrict__ g_w, uint8_t* __restrict__ xq,
    uint8_t* __restrict__ xsf, float* __restrict__ tok_scale, int32_t* __restrict__ status,
    uint32_t* __restrict__ split_flags, int n_split_flags, unsigned long long* __restrict__ am_keys,
    uint32_t* __restrict__ tk_hist, int tk_hstride) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (blockIdx.x == 0) {
    if (threadIdx.x == 0) *status = NVFP4_OK;
    for (int i = threadIdx.x; i < n_split_flags; i += blockDim.x) split_flags[i] = 0;
  }
  const int64_t m = blockIdx.x;  // 0 .. round_up(M, 128) - 1
  const int64_t kb = K / 16;                      // scale columns
  const int64_t kbp = (kb + 3) / 4 * 4;           // ... padded to whole atoms (zero scales)
  const int64_t xs = (K / 2 + 15) / 16 * 16;      // code row stride (a TMA row stride)
  const float g = *g_in;
  if (threadIdx.x == 0) {
    if (m < m_pad) tok_scale[m] = m < M ? __fmul_rn(g, *g_w) : 0.0f;
    if (m == 0 && !(g > 0.0f && g < __int_as_float(0x7F800000)))
      raise_status(status, NVFP4_ERR_NONFINITE);  // the input global must be positive and finite
  }
  if (m < m_pad)  // argmax / top-k
    token_state_clear(am_keys, tk_hist, tk_hstride, m, threadIdx.x, blockDim.x);
  const float ig = __frcp_rn(g);
  const float inv6 = 1.0f / 6.0f;
  for (int64_t c = threadIdx.x; c < kbp; c += blockDim.x) {
    uint32_t word0 = 0, word1 = 0;
    uint8_t s8 = 0;
    if (m < M && c < kb) {
      const uint4* src = reinterpret_cast<const uint4*>(x + m * K + c * 16);
      const uint4 v0 = src[0], v1 = src[1];
      const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      uint32_t mx = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) mx = __vmaxu2(mx, w[i] & 0x7FFF7FFFu);
      mx = max(mx & 0xFFFFu, mx >> 16);
      const float vmax = __uint_as_float(mx << 16);
      const float t = fminf(__fmul_rn(__fmul_rn(vmax, inv6), ig), 448.0f);
      s8 = (uint8_t)__nv_cvt_float_to_fp8(t, __NV_SATFINITE, __NV_E4M3);
      const float sf =
          __half2float(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)s8, __NV_E4M3)));
      const float r = sf == 0.0f ? 0.0f : __frcp_rn(__fmul_rn(sf, g));
      float q[8];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          q[2 * i] = __fmul_rn(__uint_as_float(w[4 * h + i] << 16), r);
          q[2 * i + 1] = __fmul_rn(__uint_as_float(w[4 * h + i] & 0xFFFF0000u), r);
        }
        (h == 0 ? word0 : word1) = cvt_e2m1x8(q);
      }
    }
    if (m < m_pad && c < kb) reinterpret_cast<uint2*>(xq + m * xs)[c] = make_uint2(word0, word1);
    xsf[sf_offset(m, c, kbp)] = s8;
  }
}

// ------------------------------------------------------------ the GEMM
constexpr int kW4FirstEpiWarp = 3;
constexpr int kW4Threads = 32 * (kW4FirstEpiWarp + 4);
// threads of one CTA: the roles above, plus the threshold warp in top-k mode
template <int kOut>
constexpr int w4a4_threads() { return kW4Threads + (kOut == kOutTopk ? 32 : 0); }
constexpr uint32_t kW4AStageBytes = kRows * (kKB / 2);  // 128 rows x 256 fp4 = 16 KB
constexpr uint32_t kW4SfStageBytes = 4 * 512;            // 4 atoms (16 k-blocks) x 128 rows
constexpr uint32_t kW4SfCols = 32;                       // TMEM columns per stage: A 16 + B 16

// Scale atoms (one per 64 k, 512 bytes for 128 rows) of 256-k stage kb:
// four, except in the last stage of a K that is not a multiple of 256.
__device__ __forceinline__ uint32_t stage_atoms(int64_t kb4, uint32_t kb) {
  const int64_t left = kb4 - 4 * (int64_t)kb;
  return left < 4 ? (uint32_t)left : 4u;
}

template <int kOut, int kStages>
__global__ void __launch_bounds__(w4a4_threads<kOut>(), 1)
    w4a4_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                   const uint8_t* __restrict__ wsf, const uint8_t* __restrict__ xsf,
                   const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int BN = p.BN;
  const uint32_t x_stage_bytes = (uint32_t)BN * 128;
  uint8_t* s_a = smem;                                       // kStages x 16 KB
  uint8_t* s_x = s_a + kStages * kW4AStageBytes;             // kStages x BN x 128 B
  uint8_t* s_sfa = s_x + kStages * x_stage_bytes;            // kStages x 2 KB
  uint8_t* s_sfb = s_sfa + kStages * kW4SfStageBytes;        // kStages x 2 KB
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_sfb + kStages * kW4SfStageBytes);
  uint64_t* s_full = bars;
  uint64_t* s_empty = s_full + kStages;
  uint64_t* d_full = s_empty + kStages;
  uint64_t* d_empty = d_full + 2;
  uint64_t* done_bar = d_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(tmem_slot + 1);
  float* s_tok = reinterpret_cast<float*>(bars + 32);
  int32_t* s_last = reinterpret_cast<int32_t*>(s_tok + 4 * kMaxBN);
  float* s_thr = reinterpret_cast<float*>(s_last + 4);

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
  const int64_t kb4 = (p.K + 63) / 64;  // scale atoms per 128-row band (K/16 padded to 4)

  if (warp == 0) {
    // ---------------- weight codes (TMA) + their scale atoms (bulk copy)
    const uint64_t pol = p.n_ttiles == 1 ? policy_evict_first() : policy_evict_last();
    uint32_t issued = 0;
    for_each_piece(p, [&](const Piece& pc) {
      const uint32_t nt = pc.u / p.n_ttiles;
      for (uint32_t kb = pc.kb0; kb < pc.kb1; ++kb, ++issued) {
        const uint32_t st = issued % kStages, ph = (issued / kStages) & 1;
        if (!warp_wait(&s_empty[st], ph ^ 1, wc)) return false;
        if (elect_one()) {
          const uint32_t sf_bytes = stage_atoms(kb4, kb) * 512;
          mbar_arrive_expect_tx(&s_full[st], kW4AStageBytes + sf_bytes);
          tma_load_2d_hint(s_a + st * kW4AStageBytes, &tm_w, kb * (kKB / 2), (int32_t)(nt * kRows),
                           &s_full[st], pol);
          bulk_load(s_sfa + st * kW4SfStageBytes, wsf + ((int64_t)nt * kb4 + 4 * kb) * 512,
                    sf_bytes, &s_full[st], pol);
        }
        __syncwarp();
      }
      return true;
    });
    drain_loads(s_full, kStages, issued, 2, p.status);
  } else if (warp == 1) {
    // ---------------- activation codes + scale atoms (after the prep kernel)
    grid_dependency_wait();
    const uint64_t pol = policy_evict_last();
    uint32_t issued = 0;
    for_each_piece(p, [&](const Piece& pc) {
      const int64_t t0 = (int64_t)(pc.u % p.n_ttiles) * BN;  // 0 or a multiple of 128
      for (uint32_t kb = pc.kb0; kb < pc.kb1; ++kb, ++issued) {
        const uint32_t st = issued % kStages, ph = (issued / kStages) & 1;
        if (!warp_wait(&s_empty[st], ph ^ 1, wc)) return false;
        if (elect_one()) {
          const uint32_t sf_bytes = stage_atoms(kb4, kb) * 512;
          mbar_arrive_expect_tx(&s_full[st], x_stage_bytes + sf_bytes);
          tma_load_2d_hint(s_x + st * x_stage_bytes, &tm_x, kb * (kKB / 2), (int32_t)t0,
                           &s_full[st], pol);
          bulk_load(s_sfb + st * kW4SfStageBytes, xsf + ((t0 >> 7) * kb4 + 4 * kb) * 512,
                    sf_bytes, &s_full[st], pol);
        }
        __syncwarp();
      }
      return true;
    });
    drain_loads(s_full, kStages, issued, 2, p.status);
  } else if (warp == 2) {
    // ---------------- scale atoms into TMEM, then 4 block-scaled MMAs per stage.
    // A stage's TMEM scale slot is reused only after its smem slot was
    // refilled, i.e. after the MMAs that read the slot completed.
    const uint32_t idesc = idesc_e2m1_bs((uint32_t)BN);
    const uint64_t adesc0 = smem_desc_sw128(smem_u32(s_a));
    const uint64_t xdesc0 = smem_desc_sw128(smem_u32(s_x));
    const uint32_t sf_base = tmem_base + 2 * BN;
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
        const uint64_t ad = adesc0 + ((st * kW4AStageBytes) >> 4);
        const uint64_t xd = xdesc0 + ((st * x_stage_bytes) >> 4);
        const uint32_t sfa = sf_base + st * kW4SfCols, sfb = sfa + 16;
        // one scale atom per MMA of K = 64; the last stage of a K that is not a
        // multiple of 256 has fewer (the k past the last atom is not multiplied)
        const uint32_t n_at = stage_atoms(kb4, kb);
        if (elect_one()) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if ((uint32_t)j < n_at) {
              tc_cp_32x128b_x4(sfa + 4 * j, smem_u32(s_sfa + st * kW4SfStageBytes + 512 * j));
              tc_cp_32x128b_x4(sfb + 4 * j, smem_u32(s_sfb + st * kW4SfStageBytes + 512 * j));
            }
          }
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if ((uint32_t)j < n_at)
              tc_mma_fp4_bs(d_tmem, ad + 2 * j, xd + 2 * j, idesc, sfa + 4 * j, sfb + 4 * j,
                            (kb != pc.kb0) || (j != 0));
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
  } else if (warp < kW4FirstEpiWarp + 4) {
    // ---------------- epilogue: x alpha (the token multiplier)
    epilogue_role<kOut, false>(p, plain_sched(p), warp, warp - kW4FirstEpiWarp, lane, tmem_base, d_full, d_empty,
                               wc, s_tok, s_thr);
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
  if constexpr (kOut == kOutArgmax) argmax_finish(p, 32 * kW4FirstEpiWarp, s_last);
}

// ------------------------------------------------------------ host side
static int64_t round_up128(int64_t v) { return (v + 127) / 128 * 128; }

size_t nvfp4_swizzled_scales_size(int64_t N, int64_t K) {
  return (size_t)round_up128(N) * (size_t)interleaved_sf_cols(K);
}

nvfp4_status swizzle_scales_launch(const uint8_t* scales, int64_t N, int64_t K, uint8_t* out,
                                   cudaStream_t stream) {
  const int64_t n_words = (int64_t)nvfp4_swizzled_scales_size(N, K) / 4;
  const int64_t blocks = (n_words + 255) / 256;
  nvfp4_swizzle_scales_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
      scales, N, K / 16, interleaved_sf_cols(K), out, n_words);
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

static size_t w4a4_smem_bytes(int BN, int stages, bool argmax) {
  return 1024 + stages * ((size_t)kW4AStageBytes + (size_t)BN * 128 + 2 * kW4SfStageBytes) + 256 +
         4 * kMaxBN * sizeof(float) + (argmax ? 16 + 4 * kMaxBN * sizeof(float) : 0);
}

// Workspace: the generic layout with the x codes (M_pad rows, a 16-byte
// multiple apart) and the interleaved x scales (round_up(M, 128) x
// round_up(K/16, 4) bytes) as the activation region; then, where K % 32 !=
// 0, the weight codes staged to a TMA-readable row stride.
size_t w4a4_workspace_bytes(int64_t M, int64_t N, int64_t K, bool argmax) {
  const WsLayout L = ws_layout(M, N, K, std::max(sm_count(), 1), argmax, ActFormat::kE2M1);
  return weight_stage(N, K, L.total, false).total;
}

size_t w4a4_topk_workspace_bytes(int64_t M, int64_t N, int64_t K, int k) {
  const int sms = std::max(sm_count(), 1);
  if (M <= kTopkLogitsMaxM && topk_logits_fits(N)) {  // fp32 logits, then the selection
    const WsLayout L = ws_layout(M, N, K, sms, false, ActFormat::kE2M1);
    return weight_stage(N, K, topk_logits_layout(L.total, M, N).total, false).total;
  }
  const WsLayout L = ws_layout(M, N, K, sms, false, ActFormat::kE2M1, k);
  return weight_stage(N, K, L.total, false).total;
}

template <int kOut, int kStages>
static cudaError_t launch_w4a4(const CUtensorMap& tm_w, const CUtensorMap& tm_x,
                               const uint8_t* wsf, const uint8_t* xsf, const GemmArgs& a, int grid,
                               cudaStream_t stream) {
  auto kern = w4a4_tc_kernel<kOut, kStages>;
  constexpr bool kArgmax = kOut == kOutArgmax || kOut == kOutTopk;  // per-warp thresholds
  constexpr int kMaxTileBN = kStages >= 6 ? 64 : kMaxBN;
  static std::atomic<uint64_t> limit_set{0};
  const cudaError_t attr_err = smem_limit_once(limit_set, reinterpret_cast<const void*>(kern),
                                               w4a4_smem_bytes(kMaxTileBN, kStages, kArgmax));
  if (attr_err != cudaSuccess) return attr_err;
  PdlLaunch l(dim3((unsigned)grid), dim3(w4a4_threads<kOut>()),
              w4a4_smem_bytes(a.BN, kStages, kArgmax), stream);
  return cudaLaunchKernelEx(&l.cfg, kern, tm_w, tm_x, wsf, xsf, a);
}

// out_mode: NVFP4_OUT_F32 / NVFP4_OUT_BF16 write logits[M, N]; kOutArgmax
// writes token_ids[M] (and max_logits[M] unless null); kOutTopk (topk_k > 0)
// writes token_ids[M, k] (and max_logits[M, k]).
static nvfp4_status w4a4_run(const void* x, int64_t M, int64_t K, const uint8_t* packed,
                             const uint8_t* wsf, const float* g_w, const float* g_in, int64_t N,
                             void* logits, int out_mode, int64_t* token_ids, float* max_logits,
                             int topk_k, void* workspace, cudaStream_t stream) {
  const int sms = sm_count();
  if (sms <= 0) return NVFP4_ERR_CUDA;
  const bool argmax = out_mode == kOutArgmax;
  // top-k of a few tokens: the fp32 logits are written and selected from;
  // of many tokens: thresholded candidates in the epilogue
  const bool topk_logits =
      out_mode == kOutTopk && M <= kTopkLogitsMaxM && topk_logits_fits(N);
  const bool topk = out_mode == kOutTopk && !topk_logits;
  const int BN = lm_head_token_tile(M);
  const int n_ttiles = (int)((M + BN - 1) / BN);
  const int64_t m_pad = (int64_t)n_ttiles * BN;
  const int64_t m_pad128 = round_up128(M);
  const WsLayout L = ws_layout(M, N, K, sms, argmax, ActFormat::kE2M1, topk ? topk_k : 0);
  const TopkLogitsLayout TL = topk_logits_layout(L.total, M, N);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (topk_logits) {
    out_mode = NVFP4_OUT_F32;
    logits = ws + TL.logits;
  }
  int32_t* status = reinterpret_cast<int32_t*>(ws);
  uint8_t* xq = ws + L.x16;
  const int64_t xs = e2m1_code_stride(K);
  uint8_t* xsf = xq + align_up((size_t)m_pad * xs, 256);
  const WeightStage wst = weight_stage(N, K, topk_logits ? TL.total : L.total, false);
  float* tok_scale = reinterpret_cast<float*>(ws + L.tok);
  unsigned long long* keys =
      argmax || topk ? reinterpret_cast<unsigned long long*>(ws + L.keys) : nullptr;

  CUtensorMap tm_w, tm_x;
  // both maps end at K/2 bytes: the TMA fills the k past K with zero codes
  if (!encode_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, wst.packed ? ws + wst.packed_off : packed,
                 (uint64_t)K / 2, (uint64_t)N, wst.packed ? wst.packed_stride : (uint64_t)K / 2,
                 128, kRows, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, (uint64_t)K / 2, (uint64_t)m_pad,
                 (uint64_t)xs, 128, (uint32_t)BN, CU_TENSOR_MAP_SWIZZLE_128B))
    return NVFP4_ERR_CUDA;
  if (wst.packed && stage_rows_launch(packed, N, K / 2, ws + wst.packed_off,
                                      (int64_t)wst.packed_stride, stream) != cudaSuccess)
    return NVFP4_ERR_CUDA;

  {
    PdlLaunch l(dim3((unsigned)m_pad128), dim3(256), 0, stream);
    if (cudaLaunchKernelEx(&l.cfg, w4a4_prep_x_kernel, static_cast<const uint16_t*>(x), M, K,
                           m_pad, g_in, g_w, xq, xsf, tok_scale, status,
                           reinterpret_cast<uint32_t*>(ws + L.cnt), (int)((L.part - L.cnt) / 4),
                           keys, topk ? reinterpret_cast<uint32_t*>(ws + L.hist) : nullptr,
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
  a.n_kb = (int)((K + kKB - 1) / kKB);
  // later-starting CTAs take up to 4/64 fewer tail stages (same box, decode
  // M = 32 / 64: 53.0 / 54.1 -> 52.6 / 53.7 us; the W8A8 product did not move)
  schedule_units(a, L.grid, 4);
  const bool small = BN <= 64;
  const uint32_t need = 2u * BN + (small ? 6u : 5u) * kW4SfCols;
  uint32_t cols = 32;
  while (cols < need) cols *= 2;
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
  a.row_scale = nullptr;
  a.grp_max = topk_logits ? reinterpret_cast<uint32_t*>(ws + TL.gmax) : nullptr;
  if (topk) topk_args(a, ws, L, topk_k, N);
  const int grid = L.grid;
  cudaError_t err;
  if (topk_logits)
    err = small ? launch_w4a4<kOutLogitsGroups, 6>(tm_w, tm_x, wsf, xsf, a, grid, stream)
                : launch_w4a4<kOutLogitsGroups, 5>(tm_w, tm_x, wsf, xsf, a, grid, stream);
  else if (argmax)
    err = small ? launch_w4a4<kOutArgmax, 6>(tm_w, tm_x, wsf, xsf, a, grid, stream)
                : launch_w4a4<kOutArgmax, 5>(tm_w, tm_x, wsf, xsf, a, grid, stream);
  else if (topk) {
    err = small ? launch_w4a4<kOutTopk, 6>(tm_w, tm_x, wsf, xsf, a, grid, stream)
                : launch_w4a4<kOutTopk, 5>(tm_w, tm_x, wsf, xsf, a, grid, stream);
    if (err == cudaSuccess)
      err = topk_select_launch(a.am_keys, a.tk_grp, a.tk_cand, a.tk_hist, a.tk_hstride, M, N,
                               topk_k, token_ids, max_logits, stream);
  } else if (out_mode == NVFP4_OUT_BF16)
    err = small ? launch_w4a4<NVFP4_OUT_BF16, 6>(tm_w, tm_x, wsf, xsf, a, grid, stream)
                : launch_w4a4<NVFP4_OUT_BF16, 5>(tm_w, tm_x, wsf, xsf, a, grid, stream);
  else
    err = small ? launch_w4a4<NVFP4_OUT_F32, 6>(tm_w, tm_x, wsf, xsf, a, grid, stream)
                : launch_w4a4<NVFP4_OUT_F32, 5>(tm_w, tm_x, wsf, xsf, a, grid, stream);
  if (err == cudaSuccess && topk_logits)
    err = topk_logits_launch(reinterpret_cast<const float*>(ws + TL.logits), a.grp_max, M, N,
                             topk_k, token_ids, max_logits, stream);
  if (err != cudaSuccess || cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
  return NVFP4_OK;
}

nvfp4_status w4a4_launch(const void* x, int64_t M, int64_t K, const uint8_t* packed,
                         const uint8_t* wsf, const float* g_w, const float* g_in, int64_t N,
                         void* logits, int out_mode, int64_t* token_ids, float* max_logits,
                         void* workspace, cudaStream_t stream) {
  return w4a4_run(x, M, K, packed, wsf, g_w, g_in, N, logits, out_mode, token_ids, max_logits, 0,
                  workspace, stream);
}

nvfp4_status w4a4_topk_launch(const void* x, int64_t M, int64_t K, const uint8_t* packed,
                              const uint8_t* wsf, const float* g_w, const float* g_in, int64_t N,
                              int k, int64_t* token_ids, float* values, void* workspace,
                              cudaStream_t stream) {
  return w4a4_run(x, M, K, packed, wsf, g_w, g_in, N, nullptr, kOutTopk, token_ids, values, k,
                  workspace, stream);
}

}  // namespace nvfp4
