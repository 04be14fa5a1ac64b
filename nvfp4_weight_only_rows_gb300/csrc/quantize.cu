// quantize.cu -- the NVFP4 row quantizer (`_quantize_nvfp4` on the page
// "vllm.model_executor.layers.quantization.online.lm_head") for sm_103a.
//
// Two HBM passes over W, because every block scale depends on the
// tensor-wide amax:
//   pass 1 (nvfp4_amax_kernel): grid-stride 16-byte loads, |bf16| maxima
//          taken on the integer bit patterns (exact), one partial per CTA.
//   pass 2 (nvfp4_encode_kernel): every CTA folds the partials into amax,
//          derives global = max(amax / 2688, 1e-12) and its reciprocal,
//          then each warp encodes whole rows in 256-value segments: each
//          lane loads 8 bf16 (16 bytes), a lane pair forms one 16-value
//          block, one shuffle gives the block max, and each lane stores one
//          32-bit word of 8 packed codes; even lanes store the E4M3 scale
//          byte.  Rows are walked from the end of W backwards so the tail
//          that pass 1 left in L2 is consumed first.
//
// Arithmetic (each an IEEE binary32 operation, round to nearest even):
//   t  = min((vmax * fl(1/6)) * inv_global, 448)     block scale before E4M3
//   s  = e4m3_rn_satfinite(t)
//   r  = s == 0 ? 0 : 1 / (f32(s) * global)
//   q  = x * r, rounded to E2M1 with satfinite (+-6) and ties to even code
//   code 0x8 (negative zero) is rewritten to 0x0: the sign bit is set only
//   for values < 0.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "common.cuh"

namespace nvfp4 {

constexpr int kAmaxThreads = 256;
constexpr int kEncodeThreads = 256;
constexpr int kMaxAmaxBlocks = 4096;

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// max of |bf16| over the 8 values of a 16-byte vector, as packed u16 pairs
__device__ __forceinline__ uint32_t absmax8(uint4 v, uint32_t m) {
  const uint32_t k = 0x7FFF7FFFu;
  m = __vmaxu2(m, v.x & k);
  m = __vmaxu2(m, v.y & k);
  m = __vmaxu2(m, v.z & k);
  m = __vmaxu2(m, v.w & k);
  return m;
}

__device__ __forceinline__ uint32_t fold_u16x2(uint32_t m) { return max(m & 0xFFFFu, m >> 16); }

__global__ void __launch_bounds__(kAmaxThreads) nvfp4_amax_kernel(const uint4* __restrict__ W,
                                                                  int64_t n_vec,
                                                                  uint32_t* __restrict__ partial,
                                                                  int32_t* __restrict__ status) {
  // launched as a programmatic dependent of whatever ran before it: wait for
  // that kernel's results before touching memory
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (blockIdx.x == 0 && threadIdx.x == 0) *status = NVFP4_OK;  // a fresh call: clear the word
  uint32_t m = 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  constexpr int kInFlight = 8;  // 128 bytes per thread in flight
  for (; i + (kInFlight - 1) * stride < n_vec; i += kInFlight * stride) {
    uint4 v[kInFlight];
#pragma unroll
    for (int j = 0; j < kInFlight; ++j) v[j] = ld_stream(W + i + j * stride);
#pragma unroll
    for (int j = 0; j < kInFlight; ++j) m = absmax8(v[j], m);
  }
  for (; i < n_vec; i += stride) m = absmax8(ld_stream(W + i), m);
  // this block's loads are done: the encode kernel may be launched (it waits
  // for this grid's completion before reading the partials)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  m = fold_u16x2(m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  __shared__ uint32_t red[kAmaxThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t r = 0;
    for (int w = 0; w < kAmaxThreads / 32; ++w) r = max(r, red[w]);
    partial[blockIdx.x] = r;
  }
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__global__ void __launch_bounds__(kEncodeThreads) nvfp4_encode_kernel(
    const uint16_t* __restrict__ W, int64_t N, int64_t K, const uint32_t* __restrict__ partial,
    int n_partial, uint32_t* __restrict__ packed, uint8_t* __restrict__ scales,
    float* __restrict__ global_out, int32_t* __restrict__ status) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // pass 1 complete and visible
  // ---- amax from the pass-1 partials (every CTA, from L2)
  __shared__ uint32_t red[kEncodeThreads / 32];
  __shared__ float sg[2];
  uint32_t m = 0;
  for (int i = threadIdx.x; i < n_partial; i += blockDim.x) m = max(m, partial[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t a = 0;
    for (int w = 0; w < kEncodeThreads / 32; ++w) a = max(a, red[w]);
    if (a >= 0x7F80u) {  // Inf or NaN somewhere in W
      sg[0] = __int_as_float(0x7FC00000);
      if (blockIdx.x == 0) {
        raise_status(status, NVFP4_ERR_NONFINITE);
        *global_out = __int_as_float(0x7FC00000);
      }
    } else {
      const float amax = __uint_as_float(a << 16);
      float g = __fdiv_rn(amax, 2688.0f);  // amax / (6 * 448)
      g = fmaxf(g, 1e-12f);
      sg[0] = g;
      sg[1] = __frcp_rn(g);
      if (blockIdx.x == 0) *global_out = g;
    }
  }
  __syncthreads();
  const float g = sg[0];
  if (!(g == g)) return;  // non-finite W: nothing to encode
  const float ig = sg[1];
  const float inv6 = 1.0f / 6.0f;
  // r = 1 / (f32(scale) * global) for every E4M3 scale code the cast can
  // produce (0x00..0x7E; satfinite never gives the NaN code 0x7F)
  __shared__ float r_of_code[128];
  if (threadIdx.x < 128) {
    const float sf =
        __half2float(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)threadIdx.x, __NV_E4M3)));
    r_of_code[threadIdx.x] =
        (sf == 0.0f || threadIdx.x == 127) ? 0.0f : __frcp_rn(__fmul_rn(sf, g));
  }
  __syncthreads();

  // ---- encode: each warp takes whole rows, from the last row backwards
  // (pass 1 left the tail of W in L2); a row is walked in 256-value
  // segments, four segment loads in flight per lane
  const int lane = threadIdx.x & 31;
  const int segs = (int)((K + 255) / 256);
  const int64_t warp_id = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  constexpr int kU = 4;
  for (int64_t row = N - 1 - warp_id; row >= 0; row -= n_warps) {
    const uint16_t* wrow = W + row * K;
    uint32_t* prow = packed + row * (K / 8);
    uint8_t* srow = scales + row * (K / 16);
    for (int s0 = 0; s0 < segs; s0 += kU) {
      uint4 v[kU];
#pragma unroll
      for (int i = 0; i < kU; ++i) {
        const int col = (s0 + i) * 256 + lane * 8;
        v[i] = make_uint4(0, 0, 0, 0);
        if (col < K) v[i] = ld_stream(reinterpret_cast<const uint4*>(wrow + col));
      }
#pragma unroll
      for (int i = 0; i < kU; ++i) {
        const int col = (s0 + i) * 256 + lane * 8;
        // block max over the lane pair (16 values); K % 16 == 0, so both
        // lanes of a pair are in or out of the row together
        uint32_t bm = fold_u16x2(absmax8(v[i], 0));
        bm = max(bm, __shfl_xor_sync(0xFFFFFFFFu, bm, 1));
        const float vmax = __uint_as_float(bm << 16);
        float t = __fmul_rn(__fmul_rn(vmax, inv6), ig);
        t = fminf(t, 448.0f);
        const __nv_fp8_storage_t s8 = __nv_cvt_float_to_fp8(t, __NV_SATFINITE, __NV_E4M3);
        const float r = r_of_code[s8 & 0x7F];
        // x * r, two values per packed multiply (each lane rounds like the
        // scalar binary32 multiply)
        const float2 r2 = make_float2(r, r);
        const uint32_t w4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        float q[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 p2 = __fmul2_rn(make_float2(bf16_lo(w4[j]), bf16_hi(w4[j])), r2);
          q[2 * j] = p2.x;
          q[2 * j + 1] = p2.y;
        }
        const uint32_t word = cvt_e2m1x8(q);
        if (col < K) {
          prow[col >> 3] = word;
          if ((lane & 1) == 0) srow[col >> 4] = (uint8_t)s8;
        }
      }
    }
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------ host side
static int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

size_t quantize_workspace_bytes() {
  return kWsHeader + align_up(sizeof(uint32_t) * kMaxAmaxBlocks, 256);
}

nvfp4_status quantize_launch(const void* W, int64_t N, int64_t K, uint8_t* packed,
                             uint8_t* scales, float* global_scale, void* workspace,
                             cudaStream_t stream) {
  const int sms = device_sms();
  if (sms <= 0) return NVFP4_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* status = reinterpret_cast<int32_t*>(ws);
  uint32_t* partial = reinterpret_cast<uint32_t*>(ws + kWsHeader);

  const int64_t n_vec = N * K / 8;
  int64_t want = (n_vec + kAmaxThreads * 4 - 1) / (kAmaxThreads * 4);
  int blocks1 = (int)std::min<int64_t>(std::min<int64_t>(want, (int64_t)sms * 8), kMaxAmaxBlocks);
  if (blocks1 < 1) blocks1 = 1;

  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kAmaxThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3((unsigned)blocks1);
  if (cudaLaunchKernelEx(&cfg, nvfp4_amax_kernel, static_cast<const uint4*>(W), n_vec, partial,
                         status) != cudaSuccess)
    return NVFP4_ERR_CUDA;

  const int64_t warps_per_block = kEncodeThreads / 32;
  int64_t want2 = (N + warps_per_block - 1) / warps_per_block;
  int blocks2 = (int)std::min<int64_t>(want2, (int64_t)sms * 8);
  if (blocks2 < 1) blocks2 = 1;
  cfg.gridDim = dim3((unsigned)blocks2);
  cfg.blockDim = dim3(kEncodeThreads);
  if (cudaLaunchKernelEx(&cfg, nvfp4_encode_kernel, static_cast<const uint16_t*>(W), N, K,
                         static_cast<const uint32_t*>(partial), blocks1,
                         reinterpret_cast<uint32_t*>(packed), scales, global_scale,
                         status) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  return NVFP4_OK;
}

}  // namespace nvfp4
