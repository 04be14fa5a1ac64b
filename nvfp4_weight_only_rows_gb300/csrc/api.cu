// api.cu -- the extern "C" entry points declared in include/nvfp4_lm_head.h:
// host-side argument checks, workspace sizing and dispatch to the kernels in
// quantize.cu and lm_head.cu.  No entry point allocates device memory.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"

namespace nvfp4 {
size_t quantize_workspace_bytes();
nvfp4_status quantize_launch(const void* W, int64_t N, int64_t K, uint8_t* packed,
                             uint8_t* scales, float* global_scale, void* workspace,
                             cudaStream_t stream);
size_t lm_head_workspace_bytes(int64_t M, int64_t N, int64_t K, bool argmax);
nvfp4_status lm_head_launch(const void* x, int64_t M, int64_t K, const uint8_t* packed,
                            const uint8_t* scales, const float* global_scale, int64_t N,
                            void* logits, int out_mode, int64_t* token_ids, float* max_logits,
                            void* workspace, cudaStream_t stream);
constexpr int kOutArgmax = 2;  // lm_head_launch's third output mode
size_t lm_head_topk_workspace_bytes(int64_t M, int64_t N, int64_t K, int k);
nvfp4_status lm_head_topk_launch(const void* x, int64_t M, int64_t K, const uint8_t* packed,
                                 const uint8_t* scales, const float* global_scale, int64_t N,
                                 int k, int64_t* token_ids, float* values, void* workspace,
                                 cudaStream_t stream);
int64_t fp8_max_k();
size_t grouped_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t n_groups);
nvfp4_status grouped_launch(const void* x, int64_t M, int64_t K, const int32_t* grp_off,
                            int64_t n_groups, const uint8_t* packed, const uint8_t* scales,
                            const float* grp_global, int64_t N, void* out, int out_dtype,
                            void* workspace, cudaStream_t stream);
constexpr int64_t kMaxGroupsApi = 256;
size_t nvfp4_swizzled_scales_size(int64_t N, int64_t K);
nvfp4_status swizzle_scales_launch(const uint8_t* scales, int64_t N, int64_t K, uint8_t* out,
                                   cudaStream_t stream);
size_t w4a4_workspace_bytes(int64_t M, int64_t N, int64_t K, bool argmax);
nvfp4_status w4a4_launch(const void* x, int64_t M, int64_t K, const uint8_t* packed,
                         const uint8_t* wsf, const float* g_w, const float* g_in, int64_t N,
                         void* logits, int out_mode, int64_t* token_ids, float* max_logits,
                         void* workspace, cudaStream_t stream);
nvfp4_status fp8_quantize_launch(const void* W, int64_t N, int64_t K, uint8_t* q,
                                 float* row_scale, void* workspace, cudaStream_t stream);
size_t w8a8_workspace_bytes(int64_t M, int64_t N, int64_t K, bool argmax);
nvfp4_status w8a8_launch(const void* x, int64_t M, int64_t K, const uint8_t* wq,
                         const float* w_scale, int64_t N, void* logits, int out_mode,
                         int64_t* token_ids, float* max_logits, void* workspace,
                         cudaStream_t stream);
size_t w8a8_topk_workspace_bytes(int64_t M, int64_t N, int64_t K, int k);
nvfp4_status w8a8_topk_launch(const void* x, int64_t M, int64_t K, const uint8_t* wq,
                              const float* w_scale, int64_t N, int k, int64_t* token_ids,
                              float* values, void* workspace, cudaStream_t stream);
size_t w4a4_topk_workspace_bytes(int64_t M, int64_t N, int64_t K, int k);
nvfp4_status w4a4_topk_launch(const void* x, int64_t M, int64_t K, const uint8_t* packed,
                              const uint8_t* wsf, const float* g_w, const float* g_in, int64_t N,
                              int k, int64_t* token_ids, float* values, void* workspace,
                              cudaStream_t stream);

static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The kernels are built for sm_103a only; refuse other devices up front.
static nvfp4_status check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  if (major != 10 || minor != 3) return NVFP4_ERR_UNSUPPORTED;
  return NVFP4_OK;
}

static constexpr int64_t kMaxDim = (int64_t)1 << 31;

static nvfp4_status check_quantize_args(const void* W, int64_t N, int64_t K, const uint8_t* packed,
                                        const uint8_t* scales, const float* global_scale,
                                        const void* workspace, size_t workspace_bytes) {
  if (N <= 0 || K <= 0 || K % 16 != 0 || N >= kMaxDim || K >= kMaxDim) return NVFP4_ERR_SHAPE;
  if (!W || !packed || !scales || !global_scale) return NVFP4_ERR_NULL;
  if (!workspace || workspace_bytes < quantize_workspace_bytes()) return NVFP4_ERR_WORKSPACE;
  if (!aligned(W, 16) || !aligned(packed, 16) || !aligned(global_scale, 4) ||
      !aligned(workspace, 256))
    return NVFP4_ERR_ALIGN;
  return check_device();
}

}  // namespace nvfp4

using namespace nvfp4;

extern "C" {

const char* nvfp4_status_string(nvfp4_status s) {
  switch (s) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_SHAPE: return "shape out of range";
    case NVFP4_ERR_ALIGN: return "pointer not aligned as required";
    case NVFP4_ERR_NULL: return "required pointer is NULL";
    case NVFP4_ERR_WORKSPACE: return "workspace missing or too small";
    case NVFP4_ERR_DTYPE: return "unknown output dtype";
    case NVFP4_ERR_CUDA: return "CUDA call failed";
    case NVFP4_ERR_NONFINITE: return "weight holds Inf or NaN";
    case NVFP4_ERR_TIMEOUT: return "device pipeline wait timed out";
    case NVFP4_ERR_UNSUPPORTED: return "device is not sm_103 (GB300)";
    case NVFP4_ERR_SCRATCH_LIMIT: return "shape needs more than the fixed scratch of the allocation-free call";
  }
  return "unknown status";
}

int nvfp4_abi_version(void) { return 100; }

size_t nvfp4_quantize_workspace_bytes(int64_t N, int64_t K) {
  if (N <= 0 || K <= 0 || K % 16 != 0) return 0;
  return quantize_workspace_bytes();
}

nvfp4_status nvfp4_quantize_rows(const void* W, int64_t N, int64_t K, uint8_t* packed,
                                 uint8_t* scales, float* global_scale, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  nvfp4_status st =
      check_quantize_args(W, N, K, packed, scales, global_scale, workspace, workspace_bytes);
  if (st != NVFP4_OK) return st;
  return quantize_launch(W, N, K, packed, scales, global_scale, workspace,
                         static_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_refresh(const void* W, int64_t N, int64_t K, uint8_t* packed, uint8_t* scales,
                           float* global_scale, void* workspace, size_t workspace_bytes,
                           void* stream) {
  // Same kernels, same buffers: re-deriving in place is what keeps the
  // addresses captured by CUDA graphs valid.
  return nvfp4_quantize_rows(W, N, K, packed, scales, global_scale, workspace, workspace_bytes,
                             stream);
}

nvfp4_status nvfp4_read_device_status(const void* workspace, int32_t* status_out, void* stream) {
  if (!workspace || !status_out) return NVFP4_ERR_NULL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  *status_out = v;
  return NVFP4_OK;
}

size_t w4a16_lm_head_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 16 || K % 16 != 0) return 0;
  return lm_head_workspace_bytes(M, N, K, false);
}

nvfp4_status w4a16_lm_head(const void* x, int64_t M, int64_t K, const uint8_t* packed,
                           const uint8_t* scales, const float* global_scale, int64_t N,
                           void* logits, int out_dtype, void* workspace, size_t workspace_bytes,
                           void* stream) {
  if (M < 0 || N < 0 || K < 16 || K % 16 != 0 || M >= kMaxDim || N >= kMaxDim ||
      K >= kMaxDim)
    return NVFP4_ERR_SHAPE;
  if (out_dtype != NVFP4_OUT_F32 && out_dtype != NVFP4_OUT_BF16) return NVFP4_ERR_DTYPE;
  if (M == 0 || N == 0) return NVFP4_OK;  // empty product: nothing to write
  if (!x || !packed || !scales || !global_scale || !logits) return NVFP4_ERR_NULL;
  if (!workspace || workspace_bytes < lm_head_workspace_bytes(M, N, K, false))
    return NVFP4_ERR_WORKSPACE;
  if (!aligned(x, 16) || !aligned(packed, 16) || !aligned(scales, 16) ||
      !aligned(global_scale, 4) || !aligned(logits, 16) || !aligned(workspace, 256))
    return NVFP4_ERR_ALIGN;
  nvfp4_status st = check_device();
  if (st != NVFP4_OK) return st;
  return lm_head_launch(x, M, K, packed, scales, global_scale, N, logits, out_dtype, nullptr,
                        nullptr, workspace, static_cast<cudaStream_t>(stream));
}

size_t w4a16_lm_head_argmax_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N <= 0 || K < 16 || K % 16 != 0) return 0;
  return lm_head_workspace_bytes(M, N, K, true);
}

nvfp4_status w4a16_lm_head_argmax(const void* x, int64_t M, int64_t K, const uint8_t* packed,
                                  const uint8_t* scales, const float* global_scale, int64_t N,
                                  int64_t* token_ids, float* max_logits, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  // N <= 0: the maximum over no logits does not exist
  if (M < 0 || N <= 0 || K < 16 || K % 16 != 0 || M >= kMaxDim || N >= kMaxDim ||
      K >= kMaxDim)
    return NVFP4_ERR_SHAPE;
  if (M == 0) return NVFP4_OK;
  if (!x || !packed || !scales || !global_scale || !token_ids) return NVFP4_ERR_NULL;
  if (!workspace || workspace_bytes < lm_head_workspace_bytes(M, N, K, true))
    return NVFP4_ERR_WORKSPACE;
  if (!aligned(x, 16) || !aligned(packed, 16) || !aligned(scales, 16) ||
      !aligned(global_scale, 4) || !aligned(token_ids, 8) || !aligned(max_logits, 4) ||
      !aligned(workspace, 256))
    return NVFP4_ERR_ALIGN;
  nvfp4_status st = check_device();
  if (st != NVFP4_OK) return st;
  return lm_head_launch(x, M, K, packed, scales, global_scale, N, nullptr, kOutArgmax, token_ids,
                        max_logits, workspace, static_cast<cudaStream_t>(stream));
}

/* ------------------------------------------------------------ fused top-k */

static bool topk_shape_ok(int64_t M, int64_t N, int64_t K, int64_t k) {
  return M >= 0 && N > 0 && K >= 16 && K % 16 == 0 && M < kMaxDim && N < kMaxDim &&
         K < kMaxDim && k >= 1 && k <= NVFP4_TOPK_MAX && k <= N && M * N <= ((int64_t)1 << 36);
}

size_t w4a16_lm_head_topk_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t k) {
  if (!topk_shape_ok(M, N, K, k)) return 0;
  return lm_head_topk_workspace_bytes(M, N, K, (int)k);
}

nvfp4_status w4a16_lm_head_topk(const void* x, int64_t M, int64_t K, const uint8_t* packed,
                                const uint8_t* scales, const float* global_scale, int64_t N,
                                int64_t k, int64_t* token_ids, float* values, void* workspace,
                                size_t workspace_bytes, void* stream) {
  if (!topk_shape_ok(M, N, K, k)) return NVFP4_ERR_SHAPE;
  if (M == 0) return NVFP4_OK;
  if (!x || !packed || !scales || !global_scale || !token_ids) return NVFP4_ERR_NULL;
  if (!workspace || workspace_bytes < lm_head_topk_workspace_bytes(M, N, K, (int)k))
    return NVFP4_ERR_WORKSPACE;
  if (!aligned(x, 16) || !aligned(packed, 16) || !aligned(scales, 16) ||
      !aligned(global_scale, 4) || !aligned(token_ids, 8) || !aligned(values, 4) ||
      !aligned(workspace, 256))
    return NVFP4_ERR_ALIGN;
  nvfp4_status st = check_device();
  if (st != NVFP4_OK) return st;
  return lm_head_topk_launch(x, M, K, packed, scales, global_scale, N, (int)k, token_ids, values,
                             workspace, static_cast<cudaStream_t>(stream));
}

/* ------------------------------------------------------------ fp8 copy */

size_t fp8_quantize_workspace_bytes(int64_t N, int64_t K) {
  if (N <= 0 || K <= 0 || K % 16 != 0 || K > fp8_max_k()) return 0;
  return kWsHeader;
}

nvfp4_status fp8_quantize_rows(const void* W, int64_t N, int64_t K, uint8_t* q, float* row_scale,
                               void* workspace, size_t workspace_bytes, void* stream) {
  if (N <= 0 || K <= 0 || K % 16 != 0 || K > fp8_max_k() || N >= kMaxDim) return NVFP4_ERR_SHAPE;
  if (!W || !q || !row_scale) return NVFP4_ERR_NULL;
  if (!workspace || workspace_bytes < kWsHeader) return NVFP4_ERR_WORKSPACE;
  if (!aligned(W, 16) || !aligned(q, 16) || !aligned(row_scale, 4) || !aligned(workspace, 256))
    return NVFP4_ERR_ALIGN;
  nvfp4_status st = check_device();
  if (st != NVFP4_OK) return st;
  return fp8_quantize_launch(W, N, K, q, row_scale, workspace, static_cast<cudaStream_t>(stream));
}

nvfp4_status fp8_refresh(const void* W, int64_t N, int64_t K, uint8_t* q, float* row_scale,
                         void* workspace, size_t workspace_bytes, void* stream) {
  // the same kernel into the same buffers: captured addresses stay valid
  return fp8_quantize_rows(W, N, K, q, row_scale, workspace, workspace_bytes, stream);
}

// The activation quantizer of the W8A8 product holds a token row in one
// 256-thread block: K <= 16384.
static constexpr int64_t kW8MaxK = 16384;

static nvfp4_status check_w8a8_shape(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 16 || K % 16 != 0 || K > kW8MaxK || M >= kMaxDim || N >= kMaxDim)
    return NVFP4_ERR_SHAPE;
  return NVFP4_OK;
}

size_t w8a8_lm_head_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (check_w8a8_shape(M, N, K) != NVFP4_OK) return 0;
  return w8a8_workspace_bytes(M, N, K, false);
}

nvfp4_status w8a8_lm_head(const void* x, int64_t M, int64_t K, const uint8_t* wq,
                          const float* w_scale, int64_t N, void* logits, int out_dtype,
                          void* workspace, size_t workspace_bytes, void* stream) {
  nvfp4_status st = check_w8a8_shape(M, N, K);
  if (st != NVFP4_OK) return st;
  if (out_dtype != NVFP4_OUT_F32 && out_dtype != NVFP4_OUT_BF16) return NVFP4_ERR_DTYPE;
  if (M == 0 || N == 0) return NVFP4_OK;
  if (!x || !wq || !w_scale || !logits) return NVFP4_ERR_NULL;
  if (!workspace || workspace_bytes < w8a8_workspace_bytes(M, N, K, false))
    return NVFP4_ERR_WORKSPACE;
  if (!aligned(x, 16) || !aligned(wq, 16) || !aligned(w_scale, 4) || !aligned(logits, 16) ||
      !aligned(workspace, 256))
    return NVFP4_ERR_ALIGN;
  st = check_device();
  if (st != NVFP4_OK) return st;
  return w8a8_launch(x, M, K, wq, w_scale, N, logits, out_dtype, nullptr, nullptr, workspace,
                     static_cast<cudaStream_t>(stream));
}

size_t w8a8_lm_head_argmax_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (check_w8a8_shape(M, N, K) != NVFP4_OK || N == 0) return 0;
  return w8a8_workspace_bytes(M, N, K, true);
}

nvfp4_status w8a8_lm_head_argmax(const void* x, int64_t M, int64_t K, const uint8_t* wq,
                                 const float* w_scale, int64_t N, int64_t* token_ids,
                                 float* max_logits, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  nvfp4_status st = check_w8a8_shape(M, N, K);
  if (st != NVFP4_OK || N == 0) return NVFP4_ERR_SHAPE;
  if (M == 0) return NVFP4_OK;
  if (!x || !wq || !w_scale || !token_ids) return NVFP4_ERR_NULL;
  if (!workspace || workspace_bytes < w8a8_workspace_bytes(M, N, K, true))
    return NVFP4_ERR_WORKSPACE;
  if (!aligned(x, 16) || !aligned(wq, 16) || !aligned(w_scale, 4) || !aligned(token_ids, 8) ||
      !aligned(max_logits, 4) || !aligned(workspace, 256))
    return NVFP4_ERR_ALIGN;
  st = check_device();
  if (st != NVFP4_OK) return st;
  return w8a8_launch(x, M, K, wq, w_scale, N, nullptr, kOutArgmax, token_ids, max_logits,
                     workspace, static_cast<cudaStream_t>(stream));
}

// top-k over the W8A8 / W4A4 logits: k in 1 .. min(N, NVFP4_TOPK_MAX), M x N <= 2^36
static bool topk_k_ok(int64_t M, int64_t N, int64_t k) {
  return N > 0 && k >= 1 && k <= NVFP4_TOPK_MAX && k <= N && M * N <= ((int64_t)1 << 36);
}

size_t w8a8_lm_head_topk_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t k) {
  if (check_w8a8_shape(M, N, K) != NVFP4_OK || !topk_k_ok(M, N, k)) return 0;
  return w8a8_topk_workspace_bytes(M, N, K, (int)k);
}

nvfp4_status w8a8_lm_head_topk(const void* x, int64_t M, int64_t K, const uint8_t* wq,
                               const float* w_scale, int64_t N, int64_t k, int64_t* token_ids,
                               float* values, void* workspace, size_t workspace_bytes,
                               void* stream) {
  nvfp4_status st = check_w8a8_shape(M, N, K);
  if (st != NVFP4_OK || !topk_k_ok(M, N, k)) return NVFP4_ERR_SHAPE;
  if (M == 0) return NVFP4_OK;
  if (!x || !wq || !w_scale || !token_ids) return NVFP4_ERR_NULL;
  if (!workspace || workspace_bytes < w8a8_topk_workspace_bytes(M, N, K, (int)k))
    return NVFP4_ERR_WORKSPACE;
  if (!aligned(x, 16) || !aligned(wq, 16) || !aligned(w_scale, 4) || !aligned(token_ids, 8) ||
      !aligned(values, 4) || !aligned(workspace, 256))
    return NVFP4_ERR_ALIGN;
  st = check_device();
  if (st != NVFP4_OK) return st;
  return w8a8_topk_launch(x, M, K, wq, w_scale, N, (int)k, token_ids, values, workspace,
                          static_cast<cudaStream_t>(stream));
}

/* --------------------------------------------------------- grouped (MoE) */

static nvfp4_status check_grouped_shape(int64_t M, int64_t N, int64_t K, int64_t n_groups) {
  if (M < 0 || N < 0 || K < 16 || K % 16 != 0 || n_groups < 1 || n_groups > kMaxGroupsApi ||
      M >= kMaxDim || N >= kMaxDim || K >= kMaxDim || n_groups * N >= kMaxDim)
    return NVFP4_ERR_SHAPE;
  return NVFP4_OK;
}

size_t w4a16_grouped_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t n_groups) {
  if (check_grouped_shape(M, N, K, n_groups) != NVFP4_OK) return 0;
  return grouped_workspace_bytes(M, N, K, n_groups);
}

nvfp4_status w4a16_grouped_gemm(const void* x, int64_t M, int64_t K, const int32_t* group_offsets,
                                int64_t n_groups, const uint8_t* packed, const uint8_t* scales,
                                const float* global_scales, int64_t N, void* out, int out_dtype,
                                void* workspace, size_t workspace_bytes, void* stream) {
  nvfp4_status st = check_grouped_shape(M, N, K, n_groups);
  if (st != NVFP4_OK) return st;
  if (out_dtype != NVFP4_OUT_F32 && out_dtype != NVFP4_OUT_BF16) return NVFP4_ERR_DTYPE;
  if (M == 0 || N == 0) return NVFP4_OK;
  if (!x || !group_offsets || !packed || !scales || !global_scales || !out) return NVFP4_ERR_NULL;
  if (!workspace || workspace_bytes < grouped_workspace_bytes(M, N, K, n_groups))
    return NVFP4_ERR_WORKSPACE;
  if (!aligned(x, 16) || !aligned(packed, 16) || !aligned(scales, 16) ||
      !aligned(group_offsets, 4) || !aligned(global_scales, 4) || !aligned(out, 16) ||
      !aligned(workspace, 256))
    return NVFP4_ERR_ALIGN;
  st = check_device();
  if (st != NVFP4_OK) return st;
  return grouped_launch(x, M, K, group_offsets, n_groups, packed, scales, global_scales, N, out,
                        out_dtype, workspace, static_cast<cudaStream_t>(stream));
}

/* ------------------------------------------------------------ W4A4 */

size_t nvfp4_swizzled_scales_bytes(int64_t N, int64_t K) {
  if (N <= 0 || K <= 0 || K % 16 != 0 || N >= kMaxDim || K >= kMaxDim) return 0;
  return nvfp4_swizzled_scales_size(N, K);
}

nvfp4_status nvfp4_swizzle_scales(const uint8_t* scales, int64_t N, int64_t K, uint8_t* out,
                                  void* stream) {
  if (N <= 0 || K <= 0 || K % 16 != 0 || N >= kMaxDim || K >= kMaxDim) return NVFP4_ERR_SHAPE;
  if (!scales || !out) return NVFP4_ERR_NULL;
  if (!aligned(scales, 4) || !aligned(out, 16)) return NVFP4_ERR_ALIGN;
  nvfp4_status st = check_device();
  if (st != NVFP4_OK) return st;
  return swizzle_scales_launch(scales, N, K, out, static_cast<cudaStream_t>(stream));
}

static nvfp4_status check_w4a4_shape(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 16 || K % 16 != 0 || M >= kMaxDim || N >= kMaxDim || K >= kMaxDim)
    return NVFP4_ERR_SHAPE;
  return NVFP4_OK;
}

size_t w4a4_lm_head_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (check_w4a4_shape(M, N, K) != NVFP4_OK) return 0;
  return w4a4_workspace_bytes(M, N, K, false);
}

size_t w4a4_lm_head_argmax_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (check_w4a4_shape(M, N, K) != NVFP4_OK || N == 0) return 0;
  return w4a4_workspace_bytes(M, N, K, true);
}

static nvfp4_status check_w4a4_ptrs(const void* x, const uint8_t* packed,
                                    const uint8_t* scales_swizzled, const float* global_scale,
                                    const float* input_global_scale, const void* workspace) {
  if (!x || !packed || !scales_swizzled || !global_scale || !input_global_scale)
    return NVFP4_ERR_NULL;
  if (!aligned(x, 16) || !aligned(packed, 16) || !aligned(scales_swizzled, 16) ||
      !aligned(global_scale, 4) || !aligned(input_global_scale, 4) || !aligned(workspace, 256))
    return NVFP4_ERR_ALIGN;
  return NVFP4_OK;
}

nvfp4_status w4a4_lm_head(const void* x, int64_t M, int64_t K, const uint8_t* packed,
                          const uint8_t* scales_swizzled, const float* global_scale,
                          const float* input_global_scale, int64_t N, void* logits,
                          int out_dtype, void* workspace, size_t workspace_bytes, void* stream) {
  nvfp4_status st = check_w4a4_shape(M, N, K);
  if (st != NVFP4_OK) return st;
  if (out_dtype != NVFP4_OUT_F32 && out_dtype != NVFP4_OUT_BF16) return NVFP4_ERR_DTYPE;
  if (M == 0 || N == 0) return NVFP4_OK;
  if (!logits) return NVFP4_ERR_NULL;
  if (!workspace || workspace_bytes < w4a4_workspace_bytes(M, N, K, false))
    return NVFP4_ERR_WORKSPACE;
  st = check_w4a4_ptrs(x, packed, scales_swizzled, global_scale, input_global_scale, workspace);
  if (st != NVFP4_OK) return st;
  if (!aligned(logits, 16)) return NVFP4_ERR_ALIGN;
  st = check_device();
  if (st != NVFP4_OK) return st;
  return w4a4_launch(x, M, K, packed, scales_swizzled, global_scale, input_global_scale, N, logits,
                     out_dtype, nullptr, nullptr, workspace, static_cast<cudaStream_t>(stream));
}

nvfp4_status w4a4_lm_head_argmax(const void* x, int64_t M, int64_t K, const uint8_t* packed,
                                 const uint8_t* scales_swizzled, const float* global_scale,
                                 const float* input_global_scale, int64_t N, int64_t* token_ids,
                                 float* max_logits, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  nvfp4_status st = check_w4a4_shape(M, N, K);
  if (st != NVFP4_OK || N == 0) return NVFP4_ERR_SHAPE;
  if (M == 0) return NVFP4_OK;
  if (!token_ids) return NVFP4_ERR_NULL;
  if (!workspace || workspace_bytes < w4a4_workspace_bytes(M, N, K, true))
    return NVFP4_ERR_WORKSPACE;
  st = check_w4a4_ptrs(x, packed, scales_swizzled, global_scale, input_global_scale, workspace);
  if (st != NVFP4_OK) return st;
  if (!aligned(token_ids, 8) || !aligned(max_logits, 4)) return NVFP4_ERR_ALIGN;
  st = check_device();
  if (st != NVFP4_OK) return st;
  return w4a4_launch(x, M, K, packed, scales_swizzled, global_scale, input_global_scale, N,
                     nullptr, kOutArgmax, token_ids, max_logits, workspace,
                     static_cast<cudaStream_t>(stream));
}

size_t w4a4_lm_head_topk_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t k) {
  if (check_w4a4_shape(M, N, K) != NVFP4_OK || !topk_k_ok(M, N, k)) return 0;
  return w4a4_topk_workspace_bytes(M, N, K, (int)k);
}

nvfp4_status w4a4_lm_head_topk(const void* x, int64_t M, int64_t K, const uint8_t* packed,
                               const uint8_t* scales_swizzled, const float* global_scale,
                               const float* input_global_scale, int64_t N, int64_t k,
                               int64_t* token_ids, float* values, void* workspace,
                               size_t workspace_bytes, void* stream) {
  nvfp4_status st = check_w4a4_shape(M, N, K);
  if (st != NVFP4_OK || !topk_k_ok(M, N, k)) return NVFP4_ERR_SHAPE;
  if (M == 0) return NVFP4_OK;
  if (!token_ids) return NVFP4_ERR_NULL;
  if (!workspace || workspace_bytes < w4a4_topk_workspace_bytes(M, N, K, (int)k))
    return NVFP4_ERR_WORKSPACE;
  st = check_w4a4_ptrs(x, packed, scales_swizzled, global_scale, input_global_scale, workspace);
  if (st != NVFP4_OK) return st;
  if (!aligned(token_ids, 8) || !aligned(values, 4)) return NVFP4_ERR_ALIGN;
  st = check_device();
  if (st != NVFP4_OK) return st;
  return w4a4_topk_launch(x, M, K, packed, scales_swizzled, global_scale, input_global_scale, N,
                          (int)k, token_ids, values, workspace,
                          static_cast<cudaStream_t>(stream));
}

}  // extern "C"
