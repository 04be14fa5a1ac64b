/*
 * nvfp4_lm_head.h -- C ABI of the GB300 (sm_103a) online NVFP4 lm_head library.
 *
 * Two operations, as the pages define them, are the core of the library:
 *
 *  1. Row quantization of an already-loaded bf16 lm_head to NVFP4 in the
 *     checkpoint layout -- page "vllm.model_executor.layers.quantization.
 *     online.lm_head", section `_quantize_nvfp4`: an fp32 global scale equal
 *     to amax(W) / (6 * 448) (clamped at 1e-12; the raw dequant multiplier,
 *     no reciprocal, as `KNvfp4Static.process` on the page of
 *     vllm/model_executor/layers/quantization/modelopt.py keeps it), one
 *     E4M3 scale per 16 consecutive values of a row, and E2M1 codes with the
 *     sign in bit 3, two per byte with the low nibble first.  Section
 *     `refresh_quantized_lm_heads` of the same page adds the in-place
 *     re-derivation that keeps tensor addresses stable for CUDA graphs.
 *
 *  2. The weight-only W4A16 product against bf16 activations -- section
 *     `_LMHeadNvfp4Method.apply` of the first page and
 *     `CompressedTensorsW4A16Fp4.apply_weights` on the page
 *     "vllm.model_executor.layers.quantization.compressed_tensors.schemes":
 *     logits[m, n] = global * sum_k x[m, k] * e2m1(code[n, k]) * f32(scale[n, k/16]).
 *
 * Around them, in the order of the sections below: the greedy argmax and
 * the top-k of those logits fused into the product (the logits are written
 * only to the workspace, and only up to 256 tokens); the "fp8" lm_head copy
 * (per-row E4M3 weights, W8A8 product) of `quantized_lm_head_copy` on the
 * first page; the grouped W4A16 product of
 * all experts of an NVFP4 MoE layer; the W4A4 NVFP4 product of
 * `CompressedTensorsW4A4Fp4`; an allocation-free variant of the W4A16
 * product; and two self-tests.
 *
 * Conventions for every call:
 *  - All tensor pointers are DEVICE pointers on the current CUDA device,
 *    row-major and contiguous.  The caller owns every buffer; the library
 *    never allocates, frees or synchronizes (except
 *    nvfp4_read_device_status, which is documented as synchronizing).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Work is enqueued on it and the call returns at once.
 *  - bf16 tensors are passed as void* holding IEEE bfloat16 bit patterns;
 *    E4M3 scales are uint8_t holding float8_e4m3fn bit patterns.
 *  - Argument errors are detected on the host and returned as a status
 *    before anything is enqueued.  Conditions that only the device can see
 *    (non-finite weights, a pipeline wait that ran out of time) are written
 *    to a status word inside the workspace; kernels never trap.
 *  - Workspaces must be 256-byte aligned and at least the size the matching
 *    *_workspace_bytes() call returns.  Their contents need no
 *    initialisation and may be reused between calls on the same stream.
 *  - The kernels of a call are chained by programmatic dependent launch: a
 *    call's first kernel waits for the grid launched just before it on the
 *    stream to complete before it touches memory.  A workspace may be
 *    reused by the next call when every kernel enqueued between the two
 *    calls is either launched normally or, if launched as a programmatic
 *    dependent, waits for its own predecessor before it completes.
 */
#ifndef NVFP4_LM_HEAD_H_
#define NVFP4_LM_HEAD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NVFP4_OK = 0,
  NVFP4_ERR_SHAPE = 1,      /* a size is out of range (e.g. K % 16 != 0) */
  NVFP4_ERR_ALIGN = 2,      /* a pointer or row stride is not aligned as required */
  NVFP4_ERR_NULL = 3,       /* a required pointer is NULL */
  NVFP4_ERR_WORKSPACE = 4,  /* workspace missing or smaller than required */
  NVFP4_ERR_DTYPE = 5,      /* unknown output dtype code */
  NVFP4_ERR_CUDA = 6,       /* a CUDA runtime/driver call failed */
  NVFP4_ERR_NONFINITE = 7,  /* device status: W held an Inf or NaN (quantizer), or a block
                               scale read by a W4A16 product is NaN (an unloaded scale) */
  NVFP4_ERR_TIMEOUT = 8,    /* device status: a pipeline wait ran out of time */
  NVFP4_ERR_UNSUPPORTED = 9, /* no sm_103a device / kernel image for it */
  NVFP4_ERR_SCRATCH_LIMIT = 10 /* w4a16_lm_head_noalloc: M*K needs more than its fixed scratch */
} nvfp4_status;

/* Output dtype codes of w4a16_lm_head. */
#define NVFP4_OUT_F32 0
#define NVFP4_OUT_BF16 1

/* Human-readable name of a status; never NULL. */
const char *nvfp4_status_string(nvfp4_status status);

/* ABI version of this header (major * 100 + minor). */
int nvfp4_abi_version(void);

/* ------------------------------------------------------------ quantizer */

/*
 * Workspace bytes nvfp4_quantize_rows / nvfp4_refresh need for W[N, K]:
 * per-block partial maxima of the first pass plus the device status word.
 * Returns 0 for shapes the quantizer rejects.
 */
size_t nvfp4_quantize_workspace_bytes(int64_t N, int64_t K);

/*
 * NVFP4-quantize the rows of W (`_quantize_nvfp4`).
 *
 *   W            bf16 [N, K], device, 16-byte aligned.  Read only.
 *   N, K         N >= 1; K >= 16 and K % 16 == 0 (the K % 16 rule of
 *                `KNvfp4Static.create_weights`).
 *   packed       u8 [N, K/2], device, 16-byte aligned.  Written: byte j of
 *                row n holds the code of W[n, 2j] in bits 3..0 and of
 *                W[n, 2j+1] in bits 7..4; code = grid index | (value < 0) << 3.
 *   scales       u8 (float8_e4m3fn) [N, K/16], device.  Written, row-major
 *                (not swizzled).
 *   global_scale f32 [1], device.  Written: max(amax / 2688, 1e-12).
 *   workspace    device, >= nvfp4_quantize_workspace_bytes(N, K), 256-byte
 *                aligned.  Scratch; also holds the device status word.
 *
 * Two kernels run on `stream`: a grid-wide amax and the per-row encoder.
 * Nothing is read back to the host, so the call can be captured in a CUDA
 * graph.  If W holds an Inf or NaN the status word becomes
 * NVFP4_ERR_NONFINITE, global_scale is set to NaN and packed/scales are left
 * unspecified (the pages assume finite weights).
 */
nvfp4_status nvfp4_quantize_rows(const void *W, int64_t N, int64_t K, uint8_t *packed,
                                 uint8_t *scales, float *global_scale, void *workspace,
                                 size_t workspace_bytes, void *stream);

/*
 * Re-derive the quantized copy of W in place (`refresh_quantized_lm_heads`):
 * the same computation and arguments as nvfp4_quantize_rows, writing into
 * the caller's existing packed / scales / global_scale buffers, so that
 * device addresses captured by CUDA graphs stay valid.  No allocation, no
 * host synchronization.
 */
nvfp4_status nvfp4_refresh(const void *W, int64_t N, int64_t K, uint8_t *packed,
                           uint8_t *scales, float *global_scale, void *workspace,
                           size_t workspace_bytes, void *stream);

/*
 * Read the device status word that the last call using `workspace` left
 * (NVFP4_OK, NVFP4_ERR_NONFINITE or NVFP4_ERR_TIMEOUT) into *status_out.
 * SYNCHRONIZES `stream`; meant for tests and diagnostics, not the hot path.
 * Works for both quantizer and lm_head workspaces.
 */
nvfp4_status nvfp4_read_device_status(const void *workspace, int32_t *status_out, void *stream);

/*
 * Diagnostic: launch a one-CTA kernel whose pipeline wait can never complete
 * (an mbarrier phase nobody arrives on, then a flag nobody sets) and that
 * must give up after `limit_us` microseconds each, raising NVFP4_ERR_TIMEOUT
 * in the status word of `workspace` (>= 256 bytes, 256-byte aligned; only
 * its header is used).  It checks that the library's kernels report a stuck
 * pipeline as a status instead of hanging the GPU; read the result with
 * nvfp4_read_device_status.  0 < limit_us <= 10^7.
 */
nvfp4_status nvfp4_selftest_bounded_wait(void *workspace, size_t workspace_bytes,
                                         int64_t limit_us, void *stream);

/*
 * Host-only check of the fused top-k's histogram (w4a16_lm_head_topk and
 * its W8A8 / W4A4 counterparts): over every 32-bit logit order key in
 * increasing order the bin never decreases and the bin's lower edge -- the
 * threshold a raise to that bin sets -- never exceeds the key, which is
 * what keeps every one of a token's k largest logits above its threshold.
 * Returns -1 when every key passes, else the first failing key.  Runs on
 * the CPU (a few seconds); needs no GPU.
 */
int64_t nvfp4_selftest_topk_bins(void);

/*
 * Host-only check of the persistent products' work split: for a spread of
 * unit counts, grids, stages per unit and tail skews, the whole-unit waves
 * and the stream-K tail cover every stage exactly once, the tail ranges are
 * contiguous and at least one unit long, no unit is cut more than once (the
 * pairwise combine of a cut unit's partials relies on it), and an unskewed
 * tail is the even split.  Returns -1 when every case passes, else the
 * index of the first failing case.  Runs on the CPU; needs no GPU.
 */
int64_t nvfp4_selftest_schedule(void);

/* --------------------------------------------------------- W4A16 GEMM */

/*
 * Workspace bytes w4a16_lm_head needs for x[M, K] against N vocabulary rows:
 * the activations rescaled to fp16 (M * K * 2 bytes), one fp32 scale per
 * token, the device status word and room for split-K partial tiles; for a
 * K that is not a multiple of 256 also a copy of the weight rows whose
 * length is not a 16-byte multiple (block scales [N, K/16] when K % 256 != 0,
 * packed codes [N, K/2] when K % 32 != 0), with the row stride rounded up.
 * Returns 0 for shapes the call rejects.
 */
size_t w4a16_lm_head_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * logits = x . dequant(W)^T with dequant(W)[n, k] =
 * e2m1(code[n, k]) * f32(scale[n, k/16]) * global_scale.
 *
 *   x            bf16 [M, K], device, 16-byte aligned.  M >= 0 (M == 0 is a
 *                no-op), K >= 16 and K % 16 == 0 (the K % 16 rule of
 *                `KNvfp4Static.create_weights` on the page
 *                "vllm/model_executor/layers/quantization/modelopt.py").
 *                The kernels read the weights by TMA, whose row strides must
 *                be 16-byte multiples: for K % 256 == 0 (the usual lm_head
 *                widths) packed and scales are read in place; otherwise the
 *                call first copies the rows that break that rule into the
 *                workspace (one extra pass over the block scales, and over
 *                the packed codes when K % 32 != 0).
 *   packed, scales, global_scale
 *                exactly as nvfp4_quantize_rows writes them for W[N, K];
 *                packed and scales 16-byte aligned.
 *   N            vocabulary rows, N >= 0 (N == 0 is a no-op).
 *   logits       [M, N] device, 16-byte aligned; fp32 (out_dtype
 *                NVFP4_OUT_F32) or bf16 (NVFP4_OUT_BF16, round to nearest even).
 *   workspace    device, >= w4a16_lm_head_workspace_bytes(M, N, K),
 *                256-byte aligned.
 *
 * A NaN block-scale byte (0x7F / 0xFF: the "never loaded" sentinel that
 * `KNvfp4Static.process` on the page
 * "vllm/model_executor/layers/quantization/modelopt.py" rejects) raises
 * NVFP4_ERR_NONFINITE in the workspace status word (read it with
 * nvfp4_read_device_status); the logits of the rows concerned are NaN.
 *
 * Accumulation is fp32 on the tensor cores; each product x * w is exact.
 * The activations are carried into the tensor cores as fp16 after an exact
 * power-of-two rescale per token (exact for every bf16 value within 2^28
 * of the token's largest magnitude; smaller ones keep at least an absolute
 * accuracy of 2^-39 of that maximum).  The result is deterministic: no
 * floating-point atomics, fixed reduction order.
 */
nvfp4_status w4a16_lm_head(const void *x, int64_t M, int64_t K, const uint8_t *packed,
                           const uint8_t *scales, const float *global_scale, int64_t N,
                           void *logits, int out_dtype, void *workspace, size_t workspace_bytes,
                           void *stream);

/* ------------------------------------------- fused greedy argmax */

/*
 * Workspace bytes w4a16_lm_head_argmax needs: those of w4a16_lm_head plus
 * 128 bytes per token (one 64-bit maximum per line, M rounded up to the
 * token tile) and a counter.  Returns 0 for shapes the call rejects
 * (including N == 0).
 */
size_t w4a16_lm_head_argmax_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * Greedy next-token choice fused into the W4A16 product: for each token m,
 *   token_ids[m]  = the smallest n with logits[m, n] == max_n' logits[m, n'],
 *   max_logits[m] = that largest logit,
 * where logits[m, n] are bit for bit the fp32 values w4a16_lm_head writes
 * with NVFP4_OUT_F32 for the same inputs.  -0 and +0 count as equal (a zero
 * maximum is returned as +0) and a NaN logit as larger than every number
 * (first NaN wins).  The [M, N] logits are never written to memory: each
 * warp compares its logits with the token's current maximum and, where one
 * may reach it, merges its best (logit, row) with one 64-bit atomic
 * maximum, so the result does not depend on the schedule.
 *
 * The pages define the logits (the lm_head output of
 * `_LMHeadNvfp4Method.apply`), not what a sampler does with them; this call
 * is the greedy (temperature 0) reading of "pick the next token".
 *
 *   x, packed, scales, global_scale, K
 *                as for w4a16_lm_head.
 *   N            vocabulary rows, 1 <= N < 2^31 (N == 0 is NVFP4_ERR_SHAPE).
 *   M            tokens, M >= 0 (M == 0 is a no-op).
 *   token_ids    int64 [M], device, 8-byte aligned.
 *   max_logits   fp32 [M], device, 4-byte aligned, or NULL to skip.
 *   workspace    device, >= w4a16_lm_head_argmax_workspace_bytes(M, N, K),
 *                256-byte aligned.
 * A device-side timeout (NVFP4_ERR_TIMEOUT in the workspace status word)
 * leaves token_ids and max_logits undefined.
 */
nvfp4_status w4a16_lm_head_argmax(const void *x, int64_t M, int64_t K, const uint8_t *packed,
                                  const uint8_t *scales, const float *global_scale, int64_t N,
                                  int64_t *token_ids, float *max_logits, void *workspace,
                                  size_t workspace_bytes, void *stream);

/* ------------------------------------------------ fused top-k */

#define NVFP4_TOPK_MAX 128 /* largest k of w4a16_lm_head_topk */

/*
 * Workspace bytes w4a16_lm_head_topk needs (0 for rejected shapes).  Up to
 * 256 tokens and N <= 262144: those of w4a16_lm_head plus the fp32 logits,
 * M x N x 4 bytes, and 4 bytes per token and 32 rows (their maxima).
 * Otherwise: those of w4a16_lm_head_argmax plus the candidate store, M x N x
 * 4 bytes (every logit is a candidate at most once), 8 bytes per token and
 * 32 rows of candidate flags, and per token a 4,112-byte histogram and a
 * bitmap of one bit per 32 rows (rounded up to the token tile); only the
 * 32-byte pieces of the candidate store that hold a candidate reaching its
 * token's threshold (zeros beside it), and their groups' flags, are ever
 * written.
 */
size_t w4a16_lm_head_topk_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t k);

/*
 * The k largest logits of each token, fused into the W4A16 product:
 *   token_ids[m, j], values[m, j] (j = 0 .. k-1) = the rows and logits of
 *   token m's k largest, in descending order; of equal logits the smaller
 *   row comes first,
 * where the logits are bit for bit the fp32 values w4a16_lm_head writes with
 * NVFP4_OUT_F32 for the same inputs, with -0 and +0 equal (a zero is
 * returned as +0) and a NaN above every number, as in w4a16_lm_head_argmax
 * (whose answer is column 0 here).  Up to 256 tokens (N <= 262144) the
 * product writes the fp32 logits and, per token, the largest of every 32
 * rows into the workspace, and one CTA per token bounds its k-th largest
 * logit from those maxima and ranks the few logits that reach the bound.
 * Beyond, the [M, N] logits are never written: the epilogue keeps only the
 * logits that reach the token's running threshold, a lower bound of its
 * k-th largest that rises with a histogram of the largest kept candidate of
 * every 32 rows, and a second kernel selects the exact k largest of those.  The result
 * does not depend on the route or the schedule.
 *
 * The pages define the logits, not a sampler; this is the top-k filter a
 * sampler applies to them, for the same reason as the argmax.
 *
 *   x, packed, scales, global_scale, K, M, N
 *                as for w4a16_lm_head_argmax; M x N <= 2^36.
 *   k            1 <= k <= min(N, NVFP4_TOPK_MAX), else NVFP4_ERR_SHAPE.
 *   token_ids    int64 [M, k] row-major, device, 8-byte aligned.
 *   values       fp32 [M, k], device, 4-byte aligned, or NULL to skip.
 *   workspace    device, >= w4a16_lm_head_topk_workspace_bytes(M, N, K, k),
 *                256-byte aligned; no state is kept in it between calls.
 * Three kernels on `stream` (activation prep, product, selection), no host
 * synchronisation; graph-capturable.  A device-side timeout
 * (NVFP4_ERR_TIMEOUT in the workspace status word) leaves token_ids and
 * values undefined.
 */
nvfp4_status w4a16_lm_head_topk(const void *x, int64_t M, int64_t K, const uint8_t *packed,
                                const uint8_t *scales, const float *global_scale, int64_t N,
                                int64_t k, int64_t *token_ids, float *values, void *workspace,
                                size_t workspace_bytes, void *stream);

/* ------------------------------------------------------- fp8 copy */

/*
 * The "fp8" lm_head copy -- `quantized_lm_head_copy` on the page
 * "vllm.model_executor.layers.quantization.online.lm_head": per-row weight
 * scales and per-token activation scales on an FP8 linear kernel (the
 * FP8_PER_CHANNEL_PER_TOKEN scheme of "vllm/model_executor/layers/
 * quantization/modelopt.py").  The quantizer body is not on the pages; the
 * reading implemented, for one row v of W (or one token of x):
 *   s = max(fl32(max|v| / 448), fl32(1e-12)),  r = fl32(1 / s),
 *   q[k] = e4m3(fl32(v[k] * r)), nearest even, saturated to +-448, sign kept.
 */

/* Workspace bytes of fp8_quantize_rows / fp8_refresh (the status word);
 * 0 for shapes they reject. */
size_t fp8_quantize_workspace_bytes(int64_t N, int64_t K);

/*
 * Quantize the rows of W to the fp8 copy.
 *   W          bf16 [N, K], device, 16-byte aligned.  N >= 1, K % 16 == 0,
 *              K <= 65536.
 *   q          u8 (float8_e4m3fn) [N, K], device, 16-byte aligned.  Written.
 *   row_scale  f32 [N], device.  Written: s of each row (dequant = e4m3(q) * s).
 *   workspace  device, >= fp8_quantize_workspace_bytes(N, K), 256-byte
 *              aligned: the status word (NVFP4_ERR_NONFINITE if W holds an
 *              Inf or NaN; that row's outputs are then unspecified).
 * One kernel, one read of W and one write of q; no host synchronization.
 */
nvfp4_status fp8_quantize_rows(const void *W, int64_t N, int64_t K, uint8_t *q, float *row_scale,
                               void *workspace, size_t workspace_bytes, void *stream);

/* Re-derive the fp8 copy in place after W changed (`refresh_quantized_lm_heads`):
 * same arguments, same buffers, addresses unchanged. */
nvfp4_status fp8_refresh(const void *W, int64_t N, int64_t K, uint8_t *q, float *row_scale,
                         void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes of w8a8_lm_head: x as e4m3 (M_pad * K bytes), one scale
 * per token, the status word and room for split-K partials.  0 for shapes
 * the call rejects. */
size_t w8a8_lm_head_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * logits[m, n] = fl32(fl32(acc[m, n] * s_x[m]) * row_scale[n]), acc the fp32
 * sum over k of e4m3(q_x[m, k]) * e4m3(q[n, k]), where (q_x, s_x) is x
 * quantized per token by the rule above (inside the call, into the
 * workspace).
 *   x          bf16 [M, K], device, 16-byte aligned.  M >= 0 (0: no-op),
 *              K % 16 == 0, 16 <= K <= 16384.
 *   q, row_scale  as fp8_quantize_rows writes them for W[N, K].
 *   N          vocabulary rows, N >= 0 (0: no-op).
 *   logits     [M, N] fp32 (NVFP4_OUT_F32) or bf16 (NVFP4_OUT_BF16), device,
 *              16-byte aligned.
 *   workspace  device, >= w8a8_lm_head_workspace_bytes(M, N, K), 256-byte aligned.
 * Tensor-core fp32 accumulation, deterministic (no floating-point atomics).
 */
nvfp4_status w8a8_lm_head(const void *x, int64_t M, int64_t K, const uint8_t *q,
                          const float *row_scale, int64_t N, void *logits, int out_dtype,
                          void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes of w8a8_lm_head_argmax (0 for rejected shapes, N == 0 included). */
size_t w8a8_lm_head_argmax_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * The greedy argmax of the W8A8 logits fused into the product, with the
 * semantics of w4a16_lm_head_argmax: token_ids[m] is the smallest n whose
 * logit (bit for bit the fp32 value w8a8_lm_head writes) is the row maximum,
 * max_logits[m] that value (+0 for a zero maximum; NaN ranks highest).
 * Arguments as for w8a8_lm_head, with token_ids int64 [M] (8-byte aligned)
 * and max_logits fp32 [M] or NULL; N >= 1.
 */
nvfp4_status w8a8_lm_head_argmax(const void *x, int64_t M, int64_t K, const uint8_t *q,
                                 const float *row_scale, int64_t N, int64_t *token_ids,
                                 float *max_logits, void *workspace, size_t workspace_bytes,
                                 void *stream);

/* Workspace bytes of w8a8_lm_head_topk (0 for rejected shapes or k). */
size_t w8a8_lm_head_topk_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t k);

/*
 * The k largest W8A8 logits of each token, fused (semantics and limits of
 * w4a16_lm_head_topk; the logits are those w8a8_lm_head writes in fp32):
 * token_ids int64 [M, k], values fp32 [M, k] or NULL.
 */
nvfp4_status w8a8_lm_head_topk(const void *x, int64_t M, int64_t K, const uint8_t *q,
                               const float *row_scale, int64_t N, int64_t k, int64_t *token_ids,
                               float *values, void *workspace, size_t workspace_bytes,
                               void *stream);

/* ----------------------------------------------- grouped W4A16 (MoE) */

/* Workspace bytes of w4a16_grouped_gemm; 0 for rejected shapes. */
size_t w4a16_grouped_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t n_groups);

/*
 * The NVFP4 W4A16 product of a mixture-of-experts layer, all experts in one
 * call (the `w13 [E, 2I, H/2]` / `w2 [E, H, I/2]` layouts of
 * `ModelOptNvFp4FusedMoE.create_weights` on the page
 * "vllm/model_executor/layers/quantization/modelopt.py", with one global
 * scale per expert as its `w13_weight_scale_2` / `w2_weight_scale_2`):
 *   out[m, n] = global[e] * sum_k x[m, k] * e2m1(code[e, n, k]) * f32(scale[e, n, k/16])
 * for every token row m of group e, group_offsets[e] <= m < group_offsets[e + 1].
 *   x              bf16 [M, K], device: token rows already grouped by expert
 *                  (routing and the final combine are the caller's).
 *                  K % 16 == 0 (K % 256 != 0 stages rows as w4a16_lm_head).
 *   group_offsets  int32 [n_groups + 1], device, non-decreasing, [0] = 0,
 *                  [n_groups] = M (rows outside [0, M) are never read or
 *                  written).  Read by the kernels, never by the host: the call
 *                  can be captured in a CUDA graph whatever the routing.
 *   n_groups       experts, 1 <= n_groups <= 256.
 *   packed, scales u8 [n_groups, N, K/2] and [n_groups, N, K/16], each expert as
 *                  nvfp4_quantize_rows writes it; 16-byte aligned.
 *   global_scales  f32 [n_groups], device: each expert's global scale.
 *   out            [M, N] fp32 or bf16, device, 16-byte aligned.
 *   workspace      >= w4a16_grouped_workspace_bytes(M, N, K, n_groups), 256-byte aligned.
 * Accumulation and accuracy as w4a16_lm_head.
 */
nvfp4_status w4a16_grouped_gemm(const void *x, int64_t M, int64_t K, const int32_t *group_offsets,
                                int64_t n_groups, const uint8_t *packed, const uint8_t *scales,
                                const float *global_scales, int64_t N, void *out, int out_dtype,
                                void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------- W4A4 NVFP4 */

/*
 * Bytes of the 128x4-interleaved copy of NVFP4 block scales of W[N, K]:
 * round_up(N, 128) * round_up(K/16, 4).  0 for rejected shapes (K % 16 != 0).
 */
size_t nvfp4_swizzled_scales_bytes(int64_t N, int64_t K);

/*
 * Re-lay row-major E4M3 block scales [N, K/16] (as nvfp4_quantize_rows writes
 * them) into the order block-scaled FP4 tensor cores read, `swizzle_blockscale`
 * on the page "vllm.model_executor.layers.quantization.compressed_tensors.
 * schemes": rows padded to a multiple of 128 and columns (K/16) to a
 * multiple of 4, taken in 512-byte atoms of 128 rows x 4 columns, ordered
 * [row / 128][column / 4]; inside an atom, row 32 a + b and column d sit at
 * byte b * 16 + a * 4 + d.  Padding rows and columns are zero.
 *   scales  u8 [N, K/16], device, 4-byte aligned.  K % 16 == 0.
 *   out     u8, device, 16-byte aligned, nvfp4_swizzled_scales_bytes(N, K).
 * Run it after every nvfp4_quantize_rows / nvfp4_refresh that the W4A4
 * product will read.
 */
nvfp4_status nvfp4_swizzle_scales(const uint8_t *scales, int64_t N, int64_t K, uint8_t *out,
                                  void *stream);

/* Workspace bytes of w4a4_lm_head (x as NVFP4 codes and interleaved scales,
 * alpha per token, status, split-K partials); 0 for rejected shapes. */
size_t w4a4_lm_head_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * The W4A4 NVFP4 product (`CompressedTensorsW4A4Fp4.apply_weights` on the
 * page "...compressed_tensors.schemes"; alpha as `maybe_fuse_global_scales`
 * on "vllm/model_executor/layers/quantization/modelopt.py"): x is quantized
 * inside the call to NVFP4 with the weight's rule (per 16 values an E4M3
 * scale e4m3(min(vmax / 6 / input_global_scale, 448)), E2M1 codes of
 * x / (scale * input_global_scale), ties to even), then
 *   logits[m, n] = fl32(acc[m, n] * alpha),  alpha = fl32(input_global_scale * global_scale),
 * acc the fp32 tensor-core sum of the block-scaled E2M1 products (each exact).
 *   x                   bf16 [M, K], device, 16-byte aligned; K % 16 == 0 (when
 *                       K % 32 != 0 the weight codes are first copied into the
 *                       workspace with a 16-byte-multiple row stride).
 *   packed, global_scale  as nvfp4_quantize_rows writes them for W[N, K].
 *   scales_swizzled     nvfp4_swizzle_scales of that call's scales.
 *   input_global_scale  f32 [1], device: the activation dequant multiplier
 *                       (amax_x / 2688 for a calibrated amax_x; positive and
 *                       finite, else NVFP4_ERR_NONFINITE in the status word).
 *   logits              [M, N] fp32 or bf16, device, 16-byte aligned.
 *   workspace           >= w4a4_lm_head_workspace_bytes(M, N, K), 256-byte aligned.
 */
nvfp4_status w4a4_lm_head(const void *x, int64_t M, int64_t K, const uint8_t *packed,
                          const uint8_t *scales_swizzled, const float *global_scale,
                          const float *input_global_scale, int64_t N, void *logits,
                          int out_dtype, void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes of w4a4_lm_head_argmax (0 for rejected shapes, N == 0 included). */
size_t w4a4_lm_head_argmax_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* The greedy argmax of the W4A4 logits, fused (semantics of
 * w4a16_lm_head_argmax; the logits are those w4a4_lm_head writes in fp32). */
nvfp4_status w4a4_lm_head_argmax(const void *x, int64_t M, int64_t K, const uint8_t *packed,
                                 const uint8_t *scales_swizzled, const float *global_scale,
                                 const float *input_global_scale, int64_t N, int64_t *token_ids,
                                 float *max_logits, void *workspace, size_t workspace_bytes,
                                 void *stream);

/* Workspace bytes of w4a4_lm_head_topk (0 for rejected shapes or k). */
size_t w4a4_lm_head_topk_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t k);

/* The k largest W4A4 logits of each token, fused (semantics and limits of
 * w4a16_lm_head_topk; the logits are those w4a4_lm_head writes in fp32). */
nvfp4_status w4a4_lm_head_topk(const void *x, int64_t M, int64_t K, const uint8_t *packed,
                               const uint8_t *scales_swizzled, const float *global_scale,
                               const float *input_global_scale, int64_t N, int64_t k,
                               int64_t *token_ids, float *values, void *workspace,
                               size_t workspace_bytes, void *stream);

/* ------------------------------------------- allocation-free variant */

/* Size of the fixed device scratch array behind w4a16_lm_head_noalloc. */
#define NVFP4_NOALLOC_SCRATCH_BYTES (8u << 20)

/*
 * The same product as w4a16_lm_head, for callers that cannot allocate device
 * memory: runtimes that fix their device-memory budget at start-up and allow
 * no later cudaMalloc (which may also synchronize the device), or plain C
 * callers with no device allocator to take a workspace from.  The pages have
 * no counterpart of this call; it exists for such callers only.
 *
 * Arguments, layouts, ownership and accuracy are those of w4a16_lm_head
 * minus the workspace.  The scratch is one static device array of
 * NVFP4_NOALLOC_SCRATCH_BYTES (8 MiB) that every GPU loading the library
 * holds until the process exits.  Its first call on a device looks up the
 * array's device address (cudaGetSymbolAddress) with that device current;
 * make that first call before any stream capture.  Shapes whose rescaled
 * activations and split-K partials do not fit (M_pad * K * 2 bytes plus up to
 * SMs * 128 * M_pad * 4 bytes, M_pad = M rounded up to 16, or to 128 above
 * 128 tokens; for K % 256 != 0 also the staged weight rows, N * K/16 bytes
 * and more) return NVFP4_ERR_SCRATCH_LIMIT before anything is enqueued;
 * for example M <= 64 at K <= 8192 fits.  Nothing is
 * allocated: no cudaMalloc, no cudaFree, no allocating library routine.
 *
 * The array's address is looked up once per CUDA context (the primary
 * context of each device, or one the caller made current) and cached; the
 * first call in a context does the lookup, later ones read the cache
 * without a lock.
 *
 * Every call shares the array.  Each call rewrites what it reads and clears
 * the status word first, but calls that overlap on the GPU (unordered
 * streams) race on the array.  Device-side conditions (a NaN block scale, a
 * pipeline wait that timed out) go to the status word at the start of the
 * array, which w4a16_lm_head_noalloc_status reads.
 */
nvfp4_status w4a16_lm_head_noalloc(const void *x, int64_t M, int64_t K, const uint8_t *packed,
                                   const uint8_t *scales, const float *global_scale, int64_t N,
                                   void *logits, int out_dtype, void *stream);

/*
 * The device status word the last w4a16_lm_head_noalloc call on `stream` in
 * the current context left in the fixed scratch (what
 * nvfp4_read_device_status reads from a workspace).  Like that call it
 * synchronizes `stream`; the pages have no counterpart.
 *   status_out  host, receives an nvfp4_status value.
 */
nvfp4_status w4a16_lm_head_noalloc_status(int32_t *status_out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_LM_HEAD_H_ */
