/*
 * nvfp4_oracle.c -- TEST INFRASTRUCTURE: a plain, slow CPU oracle of the
 * online NVFP4 lm_head path.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg use it; the product library never links,
 * loads or calls it, and it shares no code with the CUDA sources.
 *
 * Build with -ffp-contract=off and without fast-math: every float step
 * below is one IEEE binary32 operation, rounded to nearest even.
 *
 * What it follows (page titles and sections):
 *  - vllm.model_executor.layers.quantization.online.lm_head, `_quantize_nvfp4`:
 *    global scale = amax / (FLOAT4_E2M1_MAX * finfo(e4m3fn).max) clamped at
 *    1e-12, its reciprocal handed to the per-16 block quantizer, the E2M1
 *    code map {0,1,2,3,4,6,8,12} -> 0..7 with the sign in bit 3 set for
 *    values < 0, low-nibble-first packing, E4M3 block scales.
 *  - vllm/model_executor/layers/quantization/modelopt.py, `KNvfp4Static`:
 *    K % 16 == 0; the global scale is the raw amax/2688 dequant multiplier
 *    (no reciprocal), so FLOAT4_E2M1_MAX = 6 and the e4m3 maximum is 448.
 *  - vllm.model_executor.layers.quantization.compressed_tensors.schemes,
 *    `CompressedTensorsW4A16Fp4`: logits = x . dequant(W)^T with
 *    dequant = e2m1(code) * f32(block scale) * global scale.
 *
 * The body of the per-16 block quantizer is not printed on the pages.  The
 * reading used here (and stated with each function): block scale
 * t = (vmax * fl32(1/6)) * inv_global, clamped to <= 448, rounded to E4M3
 * (nearest even); values are scaled by 1 / (f32(scale) * global), clamped
 * to [-6, 6] and rounded to the E2M1 grid, ties to the even code.
 *
 * The fp8 copy (per-row E4M3 weights, per-token E4M3 activations) is at the
 * end of the file, with its own reading stated there.
 *
 * Parity pins: every function here is checked in tests/ against facts the
 * pages or mathematics fix (code table, packing order, closed forms,
 * brute-force nearest rounding, torch's own e4m3 cast, numpy matmul).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ basics */

static float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static int bf16_is_finite(uint16_t h) { return (h & 0x7F80u) != 0x7F80u; }

/* Constants of `_quantize_nvfp4` (page 1): FLOAT4_E2M1_MAX = 6 and
 * finfo(float8_e4m3fn).max = 448, both exact in binary32. */
#define E2M1_MAX 6.0f
#define E4M3_MAX 448.0f

/* ------------------------------------------------------------ E4M3 (fn) */

/*
 * Decode one float8_e4m3fn byte: 1 sign bit, 4 exponent bits (bias 7),
 * 3 mantissa bits, no infinities, S.1111.111 is NaN.  Normal values are
 * (1 + m/8) * 2^(e-7), subnormals m * 2^-9.
 */
float oracle_e4m3_decode(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  float v = (e == 0) ? ldexpf((float)m, -9) : ldexpf((float)(8 + m), e - 10);
  return s ? -v : v;
}

/*
 * Encode a float t in [0, 448] to float8_e4m3fn with round-to-nearest-even,
 * subnormals included (the `.to(torch.float8_e4m3fn)` cast of the block
 * scales in `_quantize_nvfp4`).  Callers clamp t to <= 448 first.
 */
uint8_t oracle_e4m3_encode(float t) {
  if (!(t > 0.0f)) return 0; /* zero (and the non-positive edge) */
  int e2;
  (void)frexpf(t, &e2); /* t = f * 2^e2, f in [0.5, 1) */
  int E = e2 - 1;       /* t = 1.xxx * 2^E */
  if (E < -6) {
    /* subnormal range: t = q * 2^-9, q rounded to an integer 0..8; q = 8 is
     * the smallest normal 2^-6, whose code is 0x08 as well. */
    float q = rintf(ldexpf(t, 9)); /* exact scaling, then nearest even */
    return (uint8_t)q;
  }
  float frac = ldexpf(t, -E) - 1.0f; /* in [0, 1), exact */
  float mq = rintf(frac * 8.0f);     /* 0..8, nearest even */
  if (mq == 8.0f) {
    mq = 0.0f;
    E += 1;
  }
  return (uint8_t)(((E + 7) << 3) | (int)mq);
}

/* Element-wise encode of an array (a loop over oracle_e4m3_encode). */
void oracle_e4m3_encode_array(const float *t, int64_t n, uint8_t *out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(t[i]);
}

/* ------------------------------------------------------------ E2M1 grid */

/* E2M1 magnitudes, indexed by the 3-bit magnitude code (`_quantize_nvfp4`:
 * the doubled magnitudes 0,1,2,3,4,6,8,12 map to codes 0..7). */
static const float E2M1_GRID[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

/* code_of[2|v|]: the page's lookup from doubled magnitude to code. */
static int code_of_doubled(int twice_mag) {
  static const int table[13] = {0, 1, 2, 3, 4, -1, 5, -1, 6, -1, -1, -1, 7};
  return (twice_mag >= 0 && twice_mag <= 12) ? table[twice_mag] : -1;
}

/*
 * Round a scaled value q (already clamped to [-6, 6]) to the E2M1 grid:
 * nearest grid point, a tie goes to the point with the even code.  Written
 * as the explicit intervals between neighbouring grid points; the sign of q
 * is kept (so a negative q that rounds to zero gives -0.0).
 */
float oracle_e2m1_round(float q) {
  float a = fabsf(q), v;
  if (a <= 0.25f) v = 0.0f;       /* tie 0.25 -> 0   (code 0) */
  else if (a < 0.75f) v = 0.5f;
  else if (a <= 1.25f) v = 1.0f;  /* ties 0.75, 1.25 -> 1 (code 2) */
  else if (a < 1.75f) v = 1.5f;
  else if (a <= 2.5f) v = 2.0f;   /* ties 1.75, 2.5 -> 2 (code 4) */
  else if (a < 3.5f) v = 3.0f;
  else if (a <= 5.0f) v = 4.0f;   /* ties 3.5, 5 -> 4 (code 6) */
  else v = 6.0f;
  return copysignf(v, q);
}

/* The 4-bit code of a grid value v: code_of[2|v|] | (v < 0) << 3. */
uint8_t oracle_e2m1_code(float v) {
  int c = code_of_doubled((int)(fabsf(v) * 2.0f));
  if (c < 0) return 0xFF; /* not a grid value: caller bug */
  return (uint8_t)(c | ((v < 0.0f) ? 8 : 0));
}

/* Decode a 4-bit code: bit 3 is the sign, bits 2..0 index the grid. */
float oracle_e2m1_decode(uint8_t code) {
  float m = E2M1_GRID[code & 7];
  return (code & 8) ? -m : m;
}

/* Element-wise grid rounding of an array (a loop over oracle_e2m1_round). */
void oracle_e2m1_round_array(const float *q, int64_t n, float *out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e2m1_round(q[i]);
}

/* -------------------------------------------------------- global scale */

/*
 * weight_amax: max |W| over all N*K elements (bf16 -> f32 is exact, so the
 * max is exact).  Returns -1 if any element is not finite.
 */
int oracle_weight_amax(const uint16_t *W, int64_t n_elem, float *amax_out) {
  float amax = 0.0f;
  int bad = 0;
#pragma omp parallel for reduction(max : amax) reduction(| : bad) schedule(static)
  for (int64_t i = 0; i < n_elem; ++i) {
    if (!bf16_is_finite(W[i])) bad |= 1;
    float a = fabsf(bf16_to_f32(W[i]));
    if (a > amax) amax = a;
  }
  *amax_out = amax;
  return bad ? -1 : 0;
}

/*
 * `_quantize_nvfp4`: global = fp32(amax) / (6 * 448), clamped at 1e-12;
 * inv_global = 1 / global.  Both are binary32 (the division by the exact
 * constant 2688 and the reciprocal each round once).
 */
void oracle_global_scale(float amax, float *global_out, float *inv_global_out) {
  float g = amax / (E2M1_MAX * E4M3_MAX); /* 2688.0f, exact */
  const float lo = 1e-12f;
  if (g < lo) g = lo;
  *global_out = g;
  *inv_global_out = 1.0f / g;
}

/* ------------------------------------------------- per-16 block quantizer */

/*
 * One block of 16 consecutive values along K (the block quantizer called by
 * `_quantize_nvfp4` with block size 16):
 *   vmax  = max |x|
 *   t     = min((vmax * fl32(1/6)) * inv_global, 448)
 *   scale = e4m3(t)                               -> *scale_byte
 *   sf    = f32(scale)
 *   r     = sf == 0 ? 0 : 1 / (sf * global)
 *   v[i]  = grid(clamp(x[i] * r, -6, 6))          -> values[i]
 */
void oracle_quantize_block(const float x[16], float global, float inv_global,
                           float values[16], uint8_t *scale_byte) {
  float vmax = 0.0f;
  for (int i = 0; i < 16; ++i) {
    float a = fabsf(x[i]);
    if (a > vmax) vmax = a;
  }
  const float inv_e2m1_max = 1.0f / E2M1_MAX;
  float t = (vmax * inv_e2m1_max) * inv_global;
  if (t > E4M3_MAX) t = E4M3_MAX;
  uint8_t s8 = oracle_e4m3_encode(t);
  float sf = oracle_e4m3_decode(s8);
  float r = (sf == 0.0f) ? 0.0f : 1.0f / (sf * global);
  for (int i = 0; i < 16; ++i) {
    float q = x[i] * r;
    if (q > E2M1_MAX) q = E2M1_MAX;
    if (q < -E2M1_MAX) q = -E2M1_MAX;
    values[i] = oracle_e2m1_round(q);
  }
  *scale_byte = s8;
}

/*
 * Quantize one row w[0..K) with a given global scale into K/2 packed bytes
 * and K/16 scale bytes.  The code of a grid value is
 * code_of[2|v|] | (v < 0) << 3 and byte j holds codes 2j (low nibble) and
 * 2j+1 (high nibble), as `_quantize_nvfp4` packs them.
 */
static void quantize_one_row(const uint16_t *w, int64_t K, float global, float inv_global,
                             uint8_t *prow, uint8_t *srow) {
  for (int64_t b = 0; b < K / 16; ++b) {
    float x[16], v[16];
    for (int j = 0; j < 16; ++j) x[j] = bf16_to_f32(w[b * 16 + j]);
    oracle_quantize_block(x, global, inv_global, v, &srow[b]);
    for (int j = 0; j < 8; ++j) {
      uint8_t lo = oracle_e2m1_code(v[2 * j]);
      uint8_t hi = oracle_e2m1_code(v[2 * j + 1]);
      prow[b * 8 + j] = (uint8_t)(lo | (hi << 4));
    }
  }
}

/*
 * Quantize the listed rows of W[N, K] with a given global scale, writing
 * listed row i to row i of packed_out [n_rows, K/2] and scales_out
 * [n_rows, K/16].  Used to check a sample of rows of a large tensor.
 */
void oracle_quantize_rows(const uint16_t *W, int64_t N, int64_t K, const int64_t *rows,
                          int64_t n_rows, float global, float inv_global,
                          uint8_t *packed_out, uint8_t *scales_out) {
  (void)N;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n_rows; ++i)
    quantize_one_row(W + rows[i] * K, K, global, inv_global, packed_out + i * (K / 2),
                     scales_out + i * (K / 16));
}

/*
 * The whole of `_quantize_nvfp4` for W[N, K] (bf16 bit patterns):
 * packed u8[N, K/2], scales e4m3[N, K/16] (row-major, the checkpoint
 * layout) and the fp32 global scale.  Returns 0, or -1 for a non-finite W,
 * -2 for a shape the method rejects (K % 16 != 0, or an empty tensor).
 * The page walks the rows in chunks of 8192; chunking changes nothing
 * because the global scale is fixed before the first chunk.
 */
int oracle_quantize(const uint16_t *W, int64_t N, int64_t K, uint8_t *packed,
                    uint8_t *scales, float *global_out) {
  if (N <= 0 || K <= 0 || K % 16 != 0) return -2;
  float amax, g, ig;
  if (oracle_weight_amax(W, N * K, &amax) != 0) return -1;
  oracle_global_scale(amax, &g, &ig);
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n)
    quantize_one_row(W + n * K, K, g, ig, packed + n * (K / 2), scales + n * (K / 16));
  *global_out = g;
  return 0;
}

/* ------------------------------------------------------------- dequant */

/* w[n, k] = e2m1(code) * f32(scale[n, k/16]) * global, in double (exact). */
void oracle_dequant_rows(const uint8_t *packed, const uint8_t *scales, float global,
                         int64_t K, const int64_t *rows, int64_t n_rows, double *out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n_rows; ++i) {
    const uint8_t *p = packed + rows[i] * (K / 2);
    const uint8_t *s = scales + rows[i] * (K / 16);
    for (int64_t k = 0; k < K; ++k) {
      uint8_t byte = p[k / 2];
      uint8_t code = (k % 2 == 0) ? (byte & 15) : (byte >> 4);
      out[i * K + k] = (double)oracle_e2m1_decode(code) *
                       (double)oracle_e4m3_decode(s[k / 16]) * (double)global;
    }
  }
}

/* ------------------------------------------------------------- logits */

/*
 * logits[m, j] = sum_k x[m, k] * w[cols[j], k] in double, for the listed
 * vocabulary rows cols[0..n_cols) (all rows: cols = 0..N-1).  x is bf16
 * [M, K]; w is the dequantized weight of oracle_dequant_rows.  out is
 * [M, n_cols].  Plain loops, summed in k order.
 */
void oracle_logits_cols(const uint16_t *x, int64_t M, int64_t K, const uint8_t *packed,
                        const uint8_t *scales, float global, const int64_t *cols,
                        int64_t n_cols, double *out) {
#pragma omp parallel
  {
    double *w = (double *)malloc((size_t)K * sizeof(double));
#pragma omp for schedule(dynamic, 64)
    for (int64_t j = 0; j < n_cols; ++j) {
      oracle_dequant_rows(packed, scales, global, K, &cols[j], 1, w);
      for (int64_t m = 0; m < M; ++m) {
        const uint16_t *xr = x + m * K;
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) acc += (double)bf16_to_f32(xr[k]) * w[k];
        out[m * n_cols + j] = acc;
      }
    }
    free(w);
  }
}

/* ============================================================== W4A4 */
/*
 * W4A4 NVFP4 (`CompressedTensorsW4A4Fp4.apply_weights` on the page
 * "vllm.model_executor.layers.quantization.compressed_tensors.schemes"):
 * x is quantized per 16 values with the weight's rule against the
 * per-tensor input global scale g_x (a dequant multiplier; its inverse is
 * fl32(1/g_x)), and logits = (g_x * g_w) * sum e2m1*sf_x * e2m1*sf_w, here
 * as the float64 sum of the dequantized operands' products.
 */
void oracle_w4a4_logits_cols(const uint16_t *x, int64_t M, int64_t K, float gx,
                             const uint8_t *packed, const uint8_t *scales, float gw,
                             const int64_t *cols, int64_t n_cols, double *out) {
  const float igx = 1.0f / gx;
  uint8_t *xp = (uint8_t *)malloc((size_t)M * (K / 2));
  uint8_t *xs = (uint8_t *)malloc((size_t)M * (K / 16));
  double *xd = (double *)malloc((size_t)M * K * sizeof(double));
  for (int64_t m = 0; m < M; ++m) quantize_one_row(x + m * K, K, gx, igx, xp + m * (K / 2), xs + m * (K / 16));
  int64_t *all = (int64_t *)malloc((size_t)M * sizeof(int64_t));
  for (int64_t m = 0; m < M; ++m) all[m] = m;
  oracle_dequant_rows(xp, xs, gx, K, all, M, xd);
#pragma omp parallel
  {
    double *w = (double *)malloc((size_t)K * sizeof(double));
#pragma omp for schedule(dynamic, 64)
    for (int64_t j = 0; j < n_cols; ++j) {
      oracle_dequant_rows(packed, scales, gw, K, &cols[j], 1, w);
      for (int64_t m = 0; m < M; ++m) {
        const double *xr = xd + m * K;
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) acc += xr[k] * w[k];
        out[m * n_cols + j] = acc;
      }
    }
    free(w);
  }
  free(all);
  free(xd);
  free(xs);
  free(xp);
}

/*
 * `swizzle_blockscale` (same page): pad the [N, C] E4M3 block-scale matrix
 * to rows a multiple of 128 and columns a multiple of 4, view it as
 * [N'/128][4][32][C'/4][4] and store it in the order [N'/128][C'/4][32][4][4].
 * Plain loops over the destination.
 */
void oracle_swizzle_scales(const uint8_t *scales, int64_t N, int64_t C, uint8_t *out) {
  const int64_t Np = (N + 127) / 128 * 128, Cp = (C + 3) / 4 * 4;
  int64_t o = 0;
  for (int64_t i0 = 0; i0 < Np / 128; ++i0)
    for (int64_t i4 = 0; i4 < Cp / 4; ++i4)
      for (int64_t i3 = 0; i3 < 32; ++i3)
        for (int64_t i2 = 0; i2 < 4; ++i2)
          for (int64_t i5 = 0; i5 < 4; ++i5) {
            const int64_t r = i0 * 128 + i2 * 32 + i3, c = i4 * 4 + i5;
            out[o++] = (r < N && c < C) ? scales[r * C + c] : 0;
          }
}

/* ============================================================ fp8 copy */
/*
 * The "fp8" lm_head copy of the page
 * "vllm.model_executor.layers.quantization.online.lm_head"
 * (`quantized_lm_head_copy`): per-row weight scales and per-token
 * activation scales on an FP8 (E4M3) linear kernel -- the
 * FP8_PER_CHANNEL_PER_TOKEN scheme of the page
 * "vllm/model_executor/layers/quantization/modelopt.py" (static per-channel
 * weight scale, dynamic per-token activation scale).  The quantizer body is
 * not printed; the reading used here, for a row v[0..K) of W (or of x):
 *   amax = max |v|;  s = max(fl32(amax / 448), fl32(1e-12));  r = fl32(1 / s);
 *   q[k] = e4m3(clamp(fl32(v[k] * r), -448, 448)), round to nearest even,
 *          the sign of the product kept (so -0 encodes as 0x80, as a cast does).
 * The dequantized value is e4m3(q) * s.
 */

/* Signed E4M3 encode of a float already clamped to [-448, 448]. */
static uint8_t e4m3_encode_signed(float v) {
  uint8_t mag = oracle_e4m3_encode(fabsf(v));
  return signbit(v) ? (uint8_t)(mag | 0x80u) : mag;
}

/* Per-row fp8 quantization of bf16 rows (weights, or activation tokens).
 * Returns 0, or -1 if a row holds a non-finite value (outside the method). */
int oracle_fp8_quantize_rows(const uint16_t *W, int64_t N, int64_t K, uint8_t *q,
                             float *scale) {
  int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
  for (int64_t n = 0; n < N; ++n) {
    const uint16_t *w = W + n * K;
    float amax = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
      if (!bf16_is_finite(w[k])) bad = 1;
      float a = fabsf(bf16_to_f32(w[k]));
      if (a > amax) amax = a;
    }
    float s = amax / E4M3_MAX;
    const float floor_s = 1e-12f;
    if (s < floor_s) s = floor_s;
    const float r = 1.0f / s;
    scale[n] = s;
    for (int64_t k = 0; k < K; ++k) {
      float v = bf16_to_f32(w[k]) * r;
      if (v > E4M3_MAX) v = E4M3_MAX;
      if (v < -E4M3_MAX) v = -E4M3_MAX;
      q[n * K + k] = e4m3_encode_signed(v);
    }
  }
  return bad ? -1 : 0;
}

/*
 * W8A8 logits: out[m, j] = xs[m] * ws[c] * sum_k e4m3(xq[m, k]) * e4m3(wq[c, k])
 * for c = cols[j], in double (every product and partial sum is exact in
 * double for K <= 2^20), then scaled by the two fp32 scales.
 */
void oracle_fp8_logits_cols(const uint8_t *xq, const float *xs, int64_t M, int64_t K,
                            const uint8_t *wq, const float *ws, const int64_t *cols,
                            int64_t n_cols, double *out) {
  double lut[256];
  for (int i = 0; i < 256; ++i) lut[i] = (double)oracle_e4m3_decode((uint8_t)i);
#pragma omp parallel for schedule(dynamic, 64)
  for (int64_t j = 0; j < n_cols; ++j) {
    const uint8_t *w = wq + cols[j] * K;
    for (int64_t m = 0; m < M; ++m) {
      const uint8_t *x = xq + m * K;
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k) acc += lut[x[k]] * lut[w[k]];
      out[m * n_cols + j] = acc * (double)xs[m] * (double)ws[cols[j]];
    }
  }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads of the parallel loops above (n <= 0: one per processor).  Only
 * the CPU baseline uses this, to time the oracle on one core and on all. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  omp_set_num_threads(n > 0 ? n : omp_get_num_procs());
#else
  (void)n;
#endif
}
