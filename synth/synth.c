/*
 * synth.c -- seeded synthetic inputs for the NVFP4 lm_head workloads.
 *
 * This module holds no arithmetic of the quantization method.  It only
 * draws random numbers and rounds them to bf16, so that the CPU oracle and
 * the GPU path are fed the very same bytes.  Both sides receive these
 * arrays as inputs; neither side calls into the other.
 *
 * Generator: a counter-based SplitMix64 stream.  Draw i of stream (seed, s)
 * is mix64(key(seed, s) + (i + 1) * GOLDEN), where mix64 is the SplitMix64
 * output function (Steele, Lea and Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014).  Uniforms take the top 53 bits; normals
 * use the Box-Muller transform on draw pairs (2j, 2j+1).  Being
 * counter-based, every element can be produced independently, so the fills
 * run in parallel and give the same bytes for any thread count.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define GOLDEN 0x9E3779B97F4A7C15ULL
#define TWO_PI 6.283185307179586476925286766559

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix64(seed * GOLDEN + 0x632BE59BD9B4E019ULL) ^
         mix64(stream + 0xD1B54A32D192ED03ULL);
}

static inline uint64_t draw(uint64_t key, uint64_t i) {
  return mix64(key + (i + 1) * GOLDEN);
}

/* uniform in [0, 1) */
static inline double u01(uint64_t r) { return (double)(r >> 11) * 0x1.0p-53; }

/* normal pair j of a stream: elements 2j and 2j+1 */
static inline void normal_pair(uint64_t key, uint64_t j, double *z0, double *z1) {
  double u1 = 1.0 - u01(draw(key, 2 * j)); /* (0, 1] keeps log finite */
  double u2 = u01(draw(key, 2 * j + 1));
  double r = sqrt(-2.0 * log(u1));
  double a = TWO_PI * u2;
  *z0 = r * cos(a);
  *z1 = r * sin(a);
}

static inline double normal_at(uint64_t key, uint64_t i) {
  double z0, z1;
  normal_pair(key, i >> 1, &z0, &z1);
  return (i & 1) ? z1 : z0;
}

/* double -> float (C conversion, round to nearest even) -> bf16 (RNE on the
 * bit pattern).  Inputs here are always finite. */
static inline uint16_t to_bf16(double v) {
  float f = (float)v;
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* Uniform draws of a stream, as doubles in [0, 1). */
void synth_uniform(double *out, int64_t n, uint64_t seed, uint64_t stream) {
  uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = u01(draw(key, (uint64_t)i));
}

/* Standard normal draws of a stream, as doubles. */
void synth_normal(double *out, int64_t n, uint64_t seed, uint64_t stream) {
  uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = normal_at(key, (uint64_t)i);
}

/*
 * Weight matrix W[N, K] (row-major, bf16 bit patterns):
 *   W[n, k] = bf16( sigma * row_mult[n] * z[n*K + k] * (u[n*K + k] < p ? mult : 1) )
 * z: normal stream 0 of `seed`; u: uniform stream 2 of `seed` (only drawn
 * when p > 0).  row_mult may be NULL (all ones).
 */
void synth_weight(uint16_t *W, int64_t N, int64_t K, uint64_t seed, double sigma,
                  const double *row_mult, double p, double mult) {
  uint64_t kz = stream_key(seed, 0);
  uint64_t ku = stream_key(seed, 2);
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n) {
    double rm = row_mult ? row_mult[n] : 1.0;
    for (int64_t k = 0; k < K; ++k) {
      uint64_t i = (uint64_t)(n * K + k);
      double v = sigma * rm * normal_at(kz, i);
      if (p > 0.0 && u01(draw(ku, i)) < p) v *= mult;
      W[n * K + k] = to_bf16(v);
    }
  }
}

/*
 * Activations x[M, K] (bf16 bit patterns) from normal stream 0 of `seed`.
 * With rms_normalize, each row is divided by its root-mean-square (in
 * double) before rounding to bf16.
 */
void synth_activations(uint16_t *x, int64_t M, int64_t K, uint64_t seed,
                       int rms_normalize) {
  uint64_t kz = stream_key(seed, 0);
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    double ss = 0.0;
    if (rms_normalize) {
      for (int64_t k = 0; k < K; ++k) {
        double z = normal_at(kz, (uint64_t)(m * K + k));
        ss += z * z;
      }
    }
    double inv = (rms_normalize && ss > 0.0) ? 1.0 / sqrt(ss / (double)K) : 1.0;
    for (int64_t k = 0; k < K; ++k)
      x[m * K + k] = to_bf16(normal_at(kz, (uint64_t)(m * K + k)) * inv);
  }
}

int synth_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
