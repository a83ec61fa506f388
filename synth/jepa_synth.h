/*
 * jepa_synth.h -- seeded, counter-based synthetic inputs (weights and pixels).
 *
 * This header is the ONE piece of code shared by the GPU library and the CPU
 * oracle. It holds no arithmetic of the encoder itself: it only turns
 * (seed, tensor name, element index) into a number with a stated distribution,
 * so that both sides see bit-identical weights and pixels.
 *
 * Generator (published definitions, written from them):
 *   - FNV-1a 64-bit hash of the tensor name (offset basis 0xcbf29ce484222325,
 *     prime 0x100000001b3).
 *   - SplitMix64 (Steele, Lea, Flood 2014; Vigna's reference form): state
 *     advances by the golden gamma 0x9e3779b97f4a7c15, output = mix(state) with
 *     the 30/27/31 xor-shift-multiply finaliser. Output #i of a SplitMix64
 *     started at state s is mix(s + (i+1)*gamma), so any element can be drawn
 *     without drawing the ones before it (counter-based).
 *   - stream key of a tensor = output #0 of SplitMix64 started at
 *     (seed ^ fnv1a64(name)).
 *   - uniform double in [0,1): top 53 bits of a 64-bit output times 2^-53.
 *   - normal: Box-Muller, z = sqrt(-2 ln(1-u1)) * cos(2 pi u2) with u1, u2 the
 *     uniforms of outputs #2i and #2i+1 (the sine branch is discarded).
 *
 * ln and cos are computed here with IEEE basic operations only (textbook
 * series: ln m = 2 atanh((m-1)/(m+1)) after frexp, and Taylor series of sin/cos
 * after quadrant reduction), so the numbers do not depend on the platform's
 * libm. Every translation unit that includes this header must be compiled with
 * floating-point contraction off (-ffp-contract=off) so that x86-64 and aarch64
 * builds produce the same bits.
 *
 * Rounding to bfloat16 (round to nearest, ties to even) is part of defining a
 * bf16 input tensor and is done here too.
 */
#ifndef JEPA_SYNTH_H
#define JEPA_SYNTH_H

#include <stdint.h>
#include <stddef.h>
#include <string.h>
#include <math.h>

#ifdef __cplusplus
extern "C" {
#endif

#define JSYNTH_GAMMA 0x9e3779b97f4a7c15ULL

static inline uint64_t jsynth_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
  return z ^ (z >> 31);
}

/* Output #i (i >= 0) of a SplitMix64 generator whose state starts at s. */
static inline uint64_t jsynth_splitmix_at(uint64_t s, uint64_t i) {
  return jsynth_mix64(s + (i + 1ULL) * JSYNTH_GAMMA);
}

static inline uint64_t jsynth_fnv1a64(const char* name) {
  uint64_t h = 0xcbf29ce484222325ULL;
  for (const unsigned char* p = (const unsigned char*)name; *p; ++p) {
    h ^= (uint64_t)(*p);
    h *= 0x100000001b3ULL;
  }
  return h;
}

static inline uint64_t jsynth_stream(uint64_t seed, const char* name) {
  return jsynth_splitmix_at(seed ^ jsynth_fnv1a64(name), 0);
}

static inline double jsynth_uniform01(uint64_t stream, uint64_t ctr) {
  return (double)(jsynth_splitmix_at(stream, ctr) >> 11) * (1.0 / 9007199254740992.0);
}

/* ln(x) for x > 0 finite: x = m * 2^e with m in [sqrt(1/2), sqrt(2)),
 * ln m = 2 (z + z^3/3 + z^5/5 + ...), z = (m-1)/(m+1), |z| <= 0.1716. */
static inline double jsynth_ln(double x) {
  int e = 0;
  double m = frexp(x, &e); /* m in [0.5, 1) exactly */
  if (m < 0.70710678118654752440) { m *= 2.0; e -= 1; }
  double z = (m - 1.0) / (m + 1.0);
  double z2 = z * z;
  double term = z, sum = 0.0;
  for (int k = 1; k <= 41; k += 2) { sum += term / (double)k; term *= z2; }
  return 2.0 * sum + (double)e * 0.69314718055994530942;
}

/* sin and cos of r for |r| <= pi/4 by Taylor series to degree 25. */
static inline double jsynth_sin_small(double r) {
  double r2 = r * r, term = r, sum = 0.0;
  for (int k = 1; k <= 25; k += 2) { sum += term; term *= -r2 / (double)((k + 1) * (k + 2)); }
  return sum;
}
static inline double jsynth_cos_small(double r) {
  double r2 = r * r, term = 1.0, sum = 0.0;
  for (int k = 0; k <= 24; k += 2) { sum += term; term *= -r2 / (double)((k + 1) * (k + 2)); }
  return sum;
}

/* cos(2 pi v) for v in [0, 1): quadrant q = nearest multiple of 1/4,
 * remainder r = v - q/4 (exact), angle a = 2 pi r in [-pi/4, pi/4]. */
static inline double jsynth_cos2pi(double v) {
  double q = floor(4.0 * v + 0.5);
  double r = v - 0.25 * q;
  double a = 6.28318530717958647692 * r;
  int qi = ((int)q) & 3;
  switch (qi) {
    case 0: return jsynth_cos_small(a);
    case 1: return -jsynth_sin_small(a);
    case 2: return -jsynth_cos_small(a);
    default: return jsynth_sin_small(a);
  }
}

/* Standard normal element i of a stream. */
static inline double jsynth_normal(uint64_t stream, uint64_t i) {
  double u1 = jsynth_uniform01(stream, 2 * i);
  double u2 = jsynth_uniform01(stream, 2 * i + 1);
  return sqrt(-2.0 * jsynth_ln(1.0 - u1)) * jsynth_cos2pi(u2);
}

/* float -> bfloat16 bits, round to nearest even (NaN kept quiet). */
static inline uint16_t jsynth_f32_to_bf16_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}
static inline float jsynth_bf16_bits_to_f32(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}
static inline float jsynth_round_bf16(float f) {
  return jsynth_bf16_bits_to_f32(jsynth_f32_to_bf16_bits(f));
}

/* Distribution kinds of a synthetic tensor. */
enum {
  JSYNTH_NORMAL = 0,  /* a + b * N(0,1) */
  JSYNTH_UNIFORM = 1  /* a + (b - a) * U[0,1) */
};

/* Fill dst[0..n) with elements [first, first+n) of tensor `name`.
 * round_bf16 != 0 rounds every value to the nearest bfloat16 (kept as float). */
static inline void jsynth_fill(uint64_t seed, const char* name, int kind, double a, double b,
                               int round_bf16, uint64_t first, size_t n, float* dst) {
  uint64_t s = jsynth_stream(seed, name);
  for (size_t j = 0; j < n; ++j) {
    uint64_t i = first + (uint64_t)j;
    double v = (kind == JSYNTH_NORMAL) ? a + b * jsynth_normal(s, i)
                                       : a + (b - a) * jsynth_uniform01(s, i);
    float f = (float)v;
    dst[j] = round_bf16 ? jsynth_round_bf16(f) : f;
  }
}

/* ---- The init recipe of the synthetic encoder (one place, used by both sides) ----
 * matrix weights            N(0, 0.02)      (bf16-rounded in the bf16 mode)
 * biases                    0.01 * N(0,1)
 * LayerNorm gamma           1 + 0.1 * N(0,1)
 * LayerNorm beta            0.01 * N(0,1)
 * cls / pos / modality      N(0, 0.02)
 * pixels                    U(-2, 2), stream "input.pixels" of seed + 1
 * jsynth_param_init() maps a GGUF tensor name (enc.*, pred.*, head.*) to its (kind, a, b, is_matrix):
 * LayerNorm gains (ln1 / ln2 / *norm / ln_kv weights) 1 + 0.1 N(0,1), biases 0.01 N(0,1), other
 * weights (matrices) N(0, 0.02), everything else (tokens, tables, vectors) N(0, 0.02). */
static inline int jsynth_ends_with(const char* s, const char* suffix) {
  size_t ls = strlen(s), lf = strlen(suffix);
  return ls >= lf && memcmp(s + ls - lf, suffix, lf) == 0;
}

static inline void jsynth_param_init(const char* name, int* kind, double* a, double* b, int* is_matrix) {
  *kind = JSYNTH_NORMAL;
  *is_matrix = 0;
  if (jsynth_ends_with(name, "ln1.weight") || jsynth_ends_with(name, "ln2.weight") ||
      jsynth_ends_with(name, "norm.weight") || jsynth_ends_with(name, "ln_kv.weight")) {
    *a = 1.0; *b = 0.1;
  } else if (jsynth_ends_with(name, ".bias")) {
    *a = 0.0; *b = 0.01;
  } else if (jsynth_ends_with(name, ".weight")) {
    *a = 0.0; *b = 0.02; *is_matrix = 1;
  } else { /* enc.cls_token, enc.pos_embed, enc.mod_embed_video, ... */
    *a = 0.0; *b = 0.02;
  }
}

/* Fill a whole enc.* parameter tensor of n elements following the recipe. */
static inline void jsynth_param(uint64_t seed, const char* name, int bf16_matrices, size_t n, float* dst) {
  int kind, is_matrix;
  double a, b;
  jsynth_param_init(name, &kind, &a, &b, &is_matrix);
  jsynth_fill(seed, name, kind, a, b, bf16_matrices && is_matrix, 0, n, dst);
}

/* Pixels of a clip batch: U(-2, 2), n = B*T*C*H*W values in the caller's layout order. */
static inline void jsynth_pixels(uint64_t seed, uint64_t first, size_t n, float* dst) {
  jsynth_fill(seed + 1ULL, "input.pixels", JSYNTH_UNIFORM, -2.0, 2.0, 0, first, n, dst);
}

#ifdef __cplusplus
}
#endif
#endif /* JEPA_SYNTH_H */
