/*
 * synth.c -- seeded synthetic inputs for the W4A8 / W4A16 / W8A16 linears.
 *
 * Test and benchmark infrastructure shared by the CPU oracle and the CUDA
 * path. It holds none of the method's arithmetic: it only draws codes, zero
 * points, scales and activations. Every stream is counter based, so element i
 * of a tensor depends only on (seed, i) and any slice can be regenerated.
 *
 *   uniform64(seed, i) = splitmix64_mix(seed + (i + 1) * 0x9E3779B97F4A7C15)
 *
 * splitmix64 is the published generator of Steele, Lea and Flood ("Fast
 * splittable pseudorandom number generators", OOPSLA 2014); the mix below is
 * its output function. Normals use the Box-Muller transform (Box and Muller,
 * 1958) on the uniforms at counters 2i and 2i+1, keeping the cosine branch.
 *
 * Distributions (weights are int4 group-wise asymmetric with group 128, the
 * form the "EgoPQ Real-Serving Handoff" page calls _gptq_scale/_gptq_zero and
 * "The 4-bit CPU path" page, section "Building a checkpoint", packs with
 * --group-size 128):
 *   codes, zeros  uniform integers in [0, 15] (top four bits of a draw)
 *   scales        fp16_rn(|N(0, sigma)| / div + add)
 *   activations   bf16_rn(N(0, 1) * (mult if the channel is an outlier))
 *   int8 weights  uniform integers in [-127, 127]
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

uint64_t synth_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t draw(uint64_t seed, uint64_t i) {
  return synth_mix(seed + (i + 1) * GOLDEN);
}

/* Per-tensor seed: config, layer, linear index and tensor id folded into one
 * word, then mixed once. */
uint64_t synth_tensor_seed(int64_t config, int64_t layer, int64_t linear,
                           int64_t tensor_id) {
  uint64_t w = 0xE90B0000ULL ^ ((uint64_t)config << 24) ^
               ((uint64_t)layer << 16) ^ ((uint64_t)linear << 8) ^
               (uint64_t)tensor_id;
  return synth_mix(w);
}

/* uniform in (0, 1]: 53 random bits, shifted by one ulp so log() is finite */
static inline double u01_open0(uint64_t x) {
  return (double)((x >> 11) + 1) * (1.0 / 9007199254740992.0);
}
/* uniform in [0, 1) */
static inline double u01(uint64_t x) {
  return (double)(x >> 11) * (1.0 / 9007199254740992.0);
}

static inline double normal_at(uint64_t seed, uint64_t i) {
  double u1 = u01_open0(draw(seed, 2 * i));
  double u2 = u01(draw(seed, 2 * i + 1));
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

/* Round a double to the nearest value of a binary format with `mant` stored
 * fraction bits and minimum normal exponent `emin`, ties to even, returning the
 * rounded value as a double. Used only to shape generated inputs. */
static double round_to_format(double x, int mant, int emin) {
  if (x == 0.0 || !isfinite(x)) return x;
  int e;
  frexp(fabs(x), &e); /* |x| = f * 2^e, f in [0.5, 1) */
  int E = e - 1;      /* |x| in [2^E, 2^(E+1)) */
  if (E < emin) E = emin;
  double q = ldexp(1.0, E - mant);
  return nearbyint(x / q) * q;
}

static uint16_t to_fp16_bits(double x) {
  double r = round_to_format(x, 10, -14);
  uint16_t sign = (r < 0 || (r == 0 && signbit(r))) ? 0x8000 : 0;
  double a = fabs(r);
  if (a >= 65520.0) return sign | 0x7C00;
  if (a == 0.0) return sign;
  int e;
  double f = frexp(a, &e); /* a = f*2^e */
  int E = e - 1;
  if (E < -14) { /* subnormal: a = m * 2^-24 */
    return sign | (uint16_t)llround(ldexp(a, 24));
  }
  uint16_t m = (uint16_t)llround((ldexp(f, 1) - 1.0) * 1024.0);
  return sign | (uint16_t)((E + 15) << 10) | m;
}

static uint16_t to_bf16_bits(double x) {
  double r = round_to_format(x, 7, -126);
  float f = (float)r; /* exact: r has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

void synth_u4(uint64_t seed, int64_t n, uint8_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)(draw(seed, (uint64_t)i) >> 60);
}

void synth_i8_sym(uint64_t seed, int64_t n, int8_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    double u = u01(draw(seed, (uint64_t)i));
    out[i] = (int8_t)((int)floor(u * 255.0) - 127);
  }
}

void synth_normal(uint64_t seed, int64_t n, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = normal_at(seed, (uint64_t)i);
}

void synth_scales_f16(uint64_t seed, int64_t n, double sigma, double div,
                      double add, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i)
    out[i] = to_fp16_bits(fabs(sigma * normal_at(seed, (uint64_t)i)) / div + add);
}

/* Number of outlier channels: round-half-even(frac * K). */
int64_t synth_outlier_count(int64_t K, double frac) {
  return (int64_t)nearbyint(frac * (double)K);
}

/* Outlier channels for a K-wide activation: a partial Fisher-Yates shuffle of
 * 0..K-1 driven by its own stream (seed ^ 0x5A5A...), first `count` entries. */
void synth_outlier_channels(uint64_t seed, int64_t K, int64_t count, int64_t* out) {
  int64_t* perm = (int64_t*)malloc(sizeof(int64_t) * (size_t)K);
  for (int64_t i = 0; i < K; ++i) perm[i] = i;
  uint64_t s2 = seed ^ 0x5A5A5A5A5A5A5A5AULL;
  for (int64_t i = 0; i < count; ++i) {
    uint64_t r = draw(s2, (uint64_t)i);
    int64_t j = i + (int64_t)(r % (uint64_t)(K - i));
    int64_t t = perm[i]; perm[i] = perm[j]; perm[j] = t;
  }
  for (int64_t i = 0; i < count; ++i) out[i] = perm[i];
  free(perm);
}

/* Activations x[M][K] as bf16 bits: N(0,1), multiplied by `mult` on the
 * outlier channels (shared by every token of the tensor). */
void synth_act_bf16(uint64_t seed, int64_t M, int64_t K, double frac, double mult,
                    uint16_t* out) {
  int64_t count = synth_outlier_count(K, frac);
  unsigned char* is_out = (unsigned char*)calloc((size_t)K, 1);
  if (count > 0) {
    int64_t* ch = (int64_t*)malloc(sizeof(int64_t) * (size_t)count);
    synth_outlier_channels(seed, K, count, ch);
    for (int64_t i = 0; i < count; ++i) is_out[ch[i]] = 1;
    free(ch);
  }
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m)
    for (int64_t k = 0; k < K; ++k) {
      int64_t i = m * K + k;
      double v = normal_at(seed, (uint64_t)i);
      if (is_out[k]) v *= mult;
      out[i] = to_bf16_bits(v);
    }
  free(is_out);
}
