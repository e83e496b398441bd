/*
 * synth.c -- seeded synthetic inputs shared by the tests, the benchmark and the oracle
 * checks. This file draws random numbers and writes them in the exchange formats (plain
 * packed trits, fp32 vectors, int8 tables); it computes nothing of the decode method.
 *
 * Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014) used counter-style: draw i of a stream with key k is
 * mix(k + (i + 1) * 0x9E3779B97F4A7C15), where mix is the SplitMix64 finaliser. Every
 * element therefore depends only on (seed, tag, index), so the OpenMP loops below give the
 * same bytes for any thread count, on any host.
 *
 * Distributions (the workloads' stated shapes and value mixes):
 *   trit:   v = draw >> 40 (24 bits); v < 5033165 -> -1, v < 10066330 -> +1, else 0
 *           (P(-1) = P(+1) = 0.3, P(0) = 0.4 to within 2^-24).
 *   unit:   u = (draw >> 11) * 2^-53 in [0, 1).
 *   scale:  fp32((0.5 + u) / denom), computed in double.
 *   normal: Box-Muller, z = sqrt(-2 ln u1) * cos(2 pi u2), u1 = ((d1 >> 11) + 1) * 2^-53,
 *           u2 = (d2 >> 11) * 2^-53, draws 2i and 2i+1; rounded to fp32.
 *   int8:   ((draw >> 32) * 255) >> 32, minus 127: integers in [-127, 127].
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* Key of the stream named by (seed, tag). */
uint64_t synth_key(uint64_t seed, uint64_t tag) { return mix64(mix64(seed) ^ mix64(tag + GOLDEN)); }

static inline uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GOLDEN); }

static inline int trit_of(uint64_t d) {
  uint64_t v = d >> 40;
  if (v < 5033165ULL) return -1;
  if (v < 10066330ULL) return 1;
  return 0;
}

/* Raw draws, for the generator's own tests. */
void synth_draws(uint64_t seed, uint64_t tag, uint64_t first, int64_t n, uint64_t* out) {
  uint64_t key = synth_key(seed, tag);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = draw(key, first + (uint64_t)i);
}

/* Ternary matrix N x K (K % 16 == 0) in the plain exchange layout: uint32 w[N][K/16], trit k
 * in the 2-bit field at bit 2*(k%16) of word k/16, codes 00 = 0, 01 = +1, 11 = -1. Trit
 * (n, k) is draw n*K + k. */
void synth_ternary_plain(uint64_t seed, uint64_t tag, int N, int K, uint32_t* w) {
  uint64_t key = synth_key(seed, tag);
  const int64_t words = (int64_t)N * (K / 16);
#pragma omp parallel for schedule(static)
  for (int64_t wi = 0; wi < words; ++wi) {
    const uint64_t base = (uint64_t)wi * 16;
    uint32_t word = 0;
    for (int j = 0; j < 16; ++j) {
      int t = trit_of(draw(key, base + (uint64_t)j));
      uint32_t code = t == 0 ? 0u : (t > 0 ? 1u : 3u);
      word |= code << (2 * j);
    }
    w[wi] = word;
  }
}

/* The same draws as synth_ternary_plain, as one int8 value per trit: t[N][K]. */
void synth_ternary_dense(uint64_t seed, uint64_t tag, int N, int K, int8_t* t) {
  uint64_t key = synth_key(seed, tag);
  const int64_t n = (int64_t)N * K;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) t[i] = (int8_t)trit_of(draw(key, (uint64_t)i));
}

/* fp32 scales (0.5 + u) / denom, one per element. */
void synth_scales(uint64_t seed, uint64_t tag, int64_t n, double denom, float* s) {
  uint64_t key = synth_key(seed, tag);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    double u = (double)(draw(key, (uint64_t)i) >> 11) * 0x1.0p-53;
    s[i] = (float)((0.5 + u) / denom);
  }
}

/* fp32 standard normal values (Box-Muller, cosine branch). */
void synth_normal(uint64_t seed, uint64_t tag, int64_t n, float* x) {
  uint64_t key = synth_key(seed, tag);
  const double two_pi = 6.283185307179586476925286766559;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    double u1 = (double)((draw(key, 2 * (uint64_t)i) >> 11) + 1) * 0x1.0p-53;
    double u2 = (double)(draw(key, 2 * (uint64_t)i + 1) >> 11) * 0x1.0p-53;
    x[i] = (float)(sqrt(-2.0 * log(u1)) * cos(two_pi * u2));
  }
}

/* int8 integers uniform in [-127, 127]. */
void synth_int8(uint64_t seed, uint64_t tag, int64_t n, int8_t* t) {
  uint64_t key = synth_key(seed, tag);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    uint64_t hi = draw(key, (uint64_t)i) >> 32;
    t[i] = (int8_t)((int)((hi * 255ULL) >> 32) - 127);
  }
}
