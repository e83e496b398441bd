/*
 * oracle.c -- plain, slow, obviously correct CPU implementation of the packed ternary-weight
 * decode path. TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
 * baseline leg use it to produce expected values; the library's product path never calls,
 * links or loads it, and it shares no code, header, table or constant with the CUDA path.
 *
 * What it computes, and the passages it follows ("The Neutrino Engine", Fermion Research):
 *   - each projection weight is ternary {-1, 0, +1} and each row has a scale (§ "The file is
 *     not the traffic"); at batch one a weight feeds one multiply-accumulate per token
 *     (§ "A 104 microsecond floor inside a 694 microsecond step"), so a projection is the
 *     matrix-vector product of the trits with the activation, scaled per row;
 *   - the output table is int8 and every row is scored (§ "The file is not the traffic");
 *     the emitted token is the arg-max (greedy decoding, § "One changed token fails the
 *     release").
 * The pages fix neither the bit format, nor the activation quantizer, nor the epilogue's
 * rounding order, nor the tie rule. The readings taken here:
 *   - trit k of row n is the 2-bit field at bit 2*(k%16) of word n*(K/16) + k/16; field
 *     codes 00 = 0, 01 = +1, 11 = -1, and 10 is rejected;
 *   - quantize: m = max|x|; m == 0 gives scale 0 and all-zero codes; otherwise the scale is
 *     the fp32 quotient m / 127 and each code is rint(x / scale) (fp32 quotient, ties to
 *     even), clamped to [-127, 127];
 *   - projection output: the exact integer sum, converted to fp32 (round to nearest), times
 *     the row scale (fp32, rounded), times the activation scale (fp32, rounded); no fused
 *     multiply-add (built with -ffp-contract=off);
 *   - arg-max: the lowest index among the maximal scores, +0 and -0 being equal.
 * Integer sums are accumulated in int64 and checked against the int32 range. The fp32
 * rounding sequence is the one the kernels are specified to use, because the arg-max and the
 * int8 codes are decisions taken on fp32 values; orc_gemm also reports a double-precision
 * version of each output for the tests that bound the fp32 rounding.
 *
 * The tiled layout (orc_repack_tiled / orc_unpack_tiled) is this library's own load-time
 * arrangement; its definition is the one written in the library's public header, restated
 * here from that text.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int orc_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads the parallel loops use from now on (for timing the oracle at one thread and at all
 * of them; no result depends on it). n <= 0 selects every core. */
void orc_set_threads(int n) {
#ifdef _OPENMP
  omp_set_num_threads(n > 0 ? n : omp_get_num_procs());
#else
  (void)n;
#endif
}

/* Value of one plain field code; 2 (the invalid code) is reported through *bad. */
static int plain_trit(uint32_t code, int* bad) {
  switch (code & 3u) {
    case 0u: return 0;
    case 1u: return 1;
    case 3u: return -1;
    default: *bad = 1; return 0;
  }
}

/* Trit k of row n of a plain matrix. */
static int trit_at(const uint32_t* w, int K, int n, int k, int* bad) {
  uint32_t word = w[(int64_t)n * (K / 16) + k / 16];
  return plain_trit(word >> (2 * (k % 16)), bad);
}

/* Number of invalid (10) fields in n_words plain words. */
int64_t orc_count_invalid(const uint32_t* w, int64_t n_words) {
  int64_t bad = 0;
  for (int64_t i = 0; i < n_words; ++i)
    for (int j = 0; j < 16; ++j)
      if (((w[i] >> (2 * j)) & 3u) == 2u) ++bad;
  return bad;
}

/* Dense trits t[N][K] of a plain matrix. Returns -1 if an invalid field is present. */
int orc_unpack_plain(const uint32_t* w, int N, int K, int8_t* t) {
  int bad = 0;
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k) t[(int64_t)n * K + k] = (int8_t)trit_at(w, K, n, k, &bad);
  return bad ? -1 : 0;
}

/* Activation quantization of B vectors of length K. */
void orc_quantize(const float* x, int B, int K, int8_t* q, float* s) {
  for (int b = 0; b < B; ++b) {
    const float* xb = x + (int64_t)b * K;
    int8_t* qb = q + (int64_t)b * K;
    float m = 0.0f;
    for (int k = 0; k < K; ++k) {
      float a = fabsf(xb[k]);
      if (a > m) m = a;
    }
    if (m == 0.0f) {
      s[b] = 0.0f;
      for (int k = 0; k < K; ++k) qb[k] = 0;
      continue;
    }
    float sc = m / 127.0f;
    s[b] = sc;
    for (int k = 0; k < K; ++k) {
      float r = rintf(xb[k] / sc);
      if (r > 127.0f) r = 127.0f;
      if (r < -127.0f) r = -127.0f;
      qb[k] = (int8_t)r;
    }
  }
}

/* Ternary projection of B activation vectors:
 *   acc[b][n] = sum_k t[n][k] * q[b][k]
 *   y[b][n]   = fp32(fp32(float(acc) * s_w[n]) * s_x[b])
 *   y64[b][n] = acc * s_w[n] * s_x[b] in double (NULL to skip)
 * Returns 0, -1 on an invalid field, -2 if a sum leaves the int32 range. */
int orc_gemm(const uint32_t* w, const float* s_w, int N, int K, const int8_t* q,
             const float* s_x, int B, int32_t* acc, float* y, double* y64) {
  int status = 0;
  for (int b = 0; b < B; ++b) {
    const int8_t* qb = q + (int64_t)b * K;
#pragma omp parallel for schedule(static) reduction(min : status)
    for (int n = 0; n < N; ++n) {
      int bad = 0;
      int64_t a = 0;
      for (int k = 0; k < K; ++k) a += (int64_t)trit_at(w, K, n, k, &bad) * qb[k];
      if (bad && status > -1) status = -1;
      if (a > INT32_MAX || a < INT32_MIN) status = -2;
      int64_t o = (int64_t)b * N + n;
      acc[o] = (int32_t)a;
      float f = (float)(int32_t)a;
      f = f * s_w[n];
      f = f * s_x[b];
      y[o] = f;
      if (y64) y64[o] = (double)a * (double)s_w[n] * (double)s_x[b];
    }
  }
  return status;
}

/* int8 output projection with greedy arg-max:
 *   acc[b][v] = sum_k T[v][k] * q[b][k];   logit = fp32(fp32(float(acc) * s_T[v]) * s_x[b])
 *   argmax[b] = lowest v with the largest logit.
 * acc and logits are [B][V] (acc may be NULL). Returns 0, or -2 if a sum leaves int32. */
int orc_logits_argmax(const int8_t* T, const float* s_T, int V, int K, const int8_t* q,
                      const float* s_x, int B, int32_t* acc, float* logits, int32_t* argmax) {
  int status = 0;
  for (int b = 0; b < B; ++b) {
    const int8_t* qb = q + (int64_t)b * K;
    float* lb = logits + (int64_t)b * V;
#pragma omp parallel for schedule(static) reduction(min : status)
    for (int v = 0; v < V; ++v) {
      const int8_t* row = T + (int64_t)v * K;
      int64_t a = 0;
      for (int k = 0; k < K; ++k) a += (int64_t)row[k] * qb[k];
      if (a > INT32_MAX || a < INT32_MIN) status = -2;
      if (acc) acc[(int64_t)b * V + v] = (int32_t)a;
      float f = (float)(int32_t)a;
      f = f * s_T[v];
      f = f * s_x[b];
      lb[v] = f;
    }
    int best = 0;
    for (int v = 1; v < V; ++v)
      if (lb[v] > lb[best]) best = v;
    argmax[b] = best;
  }
  return status;
}

/* ---- tiled layout (the library header's definition) ------------------------------------
 * Np = roundup(N, 4), Kp = roundup(K, 512); tile t = rows 4t..4t+3; tile bytes = 4 * Kp / 4
 * = Kp; inside tile t, group j (16 bytes) holds 4 words, word r for row 4t+r, trits
 * 16j..16j+15. Nibble i < 4 codes (trit 16j+i, trit 16j+4+i), nibble 4+i codes
 * (trit 16j+8+i, trit 16j+12+i). Pair codes: */
static int pair_code(int a, int b) {
  if (a == 0 && b == 0) return 0;
  if (a == 1 && b == 0) return 1;
  if (a == -1 && b == 0) return 2;
  if (a == 0 && b == 1) return 3;
  if (a == 1 && b == 1) return 4;
  if (a == -1 && b == 1) return 5;
  if (a == 1 && b == -1) return 6;
  if (a == -1 && b == -1) return 7;
  return 14; /* (0, -1) */
}

static void pair_of(int code, int* a, int* b) {
  static const int ta[16] = {0, 1, -1, 0, 1, -1, 1, -1, 99, 99, 99, 99, 99, 99, 0, 99};
  static const int tb[16] = {0, 0, 0, 1, 1, 1, -1, -1, 99, 99, 99, 99, 99, 99, -1, 99};
  *a = ta[code & 15];
  *b = tb[code & 15];
}

int64_t orc_tiled_bytes(int N, int K) {
  int64_t Np = ((int64_t)N + 3) / 4 * 4, Kp = ((int64_t)K + 511) / 512 * 512;
  return Np * Kp / 4;
}

/* Trit (n, k) of the plain matrix, 0 outside [0,N) x [0,K); invalid fields read as 0. */
static int trit_or_zero(const uint32_t* w, int N, int K, int64_t n, int64_t k) {
  int bad = 0;
  if (n >= N || k >= K) return 0;
  return trit_at(w, K, (int)n, (int)k, &bad);
}

void orc_repack_tiled(const uint32_t* w, int N, int K, uint8_t* out) {
  const int64_t Np = ((int64_t)N + 3) / 4 * 4, Kp = ((int64_t)K + 511) / 512 * 512;
  const int64_t groups = Kp / 16;
  for (int64_t t = 0; t < Np / 4; ++t)
    for (int64_t j = 0; j < groups; ++j)
      for (int r = 0; r < 4; ++r) {
        const int64_t n = 4 * t + r, k0 = 16 * j;
        uint32_t word = 0;
        for (int i = 0; i < 4; ++i) {
          int lo = pair_code(trit_or_zero(w, N, K, n, k0 + i), trit_or_zero(w, N, K, n, k0 + 4 + i));
          int hi = pair_code(trit_or_zero(w, N, K, n, k0 + 8 + i), trit_or_zero(w, N, K, n, k0 + 12 + i));
          word |= (uint32_t)lo << (4 * i);
          word |= (uint32_t)hi << (4 * (4 + i));
        }
        uint8_t* dst = out + t * Kp + j * 16 + 4 * r;
        memcpy(dst, &word, 4); /* little-endian byte order, as on the GPU */
      }
}

/* Dense trits [N][K] read back from a tiled buffer. Returns -1 on an unused pair code. */
int orc_unpack_tiled(const uint8_t* tiled, int N, int K, int8_t* t) {
  const int64_t Kp = ((int64_t)K + 511) / 512 * 512;
  int status = 0;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k) {
      const int64_t tile = n / 4, r = n % 4, j = k / 16, e = k % 16;
      uint32_t word;
      memcpy(&word, tiled + tile * Kp + j * 16 + 4 * r, 4);
      /* e in [0,4): nibble e, first of pair; [4,8): nibble e-4, second; [8,12): nibble e-4,
       * first; [12,16): nibble e-8, second. */
      int nib = e < 4 ? (int)e : e < 8 ? (int)e - 4 : e < 12 ? (int)e - 4 : (int)e - 8;
      int second = (e >= 4 && e < 8) || e >= 12;
      int a, b;
      pair_of((int)(word >> (4 * nib)) & 15, &a, &b);
      int v = second ? b : a;
      if (v == 99) { status = -1; v = 0; }
      t[n * K + k] = (int8_t)v;
    }
  return status;
}

/* ---- input-table row gather ("The file is not the traffic": of the input table only the
 * rows of the current tokens are read) ----------------------------------------------------
 * x[b][k] = fp32((float)T[tok[b]][k] * s[tok[b]]) -- the int8 value is exact in fp32, one
 * rounded product. A token outside [0, V) gives a row of zeros and is counted. */
int orc_embed_rows(const int8_t* T, const float* s, int V, int K, const int32_t* tok, int B, float* x) {
  int bad = 0;
  for (int b = 0; b < B; ++b) {
    const int t = tok[b];
    for (int k = 0; k < K; ++k) {
      float v = 0.0f;
      if (t >= 0 && t < V) v = (float)T[(int64_t)t * K + k] * s[t];
      x[(int64_t)b * K + k] = v;
    }
    if (t < 0 || t >= V) ++bad;
  }
  return bad;
}

/* ---- verify-pass acceptance ("The 0.6B model does not get to decide": the large model
 * scores every drafted position in one pass, the longest prefix where the draft agrees with
 * it is kept, and at the first disagreement the large model's own token is emitted) -------
 * Positions 0..B-1 of the verify pass hold the last emitted token followed by the B-1
 * drafted tokens draft[0..B-2]; argmax[i] is the large model's greedy token after position i.
 * Draft token i is accepted when it equals argmax[i] and every earlier draft was accepted.
 * With j accepted drafts the emitted tokens are draft[0..j-1] then argmax[j]; returns j + 1. */
int orc_verify_accept(const int32_t* draft, const int32_t* argmax, int B, int32_t* emit) {
  int j = 0;
  while (j < B - 1 && draft[j] == argmax[j]) {
    emit[j] = draft[j];
    ++j;
  }
  emit[j] = argmax[j];
  return j + 1;
}
