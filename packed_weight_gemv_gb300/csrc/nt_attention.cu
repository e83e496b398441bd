// nt_attention.cu -- the attention side of a decoder layer: grouped-query attention of the
// new positions over a bf16 key-value cache, the rotary embedding with the cache append, and
// RMS normalisation ("The Neutrino Engine", § "At 26K tokens, the cache becomes larger than
// the model": 8 key-value heads of 128 dimensions, 16-bit cache entries, grouped-query
// attention).
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>

#include "nt_kernels.cuh"

namespace nt {
namespace {

constexpr int kAttnD = 128;        // dimensions per head
constexpr int kAttnSub = 64;       // cache positions per step of a work unit
constexpr int kAttnThreads = 128;  // 4 warps
constexpr int kAttnMaxSplit = 512;
constexpr int kPartRow = kAttnD + 4;  // floats per partial result: weighted sum, max, sum, padding

struct AttnArgs {
  const float* q;      // [B][Hq][D]
  const uint16_t* kc;  // [Hkv][ts][D] bf16
  const uint16_t* vc;
  float* part;         // [B][Hq][nch][kPartRow]: weighted value sum, max score (log2 units), sum
  unsigned int* done;  // [B][Hkv]: units finished; the last CTA of a group merges and resets it
  float* out;          // [B][Hq][D]
  int B, Hq, Hkv, T, ts, nch, span;  // span: positions per unit (a multiple of kAttnSub)
  float scale_log2;    // log2(e) / sqrt(D)
  const int* T_dev;    // when set, the cache length is *T_dev (T then only sized the grid)
};

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <int G>
__device__ __forceinline__ void block_reduce_max(float (&v)[G], float (*red)[4], int lane, int w) {
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float x = v[g];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    if (lane == 0) red[g][w] = x;
  }
  __syncthreads();
#pragma unroll
  for (int g = 0; g < G; ++g) v[g] = fmaxf(fmaxf(red[g][0], red[g][1]), fmaxf(red[g][2], red[g][3]));
}

// One CTA per (unit of `span` cache positions, key-value head), walking the unit in steps of
// 64 positions with an online softmax. Each step first issues all of its loads (keys: thread
// (position i/2, half i%2) takes 64 dimensions of one position; values: thread (dimension pair
// i%64, half i/64) takes 2 dimensions of 32 positions), then forms the scores (one shuffle
// joins the halves), the step's maximum, the probabilities and the rescaled weighted sums.
// Every new position b and every query head of the group uses the same keys and values. The
// unit's (weighted sum, max, sum) go to the workspace; the last CTA of each (b, key-value head)
// merges all units into out and resets the counter.
template <int G>
__global__ void __launch_bounds__(kAttnThreads) attn_unit_kernel(const AttnArgs a) {
  __shared__ __align__(16) float Qs[G][kAttnD];
  __shared__ __align__(16) float P[G][kAttnSub];
  __shared__ __align__(16) float Acc[4][G][kAttnD];
  __shared__ float red[G][4];
  __shared__ float Wm[G][kAttnMaxSplit];
  __shared__ int s_last;
  const int c = blockIdx.x, h = blockIdx.y, i = threadIdx.x, lane = i & 31, w = i >> 5;
  const int T = a.T_dev ? *a.T_dev : a.T;
  const int u0 = c * a.span, u1 = min(T, u0 + a.span);
  const uint16_t* kh = a.kc + (int64_t)h * a.ts * kAttnD;
  const uint32_t* vh = reinterpret_cast<const uint32_t*>(a.vc + (int64_t)h * a.ts * kAttnD);
  const int64_t head_stride = (int64_t)a.nch * kPartRow;
  const int kp = i >> 1, kh2 = i & 1;     // key role: position kp of the step, dims 64*kh2 ..
  const int dp = i & 63, vh2 = i >> 6;    // value role: dims 2dp, 2dp+1, positions 32*vh2 ..

  for (int b = 0; b < a.B; ++b) {
    const int vis = min(u1, T - a.B + b + 1);  // positions [u0, vis) are visible to b
    const float* qg = a.q + ((int64_t)b * a.Hq + h * G) * kAttnD;
    for (int e = i; e < G * kAttnD; e += kAttnThreads) Qs[e / kAttnD][e % kAttnD] = __fmul_rn(qg[e], a.scale_log2);
    float mrun[G], lrun[G], acc[G][2];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      mrun[g] = -INFINITY;
      lrun[g] = 0.0f;
      acc[g][0] = acc[g][1] = 0.0f;
    }
    __syncthreads();
    for (int p0 = u0; p0 < vis; p0 += kAttnSub) {
      const int nv = min(kAttnSub, vis - p0);
      // loads first
      uint4 kw[8];
      const bool kval = kp < nv;
      const uint4* kr = reinterpret_cast<const uint4*>(kh + (int64_t)(p0 + kp) * kAttnD + 64 * kh2);
#pragma unroll
      for (int u = 0; u < 8; ++u) kw[u] = kval ? __ldg(kr + u) : make_uint4(0u, 0u, 0u, 0u);
      uint32_t vw[32];
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        const int pt = 32 * vh2 + t;
        vw[t] = pt < nv ? __ldg(vh + (int64_t)(p0 + pt) * (kAttnD / 2) + dp) : 0u;
      }
      // scores
      float s[G];
#pragma unroll
      for (int g = 0; g < G; ++g) s[g] = 0.0f;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float k0 = bf_lo(kw[u].x), k1 = bf_hi(kw[u].x), k2 = bf_lo(kw[u].y), k3 = bf_hi(kw[u].y);
        const float k4 = bf_lo(kw[u].z), k5 = bf_hi(kw[u].z), k6 = bf_lo(kw[u].w), k7 = bf_hi(kw[u].w);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float4 qa = *reinterpret_cast<const float4*>(&Qs[g][64 * kh2 + 8 * u]);
          const float4 qb = *reinterpret_cast<const float4*>(&Qs[g][64 * kh2 + 8 * u + 4]);
          s[g] = fmaf(qa.x, k0, s[g]);
          s[g] = fmaf(qa.y, k1, s[g]);
          s[g] = fmaf(qa.z, k2, s[g]);
          s[g] = fmaf(qa.w, k3, s[g]);
          s[g] = fmaf(qb.x, k4, s[g]);
          s[g] = fmaf(qb.y, k5, s[g]);
          s[g] = fmaf(qb.z, k6, s[g]);
          s[g] = fmaf(qb.w, k7, s[g]);
        }
      }
      float mstep[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        s[g] += __shfl_xor_sync(0xffffffffu, s[g], 1);
        if (!kval) s[g] = -INFINITY;
        mstep[g] = s[g];
      }
      block_reduce_max<G>(mstep, red, lane, w);
      float corr[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float mn = fmaxf(mrun[g], mstep[g]);
        corr[g] = exp2f(mrun[g] - mn);  // 0 on the first step (mrun = -inf)
        mrun[g] = mn;
        if (kh2 == 0) P[g][kp] = kval ? exp2f(s[g] - mn) : 0.0f;
      }
      __syncthreads();  // P complete; red[] free
      // weighted values, rescaled
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float l = 0.0f;
        if (i < kAttnSub) l = P[g][i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0 && w < 2) red[g][w] = l;
        acc[g][0] *= corr[g];
        acc[g][1] *= corr[g];
      }
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        const float v0 = bf_lo(vw[t]), v1 = bf_hi(vw[t]);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float p = P[g][32 * vh2 + t];
          acc[g][0] = fmaf(p, v0, acc[g][0]);
          acc[g][1] = fmaf(p, v1, acc[g][1]);
        }
      }
      __syncthreads();  // step sums in red[]; P may be overwritten
#pragma unroll
      for (int g = 0; g < G; ++g) lrun[g] = fmaf(lrun[g], corr[g], red[g][0] + red[g][1]);
      __syncthreads();  // red[] free for the next step
    }
    // the unit's result for position b
    float* pb = a.part + ((int64_t)(b * a.Hq + h * G) * a.nch + c) * kPartRow;
#pragma unroll
    for (int g = 0; g < G; ++g) *reinterpret_cast<float2*>(&Acc[vh2][g][2 * dp]) = make_float2(acc[g][0], acc[g][1]);
    __syncthreads();
#pragma unroll
    for (int g = 0; g < G; ++g) {
      pb[g * head_stride + i] = Acc[0][g][i] + Acc[1][g][i];
      if (i == 0) {
        pb[g * head_stride + kAttnD] = mrun[g];
        pb[g * head_stride + kAttnD + 1] = lrun[g];
      }
    }
    // the last unit of this (b, key-value head) merges: unit weights 2^(m_c - M), then sums
    __threadfence();
    __syncthreads();
    if (i == 0) s_last = atomicAdd(&a.done[b * a.Hkv + h], 1u) == (unsigned)(a.nch - 1);
    __syncthreads();
    if (s_last) {
      __threadfence();
      const float* pg0 = a.part + (int64_t)(b * a.Hq + h * G) * head_stride;
      float M[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        M[g] = -INFINITY;
        for (int cc = i; cc < a.nch; cc += kAttnThreads) M[g] = fmaxf(M[g], __ldcg(pg0 + g * head_stride + cc * kPartRow + kAttnD));
      }
      block_reduce_max<G>(M, red, lane, w);
      float L[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        L[g] = 0.0f;
        for (int cc = i; cc < a.nch; cc += kAttnThreads) {
          const float* pc = pg0 + g * head_stride + cc * kPartRow;
          const float mc = __ldcg(pc + kAttnD);
          const float wt = mc == -INFINITY ? 0.0f : exp2f(mc - M[g]);
          Wm[g][cc] = wt;
          L[g] = fmaf(__ldcg(pc + kAttnD + 1), wt, L[g]);
        }
      }
      __syncthreads();  // red[] (maxima) read by every thread; Wm complete
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float x = L[g];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        if (lane == 0) red[g][w] = x;
      }
      __syncthreads();
      // weighted sums: warp grp takes units grp, grp + 4, ..., lane the dimensions 4*lane ..
      {
        const int grp = w, d4 = 4 * lane;
        float4 O[G];
#pragma unroll
        for (int g = 0; g < G; ++g) O[g] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int cc = grp; cc < a.nch; cc += 4) {
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float4 x = __ldcg(reinterpret_cast<const float4*>(pg0 + g * head_stride + cc * kPartRow + d4));
            const float wt = Wm[g][cc];
            O[g].x = fmaf(x.x, wt, O[g].x);
            O[g].y = fmaf(x.y, wt, O[g].y);
            O[g].z = fmaf(x.z, wt, O[g].z);
            O[g].w = fmaf(x.w, wt, O[g].w);
          }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) *reinterpret_cast<float4*>(&Acc[grp][g][d4]) = O[g];
      }
      __syncthreads();
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float Lg = (red[g][0] + red[g][1]) + (red[g][2] + red[g][3]);
        const float O = (Acc[0][g][i] + Acc[1][g][i]) + (Acc[2][g][i] + Acc[3][g][i]);
        a.out[(int64_t)(b * a.Hq + h * G + g) * kAttnD + i] = __fdiv_rn(O, Lg);
      }
      if (i == 0) a.done[b * a.Hkv + h] = 0u;
    }
    __syncthreads();  // shared buffers are reused by the next position
  }
}

// Rotary embedding of position pos0 + blockIdx.x: the angles pos * base^(-2i/D) are formed
// and reduced in double precision (a float angle of a large position would carry an error of
// about pos * 2^-24 radians), the rotations in fp32 without contraction. Keys and values go
// to the cache rows pos0 + b as bf16 (round to nearest even); queries to q_out in fp32.
__global__ void rope_append_kernel(const float* __restrict__ q, const float* __restrict__ k,
                                   const float* __restrict__ v, int Hq, int Hkv, int pos0_arg, const int* pos_dev,
                                   double log2_base,
                                   float* __restrict__ q_out, uint16_t* __restrict__ kc, uint16_t* __restrict__ vc,
                                   int ts) {
  __shared__ float cs[kAttnD / 2], sn[kAttnD / 2];
  const int pos0 = pos_dev ? *pos_dev : pos0_arg;
  const int b = blockIdx.x, pos = pos0 + b;
  constexpr int half = kAttnD / 2;
  if (threadIdx.x < half) {
    const double ang = (double)pos * exp2(-2.0 * threadIdx.x / kAttnD * log2_base);
    cs[threadIdx.x] = (float)cos(ang);
    sn[threadIdx.x] = (float)sin(ang);
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < (Hq + Hkv) * half; idx += blockDim.x) {
    const int hh = idx / half, j = idx % half;
    const bool isq = hh < Hq;
    const float* x = isq ? q + ((int64_t)b * Hq + hh) * kAttnD : k + ((int64_t)b * Hkv + (hh - Hq)) * kAttnD;
    const float lo = x[j], hi = x[j + half];
    const float ylo = __fsub_rn(__fmul_rn(lo, cs[j]), __fmul_rn(hi, sn[j]));
    const float yhi = __fadd_rn(__fmul_rn(hi, cs[j]), __fmul_rn(lo, sn[j]));
    if (isq) {
      float* y = q_out + ((int64_t)b * Hq + hh) * kAttnD;
      y[j] = ylo;
      y[j + half] = yhi;
    } else {
      uint16_t* row = kc + ((int64_t)(hh - Hq) * ts + pos) * kAttnD;
      row[j] = __bfloat16_as_ushort(__float2bfloat16_rn(ylo));
      row[j + half] = __bfloat16_as_ushort(__float2bfloat16_rn(yhi));
    }
  }
  for (int idx = threadIdx.x; idx < Hkv * kAttnD; idx += blockDim.x) {
    const int hh = idx / kAttnD, d = idx % kAttnD;
    vc[((int64_t)hh * ts + pos) * kAttnD + d] =
        __bfloat16_as_ushort(__float2bfloat16_rn(v[((int64_t)b * Hkv + hh) * kAttnD + d]));
  }
}

// y = fl(fl(x * r) * gamma) with r = fl32(1 / sqrt(mean(x^2) + eps)) formed in double (the sum
// of squares of fp32 values in double precision is order-independent to ~2^-40 relative).
__global__ void __launch_bounds__(256) rmsnorm_kernel(const float* __restrict__ x, const float* __restrict__ gamma,
                                                      int D, float eps, float* __restrict__ y) {
  __shared__ double red[8];
  const float* xb = x + (int64_t)blockIdx.x * D;
  double s = 0.0;
  for (int d = threadIdx.x; d < D; d += 256) s += (double)xb[d] * (double)xb[d];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  double t = 0.0;
#pragma unroll
  for (int w = 0; w < 8; ++w) t += red[w];
  const float r = (float)(1.0 / sqrt(t / D + (double)eps));
  for (int d = threadIdx.x; d < D; d += 256)
    y[(int64_t)blockIdx.x * D + d] = __fmul_rn(__fmul_rn(xb[d], r), gamma[d]);
}

template <int G>
nt_status launch_attn_units(const AttnArgs& a, cudaStream_t st) {
  attn_unit_kernel<G><<<dim3(a.nch, a.Hkv), kAttnThreads, 0, st>>>(a);
  return check_launch("attn_unit_kernel");
}

// Positions per unit: about four units per SM over all key-value heads, whole 64-position
// steps, at most kAttnMaxSplit units per head.
int attn_span(int T, int Hkv) {
  const int sms = device_sm_count();
  const int want = std::max(1, (4 * sms + Hkv - 1) / Hkv);
  const int steps = (T + kAttnSub - 1) / kAttnSub;
  int per = (steps + want - 1) / want;
  while ((steps + per - 1) / per > kAttnMaxSplit) ++per;
  return per * kAttnSub;
}
int attn_units(int T, int Hkv) { const int s = attn_span(T, Hkv); return (T + s - 1) / s; }
size_t attn_part_bytes(int B, int Hq, int Hkv, int T) {
  return sizeof(float) * (size_t)B * Hq * attn_units(T, Hkv) * kPartRow;
}

}  // namespace

size_t attention_ws_bytes(int B, int Hq, int Hkv, int T) {
  return attn_part_bytes(B, Hq, Hkv, T) + sizeof(unsigned int) * (size_t)B * Hkv;
}

nt_status launch_attention(const float* q, const uint16_t* kc, const uint16_t* vc, int B, int Hq, int Hkv, int T,
                           int ts, float* out, void* ws, cudaStream_t st, const int* T_dev) {
  float* part = static_cast<float*>(ws);
  unsigned int* done = reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(ws) + attn_part_bytes(B, Hq, Hkv, T));
  AttnArgs a{q, kc, vc, part, done, out, B, Hq, Hkv, T, ts, attn_units(T, Hkv), attn_span(T, Hkv),
             (float)(1.4426950408889634 / sqrt((double)kAttnD)), T_dev};
  switch (Hq / Hkv) {
    case 1: return launch_attn_units<1>(a, st);
    case 2: return launch_attn_units<2>(a, st);
    case 4: return launch_attn_units<4>(a, st);
    default: return launch_attn_units<8>(a, st);
  }
}

nt_status launch_rope_append(const float* q, const float* k, const float* v, int B, int Hq, int Hkv, int pos0,
                             float base, float* q_out, uint16_t* kc, uint16_t* vc, int ts, cudaStream_t st,
                             const int* pos_dev) {
  rope_append_kernel<<<B, 256, 0, st>>>(q, k, v, Hq, Hkv, pos0, pos_dev, log2((double)base), q_out, kc, vc, ts);
  return check_launch("rope_append_kernel");
}

nt_status launch_rmsnorm(const float* x, const float* gamma, int B, int D, float eps, float* y, cudaStream_t st) {
  rmsnorm_kernel<<<B, 256, 0, st>>>(x, gamma, D, eps, y);
  return check_launch("rmsnorm_kernel");
}

}  // namespace nt

using namespace nt;

extern "C" {

nt_status nt_attention_workspace_size(int B, int Hq, int Hkv, int T, size_t* bytes) {
  clear_error();
  if (!bytes || B < 1 || Hq < 1 || Hkv < 1 || T < 1)
    return set_error(NT_ERR_INVALID_ARG, "need B, Hq, Hkv, T >= 1 and a result pointer");
  *bytes = attention_ws_bytes(B, Hq, Hkv, T);
  return NT_OK;
}

nt_status nt_attention_decode(const float* q, const uint16_t* k_cache, const uint16_t* v_cache, int B, int Hq,
                              int Hkv, int D, int T, int t_stride, float* out, void* ws, size_t ws_bytes,
                              void* stream) {
  clear_error();
  if (!q || !k_cache || !v_cache || !out || !ws) return set_error(NT_ERR_INVALID_ARG, "NULL pointer");
  if (D != kAttnD) return set_error(NT_ERR_UNSUPPORTED, "head dimension must be 128");
  if (Hkv < 1 || Hq < Hkv || Hq % Hkv != 0) return set_error(NT_ERR_INVALID_ARG, "Hq must be a multiple of Hkv");
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return set_error(NT_ERR_UNSUPPORTED, "Hq / Hkv must be 1, 2, 4 or 8");
  if (B < 1 || B > 64 || T < B || t_stride < T) return set_error(NT_ERR_INVALID_ARG, "need 1 <= B <= 64, B <= T <= t_stride");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 4) || !aligned(ws, 16))
    return set_error(NT_ERR_ALIGNMENT, "q, caches and workspace must be 16-byte aligned");
  if (ws_bytes < attention_ws_bytes(B, Hq, Hkv, T)) return set_error(NT_ERR_WORKSPACE, "workspace too small");
  NT_TRY(check_device());
  return launch_attention(q, k_cache, v_cache, B, Hq, Hkv, T, t_stride, out, ws,
                          reinterpret_cast<cudaStream_t>(stream));
}

nt_status nt_rope_append(const float* q, const float* k_new, const float* v_new, int B, int Hq, int Hkv, int D,
                         int pos0, float base, float* q_out, uint16_t* k_cache, uint16_t* v_cache, int t_stride,
                         void* stream) {
  clear_error();
  if (!q || !k_new || !v_new || !q_out || !k_cache || !v_cache) return set_error(NT_ERR_INVALID_ARG, "NULL pointer");
  if (D != kAttnD) return set_error(NT_ERR_UNSUPPORTED, "head dimension must be 128");
  if (B < 1 || Hq < 1 || Hkv < 1 || pos0 < 0 || pos0 + B > t_stride || !(base > 1.0f))
    return set_error(NT_ERR_INVALID_ARG, "need B, Hq, Hkv >= 1, 0 <= pos0, pos0 + B <= t_stride and base > 1");
  if (!aligned(q, 4) || !aligned(k_new, 4) || !aligned(v_new, 4) || !aligned(q_out, 4) || !aligned(k_cache, 2) ||
      !aligned(v_cache, 2))
    return set_error(NT_ERR_ALIGNMENT, "misaligned pointer");
  NT_TRY(check_device());
  return launch_rope_append(q, k_new, v_new, B, Hq, Hkv, pos0, base, q_out, k_cache, v_cache, t_stride,
                            reinterpret_cast<cudaStream_t>(stream));
}

nt_status nt_rmsnorm(const float* x, const float* gamma, int B, int D, float eps, float* y, void* stream) {
  clear_error();
  if (!x || !gamma || !y) return set_error(NT_ERR_INVALID_ARG, "NULL pointer");
  if (B < 1 || D < 1 || !(eps >= 0.0f)) return set_error(NT_ERR_INVALID_ARG, "need B, D >= 1 and eps >= 0");
  if (!aligned(x, 4) || !aligned(gamma, 4) || !aligned(y, 4)) return set_error(NT_ERR_ALIGNMENT, "misaligned pointer");
  NT_TRY(check_device());
  return launch_rmsnorm(x, gamma, B, D, eps, y, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
