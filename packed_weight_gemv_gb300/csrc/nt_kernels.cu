// nt_kernels.cu -- activation quantization, load-time repack, the per-call ternary projection
// kernels (plain and tiled layouts) and the int8 output projection with fused arg-max.
//
// The arithmetic is the reading stated in nt.h of "The Neutrino Engine" (Fermion Research):
// exact int32 sums of trit x int8 products (§ "A 104 microsecond floor inside a 694
// microsecond step": each weight feeds one multiply-accumulate per token), a per-row scale
// (§ "The file is not the traffic"), and the greedy arg-max (§ "One changed token fails the
// release").
#include <float.h>
#include <math.h>
#include <limits.h>

#include "nt_kernels.cuh"
#include "nt_step.cuh"

namespace nt {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChainThreads = 256;  // stage-input kernel: one CTA per vector
constexpr int kChainWarps = kChainThreads / 32;

// 16-byte streaming load that bypasses L1 allocation (weights are read once per token).
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------------------------------
// Quantization: one CTA per vector. Absmax by block reduction (max is exact in any order),
// then q = clamp(rint(x / s)) with an IEEE fp32 quotient.
// ---------------------------------------------------------------------------------------
__device__ void quantize_vector(const float* __restrict__ x, int K, int8_t* __restrict__ q,
                                float* __restrict__ s_out) {
  __shared__ float red[kWarps];
  float m = 0.0f;
  for (int k = threadIdx.x; k < K; k += blockDim.x) m = fmaxf(m, fabsf(x[k]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  m = red[0];
  for (int i = 1; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
  const float s = (m == 0.0f) ? 0.0f : __fdiv_rn(m, 127.0f);
  if (threadIdx.x == 0) *s_out = s;
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    int v = 0;
    if (m != 0.0f) {
      v = __float2int_rn(__fdiv_rn(x[k], s));
      v = v > 127 ? 127 : (v < -127 ? -127 : v);
    }
    q[k] = (int8_t)v;
  }
  __syncthreads();  // red[] is reused by the next vector of the same CTA
}

__global__ void __launch_bounds__(kThreads) quantize_kernel(const float* __restrict__ x, int K,
                                                            int8_t* __restrict__ q,
                                                            float* __restrict__ s) {
  const int b = blockIdx.x;
  quantize_vector(x + (int64_t)b * K, K, q + (int64_t)b * K, s + b);
}

__global__ void __launch_bounds__(kThreads) quantize_jobs_kernel(const QuantJob* __restrict__ jobs,
                                                                 int max_B) {
  dependent_launch_wait();
  const QuantJob j = jobs[blockIdx.x];
  const int b = blockIdx.y;
  if (b >= j.B) return;
  quantize_vector(j.x + (int64_t)b * j.K, j.K, j.q + (int64_t)b * j.K, j.s + b);
}

// Chained stage input of vector blockIdx.x (stream / graph launchers): the fp32 values go to
// job.vbuf with the absmax (for kChainSum vbuf is the residual stream, updated in place: each
// thread rewrites only the elements it read), then the codes to every recorded q.
__global__ void __launch_bounds__(kChainThreads) chain_quant_kernel(const ChainJob* __restrict__ jobs) {
  __shared__ float red[kChainWarps];
  __shared__ float s_r;
  dependent_launch_wait();
  const ChainJob j = *jobs;
  const int b = blockIdx.x, K = j.src.K;
  float* vb = j.vbuf + (int64_t)b * K;
  float m = 0.0f, sf = 0.0f;
  for (int k = 4 * threadIdx.x; k < K; k += 4 * kChainThreads) {
    const float4 v = chain_load4(j.src, b, k);
    *reinterpret_cast<float4*>(vb + k) = v;
    m = fmaxf(fmaxf(m, fmaxf(fabsf(v.x), fabsf(v.y))), fmaxf(fabsf(v.z), fabsf(v.w)));
    sf = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, sf))));  // a few squares in fp32
  }
  float r = 1.0f;
  if (j.src.gamma) {  // RMS normalisation: the absmax is taken over the normalised values
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sf += __shfl_xor_sync(0xffffffffu, sf, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sf;
    __syncthreads();
    if (threadIdx.x == 0) {  // the warps' sums added and r formed in double by one thread
      double t = 0.0;
      for (int i = 0; i < kChainWarps; ++i) t += red[i];
      s_r = (float)(1.0 / sqrt(t / K + (double)j.src.eps));
    }
    __syncthreads();  // s_r visible; red[] is reused for the maximum
    r = s_r;
    m = 0.0f;
    for (int k = 4 * threadIdx.x; k < K; k += 4 * kChainThreads) {
      const float4 v = *reinterpret_cast<const float4*>(vb + k);
      const float4 g = *reinterpret_cast<const float4*>(j.src.gamma + k);
      m = fmaxf(m, fabsf(__fmul_rn(__fmul_rn(v.x, r), g.x)));
      m = fmaxf(m, fabsf(__fmul_rn(__fmul_rn(v.y, r), g.y)));
      m = fmaxf(m, fabsf(__fmul_rn(__fmul_rn(v.z, r), g.z)));
      m = fmaxf(m, fabsf(__fmul_rn(__fmul_rn(v.w, r), g.w)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  m = red[0];
#pragma unroll
  for (int i = 1; i < kChainWarps; ++i) m = fmaxf(m, red[i]);
  const bool nz = m != 0.0f;
  const float s = nz ? __fdiv_rn(m, 127.0f) : 0.0f;
  if (threadIdx.x == 0)
    for (int rr = 0; rr < j.n_rec; ++rr) j.s[rr][b] = s;
  for (int k = 4 * threadIdx.x; k < K; k += 4 * kChainThreads) {
    float4 v = *reinterpret_cast<const float4*>(vb + k);
    if (j.src.gamma) {
      const float4 g = *reinterpret_cast<const float4*>(j.src.gamma + k);
      v = make_float4(__fmul_rn(__fmul_rn(v.x, r), g.x), __fmul_rn(__fmul_rn(v.y, r), g.y),
                      __fmul_rn(__fmul_rn(v.z, r), g.z), __fmul_rn(__fmul_rn(v.w, r), g.w));
    }
    const uint32_t c = quant4(v, s, nz);
    if (j.src.cap) *reinterpret_cast<float4*>(j.src.cap + (int64_t)b * K + k) = v;
    for (int rr = 0; rr < j.n_rec; ++rr) *reinterpret_cast<uint32_t*>(j.q[rr] + (int64_t)b * K + k) = c;
  }
}

// ---------------------------------------------------------------------------------------
// Repack plain -> tiled. Word (row n, group g) of the tiled layout holds the same 16 trits
// as plain word g of row n, re-coded as 8 pair codes. One thread per 16-byte tiled group (the
// 4 rows of a tile at one group): its 4 plain reads are coalesced across the warp (consecutive
// threads take consecutive groups of a row) and its 16-byte store too.
// ---------------------------------------------------------------------------------------
// Pair code of trits (a, b), by index (a + 1) * 3 + (b + 1), one nibble each: 7, 2, 5, 14, 0,
// 3, 6, 1, 4 (see the pools in nt_internal.cuh).
constexpr uint64_t kPairCodes = 0x41630E527ull;

// Index a + 1 of a plain field (00 -> 1, 01 -> 2, 11 -> 0; the invalid 10 reads as 0 -> 1).
__device__ __forceinline__ uint32_t field_index(uint32_t w, int j) {
  const uint32_t c = (w >> (2 * j)) & 3u;
  return c == 1u ? 2u : (c == 3u ? 0u : 1u);
}

__device__ __forceinline__ uint32_t tiled_word(uint32_t src) {
  uint32_t word = 0;
#pragma unroll
  for (int i4 = 0; i4 < 4; ++i4) {
    const uint32_t lo = (uint32_t)(kPairCodes >> (4 * (field_index(src, i4) * 3 + field_index(src, 4 + i4)))) & 15u;
    const uint32_t hi = (uint32_t)(kPairCodes >> (4 * (field_index(src, 8 + i4) * 3 + field_index(src, 12 + i4)))) & 15u;
    word |= lo << (4 * i4);
    word |= hi << (4 * (4 + i4));
  }
  return word;
}

__global__ void __launch_bounds__(kThreads) repack_kernel(const uint32_t* __restrict__ w, int N,
                                                          int K, uint32_t* __restrict__ out,
                                                          uint32_t* __restrict__ n_invalid) {
  const int64_t groups = padded_k(K) / 16, kw = K / 16;
  const int64_t total = padded_rows(N) / 4 * groups;  // tiled groups, in memory order
  unsigned int bad = 0;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t tile = i / groups, g = i - tile * groups;
    uint32_t src[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int64_t n = tile * 4 + r;
      src[r] = (n < N && g < kw) ? __ldg(w + n * kw + g) : 0u;
    }
    uint4 o;
    uint32_t* ow = &o.x;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
#pragma unroll
      for (int f = 0; f < 16; ++f) bad += ((src[r] >> (2 * f)) & 3u) == 2u;
      ow[r] = tiled_word(src[r]);
    }
    reinterpret_cast<uint4*>(out)[i] = o;
  }
  if (n_invalid) {
    bad = __reduce_add_sync(0xffffffffu, bad);
    if ((threadIdx.x & 31) == 0 && bad) atomicAdd(n_invalid, bad);
  }
}

// Counts the invalid 10 fields of a plain matrix: a field is 10 when its high bit is set and
// its low bit clear, so (w >> 1) & ~w & 0x55555555 has one bit per invalid field.
__global__ void __launch_bounds__(kThreads) validate_kernel(const uint32_t* __restrict__ w, int64_t n_words,
                                                            unsigned long long* __restrict__ n_invalid) {
  unsigned int bad = 0;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_words; i += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t v = __ldg(w + i);
    bad += __popc((v >> 1) & ~v & 0x55555555u);
  }
  bad = __reduce_add_sync(0xffffffffu, bad);
  if ((threadIdx.x & 31) == 0 && bad) atomicAdd(n_invalid, (unsigned long long)bad);
}

// ---------------------------------------------------------------------------------------
// Plain-layout projection: one warp per row, lanes over the row's words. NB activation
// vectors per pass; larger batches loop over passes.
// ---------------------------------------------------------------------------------------
template <int NB>
__global__ void __launch_bounds__(kThreads) gemv_plain_kernel(
    const uint32_t* __restrict__ w, const float* __restrict__ s_w, int N, int K,
    const int8_t* __restrict__ q, const float* __restrict__ s_x, int B, float* __restrict__ y,
    int32_t* __restrict__ acc_out) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * kWarps;
  const int words = K / 16;
  for (int b0 = 0; b0 < B; b0 += NB) {
    for (int64_t n = warp; n < N; n += nwarps) {
      int acc[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) acc[b] = 0;
      const uint32_t* row = w + n * words;
      for (int j = lane; j < words; j += 32) {
        const uint32_t wd = __ldg(row + j);
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          if (b0 + b < B) {
            const uint4 a = *reinterpret_cast<const uint4*>(q + (int64_t)(b0 + b) * K + 16 * j);
            acc[b] = plain_word_dot(wd, a.x, a.y, a.z, a.w, acc[b]);
          }
        }
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const int total = warp_sum(acc[b]);
        if (lane == 0 && b0 + b < B) {
          const int64_t o = (int64_t)(b0 + b) * N + n;
          y[o] = scale_out(total, s_w[n], s_x[b0 + b]);
          if (acc_out) acc_out[o] = total;
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------------------
// Tiled-layout projection: one warp per tile (4 rows). Lane l reads 16-byte groups
// l, l+32, ... (4 rows x 16 trits each) and the matching 16 activation bytes; each group
// costs one shift, four byte permutes and four dp4a per row. The weight loads of U groups
// per lane go out together, so a warp keeps U x 512 bytes in flight.
// ---------------------------------------------------------------------------------------
template <int NB>
__device__ __forceinline__ void tiled_tile(const MatDesc& m, int64_t tile, int lane) {
  constexpr int U = NB <= 4 ? 4 : 2;
  const int64_t Kp = padded_k(m.K);
  const int groups = (int)(Kp / 16), kgroups = m.K / 16;
  const uint8_t* tbase = m.w + tile * Kp;
  for (int b0 = 0; b0 < m.B; b0 += NB) {
    int acc[NB][4];
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[b][r] = 0;
    for (int g0 = lane; g0 < groups; g0 += 32 * U) {
      uint4 wv[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int g = g0 + 32 * u;
        wv[u] = g < groups ? ld_stream(tbase + 16 * (int64_t)g) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int g = g0 + 32 * u;
        if (g < kgroups) {
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            if (b0 + b < m.B) {
              const uint4 a = *reinterpret_cast<const uint4*>(m.q + (int64_t)(b0 + b) * m.K + 16 * g);
              acc[b][0] = tiled_word_dot(wv[u].x, a.x, a.y, a.z, a.w, acc[b][0]);
              acc[b][1] = tiled_word_dot(wv[u].y, a.x, a.y, a.z, a.w, acc[b][1]);
              acc[b][2] = tiled_word_dot(wv[u].z, a.x, a.y, a.z, a.w, acc[b][2]);
              acc[b][3] = tiled_word_dot(wv[u].w, a.x, a.y, a.z, a.w, acc[b][3]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int total = warp_sum(acc[b][r]);
        const int64_t n = tile * 4 + r;
        if (lane == r && b0 + b < m.B && n < m.N) {
          const int64_t o = (int64_t)(b0 + b) * m.N + n;
          m.y[o] = scale_out(total, m.s_w[n], m.s_x[b0 + b]);
          if (m.acc) m.acc[o] = total;
        }
      }
    }
  }
}

template <int NB>
__global__ void __launch_bounds__(kThreads) gemv_tiled_kernel(const MatDesc m) {
  dependent_launch_wait();
  const int lane = threadIdx.x & 31;
  const int64_t tiles = padded_rows(m.N) / 4;
  for (int64_t t = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); t < tiles;
       t += (int64_t)gridDim.x * kWarps)
    tiled_tile<NB>(m, t, lane);
}

template <int NB>
__global__ void __launch_bounds__(kThreads) gemv_tiled_group_kernel(
    const MatDesc* __restrict__ mats, const int64_t* __restrict__ prefix, int n, int64_t total) {
  dependent_launch_wait();
  const int lane = threadIdx.x & 31;
  for (int64_t t = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); t < total;
       t += (int64_t)gridDim.x * kWarps) {
    int lo = 0, hi = n - 1;  // last matrix whose prefix <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const MatDesc m = mats[lo];
    tiled_tile<NB>(m, t - prefix[lo], lane);
  }
}

// ---------------------------------------------------------------------------------------
// int8 output projection with fused greedy arg-max. One warp per vocabulary row, lanes over
// 16-byte chunks; each warp keeps its best (logit, row), the CTA reduces its warps, and the
// last CTA to finish reduces all CTAs (lowest row among equal logits) and resets the
// counter, so the workspace is ready for the next call.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

template <int NB>
__global__ void __launch_bounds__(kThreads) head_kernel(
    const int8_t* __restrict__ T, const float* __restrict__ s_T, int V, int K,
    const int8_t* __restrict__ q, const float* __restrict__ s_x, int B, float* __restrict__ logits,
    int32_t* __restrict__ argmax, HeadWs* __restrict__ ws) {
  __shared__ HeadPartial wbest[kWarps][NB];
  __shared__ bool last;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int64_t warp = (int64_t)blockIdx.x * kWarps + wid, nwarps = (int64_t)gridDim.x * kWarps;
  const int chunks = K / 16;
  for (int b0 = 0; b0 < B; b0 += NB) {
    float bv[NB];
    int bi[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) { bv[b] = -INFINITY; bi[b] = INT_MAX; }
    for (int64_t v = warp; v < V; v += nwarps) {
      int acc[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) acc[b] = 0;
      const int8_t* row = T + v * K;
      for (int c = lane; c < chunks; c += 32) {
        const uint4 t = ld_stream(row + 16 * (int64_t)c);
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          if (b0 + b < B) {
            const uint4 a = *reinterpret_cast<const uint4*>(q + (int64_t)(b0 + b) * K + 16 * c);
            acc[b] = dp4a(t.x, a.x, acc[b]);
            acc[b] = dp4a(t.y, a.y, acc[b]);
            acc[b] = dp4a(t.z, a.z, acc[b]);
            acc[b] = dp4a(t.w, a.w, acc[b]);
          }
        }
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const int total = warp_sum(acc[b]);
        if (b0 + b < B) {
          const float lg = scale_out(total, s_T[v], s_x[b0 + b]);
          if (lane == 0 && logits) logits[(int64_t)(b0 + b) * V + v] = lg;
          if (lg > bv[b]) { bv[b] = lg; bi[b] = (int)v; }  // rows rise within a warp
        }
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int b = 0; b < NB; ++b) wbest[wid][b] = HeadPartial{bv[b], bi[b]};
    }
    __syncthreads();
    if (threadIdx.x < NB && b0 + (int)threadIdx.x < B) {
      const int b = threadIdx.x;
      HeadPartial best = wbest[0][b];
      for (int i = 1; i < kWarps; ++i)
        if (better(wbest[i][b].val, wbest[i][b].idx, best.val, best.idx)) best = wbest[i][b];
      ws->part[(int64_t)blockIdx.x * B + b0 + b] = best;
    }
    __syncthreads();
  }
  // Cross-CTA reduction by the last CTA to arrive.
  __threadfence();
  if (threadIdx.x == 0) last = (atomicAdd(&ws->done, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (int b = wid; b < B; b += kWarps) {
    float best_v = -INFINITY;
    int best_i = INT_MAX;
    for (int c = lane; c < (int)gridDim.x; c += 32) {
      const HeadPartial* pp = &ws->part[(int64_t)c * B + b];
      const float pv = __ldcg(&pp->val);
      const int pi = __ldcg(&pp->idx);
      if (better(pv, pi, best_v, best_i)) { best_v = pv; best_i = pi; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best_v, o);
      const int oi = __shfl_xor_sync(0xffffffffu, best_i, o);
      if (better(ov, oi, best_v, best_i)) { best_v = ov; best_i = oi; }
    }
    if (lane == 0) argmax[b] = best_i == INT_MAX ? 0 : best_i;
  }
  if (threadIdx.x == 0) ws->done = 0u;
}

int grid_for(int64_t warps_needed, int per_sm) {
  const int64_t cap = (int64_t)device_sm_count() * per_sm;
  int64_t g = (warps_needed + kWarps - 1) / kWarps;
  if (g > cap) g = cap;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace

// ---------------------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------------------
nt_status launch_quantize(const float* x, int B, int K, int8_t* q, float* s, cudaStream_t st) {
  quantize_kernel<<<B, kThreads, 0, st>>>(x, K, q, s);
  return check_launch("quantize_kernel");
}

nt_status launch_quantize_jobs(const QuantJob* d_jobs, int n_jobs, int max_B, cudaStream_t st, bool pdl) {
  NT_CUDA_TRY(launch_kernel(quantize_jobs_kernel, dim3(n_jobs, max_B), dim3(kThreads), 0, st, pdl, d_jobs, max_B));
  return check_launch("quantize_jobs_kernel");
}

nt_status launch_chain_quant(const ChainJob* d_job, int B, cudaStream_t st, bool pdl) {
  NT_CUDA_TRY(launch_kernel(chain_quant_kernel, dim3(B), dim3(kChainThreads), 0, st, pdl, d_job));
  return check_launch("chain_quant_kernel");
}

nt_status launch_repack(const uint32_t* w, int N, int K, uint8_t* out, uint32_t* n_invalid,
                        cudaStream_t st) {
  const int64_t total = padded_rows(N) / 4 * (padded_k(K) / 16);  // one thread per 16-byte group
  int64_t g = (total + kThreads - 1) / kThreads;
  const int64_t cap = (int64_t)device_sm_count() * 16;
  if (g > cap) g = cap;
  repack_kernel<<<(int)g, kThreads, 0, st>>>(w, N, K, reinterpret_cast<uint32_t*>(out), n_invalid);
  return check_launch("repack_kernel");
}

nt_status launch_validate(const uint32_t* w, int N, int K, unsigned long long* n_invalid, cudaStream_t st) {
  const int64_t words = (int64_t)N * (K / 16);
  int64_t g = (words + kThreads - 1) / kThreads;
  const int64_t cap = (int64_t)device_sm_count() * 16;
  if (g > cap) g = cap;
  validate_kernel<<<(int)g, kThreads, 0, st>>>(w, words, n_invalid);
  return check_launch("validate_kernel");
}

nt_status launch_gemv_plain(const uint32_t* w, const float* s_w, int N, int K, const int8_t* q,
                            const float* s_x, int B, float* y, int32_t* acc, cudaStream_t st) {
  const int g = grid_for(N, 8);
  if (B == 1) gemv_plain_kernel<1><<<g, kThreads, 0, st>>>(w, s_w, N, K, q, s_x, B, y, acc);
  else if (B == 2) gemv_plain_kernel<2><<<g, kThreads, 0, st>>>(w, s_w, N, K, q, s_x, B, y, acc);
  else if (B <= 4) gemv_plain_kernel<4><<<g, kThreads, 0, st>>>(w, s_w, N, K, q, s_x, B, y, acc);
  else gemv_plain_kernel<8><<<g, kThreads, 0, st>>>(w, s_w, N, K, q, s_x, B, y, acc);
  return check_launch("gemv_plain_kernel");
}

// One call: a programmatic dependent launch, so back-to-back calls overlap one call's launch
// and ramp with the previous call's drain (the kernel waits for its predecessor before it
// reads anything; after a kernel that does not signal early it simply starts after it).
nt_status launch_gemv_tiled(const MatDesc& m, cudaStream_t st) {
  const int g = grid_for(padded_rows(m.N) / 4, 8);
  auto kern = m.B == 1 ? gemv_tiled_kernel<1> : m.B == 2 ? gemv_tiled_kernel<2>
            : m.B <= 4 ? gemv_tiled_kernel<4> : m.B <= 8 ? gemv_tiled_kernel<8> : gemv_tiled_kernel<16>;
  NT_CUDA_TRY(launch_kernel(kern, dim3(g), dim3(kThreads), 0, st, true, m));
  return check_launch("gemv_tiled_kernel");
}

nt_status launch_gemv_tiled_group(const MatDesc* d_mats, const int64_t* d_prefix, int n,
                                  int64_t total, int max_B, cudaStream_t st, bool pdl) {
  const int g = grid_for(total, 8);
  auto kern = max_B == 1 ? gemv_tiled_group_kernel<1> : max_B == 2 ? gemv_tiled_group_kernel<2>
            : max_B <= 4 ? gemv_tiled_group_kernel<4> : max_B <= 8 ? gemv_tiled_group_kernel<8>
                         : gemv_tiled_group_kernel<16>;
  NT_CUDA_TRY(launch_kernel(kern, dim3(g), dim3(kThreads), 0, st, pdl, d_mats, d_prefix, n, total));
  return check_launch("gemv_tiled_group_kernel");
}

nt_status launch_head(const int8_t* T, const float* s_T, int V, int K, const int8_t* q,
                      const float* s_x, int B, float* logits, int32_t* argmax, HeadWs* ws,
                      cudaStream_t st, bool pdl) {
  if (B >= kMmaMinBatch && B <= kMmaMaxBatch)  // one pass over T on the tensor cores
    return launch_head_mma(T, s_T, V, K, q, s_x, B, logits, argmax, ws, st);
  if (persist_head_fits(K, B))  // the streaming kernel (bulk copies into per-warp rings)
    return persist_launch_head(T, s_T, V, K, q, s_x, B, logits, argmax, ws, st, pdl);
  int g = grid_for(V, 4);
  if (g > kHeadMaxCtas) g = kHeadMaxCtas;
  if (B == 1) head_kernel<1><<<g, kThreads, 0, st>>>(T, s_T, V, K, q, s_x, B, logits, argmax, ws);
  else if (B == 2) head_kernel<2><<<g, kThreads, 0, st>>>(T, s_T, V, K, q, s_x, B, logits, argmax, ws);
  else if (B <= 4) head_kernel<4><<<g, kThreads, 0, st>>>(T, s_T, V, K, q, s_x, B, logits, argmax, ws);
  else if (B <= 8) head_kernel<8><<<g, kThreads, 0, st>>>(T, s_T, V, K, q, s_x, B, logits, argmax, ws);
  else head_kernel<16><<<g, kThreads, 0, st>>>(T, s_T, V, K, q, s_x, B, logits, argmax, ws);
  return check_launch("head_kernel");
}

}  // namespace nt
