// nt_attention.cu -- the attention side of a decoder layer: grouped-query attention of the
// new positions over a bf16 key-value cache, the rotary embedding with the cache append, and
// RMS normalisation ("The Neutrino Engine", § "At 26K tokens, the cache becomes larger than
// the model": 8 key-value heads of 128 dimensions, 16-bit cache entries, grouped-query
// attention).
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>
#include <atomic>

#include "nt_kernels.cuh"

namespace nt {
namespace {

constexpr int kAttnD = 128;        // dimensions per head
constexpr int kAttnStep = 16;      // cache positions per warp step (two 8-position score tiles)
constexpr int kAttnWarps = 4;
constexpr int kAttnThreads = 32 * kAttnWarps;
constexpr int kAttnMaxSplit = 512;
constexpr int kPartRow = kAttnD + 4;  // floats per partial result: weighted sum, max, sum, padding
constexpr float kAttnLazy = 8.0f;     // a running maximum is raised only once a score exceeds it by 2^8

// CTAs of the unit kernel resident per SM (its launch bounds).
constexpr int attn_resident(int G) { return G > 4 ? 1 : 2; }

struct AttnArgs {
  const float* q;      // [B][Hq][D]
  const uint16_t* kc;  // [Hkv][ts][D] bf16
  const uint16_t* vc;
  float* part;         // [B][Hq][nch][kPartRow]: weighted value sum, reference max (log2 units), sum
  unsigned int* done;  // [B][Hkv]: units finished; the last CTA of a group merges and resets it
  float* out;          // [B][Hq][D]
  int B, Hq, Hkv, T, ts, nch, span;  // span: positions per unit (a multiple of kAttnStep)
  float scale_log2;    // log2(e) / sqrt(D)
  const int* T_dev;    // when set, the cache length is *T_dev (T then only sized the grid)
};

__device__ __forceinline__ unsigned int atom_add_acq_rel(unsigned int* p, unsigned int v) {
  unsigned int old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// D += A * B on the tensor cores: A 16 x 16 bf16 (row major), B 16 x 8 bf16, D 16 x 8 fp32.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ float bf16_rn(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

__device__ __forceinline__ uint32_t word(const uint4& v, int c) {
  return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w;
}

template <int N>
__device__ __forceinline__ float pick(const float (&v)[N], int i) {
  float r = v[0];
#pragma unroll
  for (int k = 1; k < N; ++k) r = i == k ? v[k] : r;
  return r;
}

// ---- per-warp ring of cache rows in shared memory, filled by bulk copies ------------------
constexpr int kAttnStages = 3;                               // steps in flight per warp
constexpr int kRowPitch = kAttnD * 2;                        // rows as in the cache
constexpr int kStageBytes = 2 * kAttnStep * kRowPitch;       // keys then values
constexpr int kRingBytes = kAttnWarps * kAttnStages * kStageBytes;
constexpr uint64_t kAttnTimeoutNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false once the deadline has passed.
__device__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t deadline = globaltimer_ns() + kAttnTimeoutNs;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0u && globaltimer_ns() > deadline) return false;
  }
}

// Issue the copies of one warp step (positions p0 .. p0 + 15, those below vis) into a stage:
// the key rows and the value rows, each one contiguous cp.async.bulk completing on the stage's
// mbarrier. Lane 0.
__device__ __forceinline__ void attn_issue(const uint16_t* kh, const uint16_t* vh, int p0, int vis, uint32_t stage,
                                           uint32_t bar, uint64_t pol, int lane) {
  if (lane != 0) return;
  const uint32_t bytes = (uint32_t)min(kAttnStep, vis - p0) * (kAttnD * 2);
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(2u * bytes) : "memory");
#pragma unroll
  for (int isv = 0; isv < 2; ++isv)
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(stage + (uint32_t)(isv * kAttnStep * kRowPitch)),
        "l"((isv ? vh : kh) + (int64_t)p0 * kAttnD), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}

// Registers of one step from its stage: keys of positions g and 8 + g (64 bytes each, dims
// 32 i + 8 t ..), values of positions 2t, 2t + 1, 2t + 8, 2t + 9 (dims 8g .. 8g + 7 and
// 64 + 8g ..). Value rows at or past vis read as zero (the stage holds stale rows there).
__device__ __forceinline__ void attn_read(const uint8_t* stage, int p0, int vis, bool full, int g, int t,
                                          uint4 (&kw)[2][4], uint4 (&vw)[4][2]) {
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const uint8_t* row = stage + (8 * nt + g) * kRowPitch + 16 * t;
#pragma unroll
    for (int ii = 0; ii < 4; ++ii) kw[nt][ii] = *reinterpret_cast<const uint4*>(row + 64 * ii);
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int pr = 2 * t + (r & 1) + 8 * (r >> 1);
    const uint8_t* row = stage + (kAttnStep + pr) * kRowPitch + 16 * g;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf)
      vw[r][hf] = full || p0 + pr < vis ? *reinterpret_cast<const uint4*>(row + 128 * hf) : make_uint4(0u, 0u, 0u, 0u);
  }
}

__device__ __forceinline__ float ex2(float x) {  // 2^x (MUFU; 2^-inf = +0)
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One warp step: scores, softmax update and weighted values of positions p0 .. p0 + 15.
// `full`: all 16 positions are below vis (the same in every lane).
template <int G, int HG>
__device__ __forceinline__ void attn_compute(const uint32_t (&qa)[HG][8][4], float (&O)[HG][8][4],
                                             float (&mref)[HG][4], float (&lsum)[HG], const uint4 (&kw)[2][4],
                                             const uint4 (&vw)[4][2], int p0, int vis, bool full, int g, int t) {
  const int hl = g & 3;
#pragma unroll
  for (int grp = 0; grp < HG; ++grp) {
    const bool used = grp * 4 + hl < G;
    float s[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      float d0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, d1[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // two chains
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
        mma_16816(d0, qa[grp][j][0], qa[grp][j][1], qa[grp][j][2], qa[grp][j][3], word(kw[nt][j >> 1], 0),
                  word(kw[nt][j >> 1], 1));
        mma_16816(d1, qa[grp][j + 1][0], qa[grp][j + 1][1], qa[grp][j + 1][2], qa[grp][j + 1][3],
                  word(kw[nt][j >> 1], 2), word(kw[nt][j >> 1], 3));
      }
      const float x0 = (d0[0] + d1[0]) + (d0[2] + d1[2]), x1 = (d0[1] + d1[1]) + (d0[3] + d1[3]);
      s[nt][0] = x0 + __shfl_xor_sync(0xffffffffu, x0, 16);
      s[nt][1] = x1 + __shfl_xor_sync(0xffffffffu, x1, 16);
      if (!full || (G < 4 && !used)) {
#pragma unroll
        for (int e = 0; e < 2; ++e)
          if (!used || p0 + 8 * nt + 2 * t + e >= vis) s[nt][e] = -INFINITY;
      }
    }
    float my = pick(mref[grp], hl);
    const float mx = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
    if (__any_sync(0xffffffffu, mx > my + kAttnLazy)) {  // rare after the first step
      float m4 = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      m4 = fmaxf(m4, __shfl_xor_sync(0xffffffffu, m4, 2));
      float corr[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float sm = __shfl_sync(0xffffffffu, m4, 4 * k);
        const float mn = fmaxf(mref[grp][k], sm);
        corr[k] = mn == mref[grp][k] ? 1.0f : ex2(mref[grp][k] - mn);
        mref[grp][k] = mn;
      }
      const float c0 = (t & 1) ? corr[2] : corr[0], c1 = (t & 1) ? corr[3] : corr[1];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        O[grp][mt][0] *= c0;
        O[grp][mt][2] *= c0;
        O[grp][mt][1] *= c1;
        O[grp][mt][3] *= c1;
      }
      lsum[grp] *= pick(corr, hl);
      my = pick(mref[grp], hl);
    }
    uint32_t pb[2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const float q0 = used ? ex2(s[nt][0] - my) : 0.0f, q1 = used ? ex2(s[nt][1] - my) : 0.0f;
      const __nv_bfloat162 hi = __floats2bfloat162_rn(q0, q1);
      const __nv_bfloat162 lo = __floats2bfloat162_rn(__fsub_rn(q0, __low2float(hi)), __fsub_rn(q1, __high2float(hi)));
      lsum[grp] += q0 + q1;
      const __nv_bfloat162 term = g < 4 ? hi : lo;
      pb[nt] = *reinterpret_cast<const uint32_t*>(&term);
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int hf = mt >> 2, cc = mt & 3;
      const uint32_t x0 = word(vw[0][hf], cc), x1 = word(vw[1][hf], cc);
      const uint32_t x2 = word(vw[2][hf], cc), x3 = word(vw[3][hf], cc);
      mma_16816(O[grp][mt], __byte_perm(x0, x1, 0x5410), __byte_perm(x0, x1, 0x7632),
                __byte_perm(x2, x3, 0x5410), __byte_perm(x2, x3, 0x7632), pb[0], pb[1]);
    }
  }
}

// One CTA of 4 warps per (unit of `span` cache positions, key-value head), two CTAs per SM.
// Each warp walks 16-position steps of the unit (warp w takes steps w, w + 4, ...): its lane 0
// keeps three steps of key and value rows in flight (bulk copies into the warp's ring in shared
// memory, completing on one mbarrier per stage), and both products run on the tensor cores
// (mma.sync m16n8k16, bf16 operands, fp32 accumulation):
//
// * scores S[16 x 8] = Q[16 x 128] K^T per 8 positions. The rows of Q are the group's 4 query
//   heads, each split into three bf16 terms (hi, mid, lo: q = hi + mid + lo to ~2^-26
//   relative), row = 4 * term + head; K is the MMA's column operand, lane (g, t) reading 16
//   contiguous bytes of position g per 32 dimensions (the dimension order inside the MMA is
//   permuted; Q uses the same permutation). The three terms' rows are added in fp32, one
//   shuffle joining the lanes that hold them.
// * softmax: scores are in log2 units (q carries log2(e) / sqrt(D)); a running reference max per
//   head is raised only when a score exceeds it by more than 2^8 (a warp vote; weights stay
//   <= 256, so nothing overflows), and the accumulators are rescaled then.
// * weighted values O^T[128 x 8] += V^T[128 x 16] P^T[16 x 8]. The columns of P^T are the 4
//   heads' weights split into two bf16 terms (hi, lo: p = hi + lo to ~2^-17 relative); the score
//   tile's register layout is exactly the B operand's, so the weights never leave their lanes.
//   V^T comes from the cache rows with one byte permute per register (two positions' values
//   of one dimension).
//
// Keys and values are exact in bf16, so every product is exact; the sums run in fp32. The 4
// warps' (weighted sums, reference max, weight sum) are merged in shared memory into the unit's
// partial result; the last CTA of each (b, key-value head) to finish merges all units into out
// in one pass.
template <int G>
__global__ void __launch_bounds__(kAttnThreads, attn_resident(G)) attn_unit_kernel(const AttnArgs a) {
  constexpr int HG = (G + 3) / 4;  // groups of 4 query heads
  extern __shared__ __align__(128) uint8_t attn_smem[];
  // the ring; after a position's main loop (no copy in flight) it holds Acc
  float (*Acc)[G][kAttnD] = reinterpret_cast<float (*)[G][kAttnD]>(attn_smem);
  __shared__ __align__(8) uint64_t bars[kAttnWarps][kAttnStages];
  __shared__ float mw[kAttnWarps][G], lw[kAttnWarps][G];
  __shared__ int s_last;
  const int c = blockIdx.x, h = blockIdx.y, i = threadIdx.x, lane = i & 31, w = i >> 5;
  const int g = lane >> 2, t = lane & 3, hl = g & 3;
  // In a dependent-launch chain the previous kernel appends the new positions' rows and rotates
  // the queries; everything older (the cache rows before them, the cache length) was written by
  // kernels that completed before this one could start. So the copies of steps that hold only
  // older rows go out before the wait for the previous kernel, and the rest after it.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  bool waited = false;
  auto wait_previous = [&]() {
    if (!waited) asm volatile("griddepcontrol.wait;" ::: "memory");
    waited = true;
  };
  const int T = a.T_dev ? *a.T_dev : a.T;
  const int u0 = c * a.span, u1 = min(T, u0 + a.span);
  const uint16_t* kh = a.kc + (int64_t)h * a.ts * kAttnD;
  const uint16_t* vh = a.vc + (int64_t)h * a.ts * kAttnD;
  const int64_t head_stride = (int64_t)a.nch * kPartRow;
  const uint32_t ring = smem_u32(attn_smem) + (uint32_t)(w * kAttnStages * kStageBytes);
  const uint32_t bar0 = smem_u32(&bars[w][0]);
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  if (lane == 0) {
#pragma unroll
    for (int st = 0; st < kAttnStages; ++st)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar0 + 8u * st) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();  // this warp's barriers are initialised
  // steps this warp has issued and consumed (step n: stage n % S, phase parity (n / S) & 1)
  uint32_t used_steps = 0, issued_steps = 0;
  bool ok = true;  // false once a copy has not completed within the time limit

  for (int b = 0; b < a.B; ++b) {
    const int vis = min(u1, T - a.B + b + 1);  // positions [u0, vis) are visible to b
    // the warp's first steps go out before the query fragments are built
    const int pw = u0 + kAttnStep * w;
    constexpr int kStride = kAttnStep * kAttnWarps;
#pragma unroll
    for (int k = 0; k < kAttnStages; ++k) {
      const int p = pw + k * kStride;
      const uint32_t n = used_steps + k, st = n % kAttnStages;
      if (ok && p < vis) {
        if (p + kAttnStep > T - a.B) wait_previous();  // the step holds new rows (warp-uniform)
        attn_issue(kh, vh, p, vis, ring + st * kStageBytes, bar0 + 8u * st, pol, lane);
        ++issued_steps;
      }
    }
    wait_previous();  // before the queries are read
    // Q fragments: lane (g, t) holds dimensions 32 i + 8 t .. + 7 (i = 0..3) of head hl of each
    // group; rows g and g + 8 of the MMA are terms (hi, lo) for g < 4, (mid, zero) for g >= 4.
    uint32_t qa[HG][8][4];
#pragma unroll
    for (int grp = 0; grp < HG; ++grp) {
      const int hq = grp * 4 + hl;
      const bool used = hq < G;
      const float* qg = a.q + ((int64_t)b * a.Hq + h * G + (used ? hq : 0)) * kAttnD + 8 * t;
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) {
        float f[8];
        const float4 x0 = __ldg(reinterpret_cast<const float4*>(qg + 32 * ii));
        const float4 x1 = __ldg(reinterpret_cast<const float4*>(qg + 32 * ii + 4));
        f[0] = x0.x; f[1] = x0.y; f[2] = x0.z; f[3] = x0.w; f[4] = x1.x; f[5] = x1.y; f[6] = x1.z; f[7] = x1.w;
        float r0[8], r1[8];  // rows g and g + 8
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float x = __fmul_rn(f[e], a.scale_log2);
          const float hi = bf16_rn(x);
          const float r = __fsub_rn(x, hi);  // exact
          const float mid = bf16_rn(r);
          const float lo = __fsub_rn(r, mid);  // exact; rounded to bf16 by the packing
          r0[e] = !used ? 0.0f : g < 4 ? hi : mid;
          r1[e] = !used || g >= 4 ? 0.0f : lo;
        }
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {  // k-step j = 2 ii + jj uses dims 4 jj .. 4 jj + 3 of the chunk
          const int j = 2 * ii + jj, o = 4 * jj;
          qa[grp][j][0] = pack_bf16(r0[o], r0[o + 1]);
          qa[grp][j][1] = pack_bf16(r1[o], r1[o + 1]);
          qa[grp][j][2] = pack_bf16(r0[o + 2], r0[o + 3]);
          qa[grp][j][3] = pack_bf16(r1[o + 2], r1[o + 3]);
        }
      }
    }
    float O[HG][8][4], mref[HG][4], lsum[HG];
#pragma unroll
    for (int grp = 0; grp < HG; ++grp) {
      lsum[grp] = 0.0f;
#pragma unroll
      for (int k = 0; k < 4; ++k) mref[grp][k] = -INFINITY;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int k = 0; k < 4; ++k) O[grp][mt][k] = 0.0f;
    }

    for (int p0 = pw; ok && p0 < vis; p0 += kStride, ++used_steps) {
      const uint32_t st = used_steps % kAttnStages;
      if (!mbar_wait_bounded(bar0 + 8u * st, (used_steps / kAttnStages) & 1u)) {
        ok = false;  // leave the rest of this position's steps; the result is not valid
        break;
      }
      uint4 kw[2][4], vw[4][2];
      const bool full = p0 + kAttnStep <= vis;
      attn_read(attn_smem + (size_t)w * kAttnStages * kStageBytes + st * kStageBytes, p0, vis, full, g, t, kw, vw);
      attn_compute<G, HG>(qa, O, mref, lsum, kw, vw, p0, vis, full, g, t);
      __syncwarp();  // every lane's reads of the stage are done (their values fed the MMAs)
      const int pn = p0 + kAttnStages * kStride;
      if (pn < vis) {
        attn_issue(kh, vh, pn, vis, ring + st * kStageBytes, bar0 + 8u * st, pol, lane);
        ++issued_steps;
      }
    }
    if (!ok) {  // wait (bounded) for the copies still in flight, then flag the CTA
      for (uint32_t n = used_steps; n < issued_steps; ++n)
        if (!mbar_wait_bounded(bar0 + 8u * (n % kAttnStages), (n / kAttnStages) & 1u)) break;
      used_steps = issued_steps;
    }
    // every warp's ring is idle: it holds Acc from here on; a failed wait anywhere in the CTA
    // marks the unit's result
    const bool fail = __syncthreads_or(!ok);
    // the warp's result: weight sums over the lanes of a head, the two weight terms added
    // (columns 2t, 2t + 1 and 2t + 4, 2t + 5 hold the same heads), into shared memory
#pragma unroll
    for (int grp = 0; grp < HG; ++grp) {
      float ls = lsum[grp];
      ls += __shfl_xor_sync(0xffffffffu, ls, 1);
      ls += __shfl_xor_sync(0xffffffffu, ls, 2);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int k = 0; k < 4; ++k) O[grp][mt][k] += __shfl_xor_sync(0xffffffffu, O[grp][mt][k], 2);
      const int h0 = grp * 4 + 2 * t;  // heads h0, h0 + 1 (lanes t < 2)
      if (t < 2) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          const int d = 64 * (mt >> 2) + 8 * g + 2 * (mt & 3);
          if (h0 < G) *reinterpret_cast<float2*>(&Acc[w][h0][d]) = make_float2(O[grp][mt][0], O[grp][mt][2]);
          if (h0 + 1 < G) *reinterpret_cast<float2*>(&Acc[w][h0 + 1][d]) = make_float2(O[grp][mt][1], O[grp][mt][3]);
        }
      }
      if (t == 0 && g < 4 && grp * 4 + g < G) {
        mw[w][grp * 4 + g] = pick(mref[grp], g);
        lw[w][grp * 4 + g] = ls;
      }
    }
    __syncthreads();
    // the unit's result for position b: warps weighted by 2^(m_w - M)
    float* pb = a.part + ((int64_t)(b * a.Hq + h * G) * a.nch + c) * kPartRow;
#pragma unroll
    for (int k = 0; k < G; ++k) {
      float M = -INFINITY;
#pragma unroll
      for (int ww = 0; ww < kAttnWarps; ++ww) M = fmaxf(M, mw[ww][k]);
      float o = 0.0f, L = 0.0f;
#pragma unroll
      for (int ww = 0; ww < kAttnWarps; ++ww) {
        const float e = mw[ww][k] == -INFINITY ? 0.0f : exp2f(mw[ww][k] - M);
        o = fmaf(Acc[ww][k][i], e, o);
        L = fmaf(lw[ww][k], e, L);
      }
      pb[k * head_stride + i] = o;
      if (i == 0) {
        pb[k * head_stride + kAttnD] = M;
        pb[k * head_stride + kAttnD + 1] = fail ? __int_as_float(0x7fc00000) : L;  // NaN marks a failed unit
      }
    }
    // The last unit of this (b, key-value head) to finish merges all units in one pass: warp w
    // folds units w, w + 4, ... (loads of kMergeU units in flight, lane: dimensions 4 lane ..
    // 4 lane + 3) with a running maximum, then the 4 warps' results are combined.
    __syncthreads();  // the partial is written by every thread
    if (i == 0) s_last = atom_add_acq_rel(&a.done[b * a.Hkv + h], 1u) == (unsigned)(a.nch - 1);
    __syncthreads();
    if (s_last) {
      constexpr int kMergeU = 4;
      const float* pg0 = a.part + (int64_t)(b * a.Hq + h * G) * head_stride;
      float Mr[G], Lr[G];
      float4 Or[G];
#pragma unroll
      for (int k = 0; k < G; ++k) {
        Mr[k] = -INFINITY;
        Lr[k] = 0.0f;
        Or[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      for (int cc0 = w; cc0 < a.nch; cc0 += kAttnWarps * kMergeU) {
        float mc[kMergeU][G], lc[kMergeU][G];
        float4 xc[kMergeU][G];
#pragma unroll
        for (int u = 0; u < kMergeU; ++u) {
          const int cc = cc0 + kAttnWarps * u;
#pragma unroll
          for (int k = 0; k < G; ++k) {
            const float* pc = pg0 + k * head_stride + (int64_t)min(cc, a.nch - 1) * kPartRow;
            mc[u][k] = cc < a.nch ? __ldcg(pc + kAttnD) : -INFINITY;
            lc[u][k] = __ldcg(pc + kAttnD + 1);
            xc[u][k] = __ldcg(reinterpret_cast<const float4*>(pc + 4 * lane));
          }
        }
#pragma unroll
        for (int u = 0; u < kMergeU; ++u)
#pragma unroll
          for (int k = 0; k < G; ++k) {
            if (mc[u][k] == -INFINITY) continue;  // an empty unit (the same in every lane)
            const float mn = fmaxf(Mr[k], mc[u][k]);
            const float sa = exp2f(Mr[k] - mn), sb = exp2f(mc[u][k] - mn);  // sa = 0 while Mr = -inf
            Or[k].x = fmaf(Or[k].x, sa, xc[u][k].x * sb);
            Or[k].y = fmaf(Or[k].y, sa, xc[u][k].y * sb);
            Or[k].z = fmaf(Or[k].z, sa, xc[u][k].z * sb);
            Or[k].w = fmaf(Or[k].w, sa, xc[u][k].w * sb);
            Lr[k] = fmaf(Lr[k], sa, lc[u][k] * sb);
            Mr[k] = mn;
          }
      }
#pragma unroll
      for (int k = 0; k < G; ++k) {
        *reinterpret_cast<float4*>(&Acc[w][k][4 * lane]) = Or[k];
        if (lane == 0) {
          mw[w][k] = Mr[k];
          lw[w][k] = Lr[k];
        }
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < G; ++k) {
        float M = -INFINITY;
#pragma unroll
        for (int ww = 0; ww < kAttnWarps; ++ww) M = fmaxf(M, mw[ww][k]);
        float o = 0.0f, L = 0.0f;
#pragma unroll
        for (int ww = 0; ww < kAttnWarps; ++ww) {
          const float e = mw[ww][k] == -INFINITY ? 0.0f : exp2f(mw[ww][k] - M);
          o = fmaf(Acc[ww][k][i], e, o);
          L = fmaf(lw[ww][k], e, L);
        }
        a.out[(int64_t)(b * a.Hq + h * G + k) * kAttnD + i] = __fdiv_rn(o, L);
      }
      if (i == 0) a.done[b * a.Hkv + h] = 0u;
    }
    __syncthreads();  // shared buffers are reused by the next position
  }
}


// Rotary embedding of head blockIdx.x (query heads, then key-value heads) at position
// pos0 + blockIdx.y, one thread per rotated pair: the angles pos * base^(-2i/D) are formed
// and reduced modulo 2 pi in double precision (a float angle of a large position would carry an
// error of about pos * 2^-24 radians), their sine and cosine taken in fp32, the rotations in fp32
// without contraction. Keys and values go to the cache rows pos0 + b as bf16 (round to nearest
// even); queries to q_out in fp32.
__global__ void __launch_bounds__(kAttnD / 2) rope_append_kernel(
    const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v, int Hq, int Hkv,
    int pos0_arg, const int* pos_dev, double log2_base, float* __restrict__ q_out, uint16_t* __restrict__ kc,
    uint16_t* __restrict__ vc, int ts) {
  dependent_launch_wait();
  const int pos0 = pos_dev ? *pos_dev : pos0_arg;
  const int hh = blockIdx.x, b = blockIdx.y, pos = pos0 + b, j = threadIdx.x;  // pair (j, j + D/2)
  constexpr int half = kAttnD / 2;
  // the angle in double, reduced to [-pi, pi] in double (one fused multiply-add by the double
  // nearest 2 pi: the reduction error is below 1e-11 rad for positions up to 10^6), then sine
  // and cosine in fp32 (FP64 transcendentals are slow on this part)
  const double ang = (double)pos * exp2(-2.0 * j / kAttnD * log2_base);
  const double two_pi = 6.283185307179586;
  const float red = (float)fma(-rint(ang * (1.0 / two_pi)), two_pi, ang);
  float sn, cs;
  sincosf(red, &sn, &cs);
  const bool isq = hh < Hq;
  const float* x = isq ? q + ((int64_t)b * Hq + hh) * kAttnD : k + ((int64_t)b * Hkv + (hh - Hq)) * kAttnD;
  const float lo = x[j], hi = x[j + half];
  const float ylo = __fsub_rn(__fmul_rn(lo, cs), __fmul_rn(hi, sn));
  const float yhi = __fadd_rn(__fmul_rn(hi, cs), __fmul_rn(lo, sn));
  if (isq) {
    float* y = q_out + ((int64_t)b * Hq + hh) * kAttnD;
    y[j] = ylo;
    y[j + half] = yhi;
  } else {
    const int g = hh - Hq;
    uint16_t* row = kc + ((int64_t)g * ts + pos) * kAttnD;
    row[j] = __bfloat16_as_ushort(__float2bfloat16_rn(ylo));
    row[j + half] = __bfloat16_as_ushort(__float2bfloat16_rn(yhi));
    const float* vr = v + ((int64_t)b * Hkv + g) * kAttnD;
    uint16_t* vrow = vc + ((int64_t)g * ts + pos) * kAttnD;
    vrow[j] = __bfloat16_as_ushort(__float2bfloat16_rn(vr[j]));
    vrow[j + half] = __bfloat16_as_ushort(__float2bfloat16_rn(vr[j + half]));
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
nt_status launch_attn_units(const AttnArgs& a, cudaStream_t st, bool pdl) {
  static std::atomic<int> attr_set[64];  // per device: the ring's dynamic shared memory allowed
  int dev = 0;
  NT_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return set_error(NT_ERR_CUDA, "device index out of range");
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    NT_CUDA_TRY(cudaFuncSetAttribute(attn_unit_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRingBytes));
    attr_set[dev].store(1, std::memory_order_release);
  }
  NT_CUDA_TRY(launch_kernel(attn_unit_kernel<G>, dim3(a.nch, a.Hkv), dim3(kAttnThreads), kRingBytes, st, pdl, a));
  return check_launch("attn_unit_kernel");
}

// Positions per unit: one wave of resident CTAs over all key-value heads, whole 16-position
// warp steps, the same number of steps for each of the 4 warps once a unit has more than 4,
// at most kAttnMaxSplit units per head.
int attn_span(int T, int Hkv, int G) {
  const int sms = device_sm_count();
  const int want = std::max(1, attn_resident(G) * sms / Hkv);
  const int steps = (T + kAttnStep - 1) / kAttnStep;
  int per = (steps + want - 1) / want;
  if (per > kAttnWarps) per = (per + kAttnWarps - 1) / kAttnWarps * kAttnWarps;
  while ((steps + per - 1) / per > kAttnMaxSplit) ++per;
  return per * kAttnStep;
}
int attn_units(int T, int Hkv, int G) { const int s = attn_span(T, Hkv, G); return (T + s - 1) / s; }
size_t attn_part_bytes(int B, int Hq, int Hkv, int T) {
  return sizeof(float) * (size_t)B * Hq * attn_units(T, Hkv, Hq / Hkv) * kPartRow;
}

}  // namespace

size_t attention_ws_bytes(int B, int Hq, int Hkv, int T) {
  return attn_part_bytes(B, Hq, Hkv, T) + sizeof(unsigned int) * (size_t)B * Hkv;
}

nt_status launch_attention(const float* q, const uint16_t* kc, const uint16_t* vc, int B, int Hq, int Hkv, int T,
                           int ts, float* out, void* ws, cudaStream_t st, const int* T_dev, bool pdl) {
  float* part = static_cast<float*>(ws);
  unsigned int* done = reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(ws) + attn_part_bytes(B, Hq, Hkv, T));
  const int G = Hq / Hkv;
  AttnArgs a{q, kc, vc, part, done, out, B, Hq, Hkv, T, ts, attn_units(T, Hkv, G), attn_span(T, Hkv, G),
             (float)(1.4426950408889634 / sqrt((double)kAttnD)), T_dev};
  switch (G) {
    case 1: return launch_attn_units<1>(a, st, pdl);
    case 2: return launch_attn_units<2>(a, st, pdl);
    case 4: return launch_attn_units<4>(a, st, pdl);
    default: return launch_attn_units<8>(a, st, pdl);
  }
}

nt_status launch_rope_append(const float* q, const float* k, const float* v, int B, int Hq, int Hkv, int pos0,
                             float base, float* q_out, uint16_t* kc, uint16_t* vc, int ts, cudaStream_t st,
                             const int* pos_dev, bool pdl) {
  NT_CUDA_TRY(launch_kernel(rope_append_kernel, dim3(Hq + Hkv, B), dim3(kAttnD / 2), 0, st, pdl, q, k, v, Hq, Hkv,
                            pos0, pos_dev, log2((double)base), q_out, kc, vc, ts));
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
  if (B < 1 || B > 65535 || Hq < 1 || Hkv < 1 || pos0 < 0 || (int64_t)pos0 + B > t_stride || !(base > 1.0f))
    return set_error(NT_ERR_INVALID_ARG,
                     "need 1 <= B <= 65535, Hq, Hkv >= 1, 0 <= pos0, pos0 + B <= t_stride and base > 1");
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
