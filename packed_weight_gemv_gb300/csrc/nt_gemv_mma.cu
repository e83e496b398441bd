// nt_gemv_mma.cu -- batched ternary projections (2..16 activation vectors) on the tensor cores.
//
// With B vectors a byte of packed weights carries 4 * B multiply-adds; dp4a (4 per instruction
// lane, ~61 per SM per clock on this part) runs out of issue slots well below the HBM rate once
// B >= 4. Here the products run as f16 mma.sync m16n8k16 with fp32 sums: a ternary weight is
// exactly an f16 value (+-1 = 0x3C00 / 0xBC00, 0 = 0) and so is every int8 activation, every
// product is an integer and every partial sum of a 1,024-trit chunk stays below 2^17 in
// magnitude, so the fp32 sums are exact and move into int32 once per chunk: the result equals
// the integer dot product bit for bit. (The e4m3 form of mma.sync, with int8 split into two
// digits, was built first: on this part it executes as about 13 instructions per MMA against
// about 1 for f16, which left it issue-bound.)
//
// Decode: two byte permutes per 16-bit half word look the pair codes up in two pools that hold
// the f16 high bytes of +1 / -1 / 0, giving quads (4 trits as 4 high bytes); two more byte
// permutes per quad place its bytes 0, 1 and 2, 3 over zero low bytes as two f16x2 operands.
// The byte-permute (ALU) pipe is the kernel's busiest: about 7.5 of its instructions per MMA.
//
// Work: a CTA of 8 warps takes one 1,024-trit chunk of K and up to 32 units of 32 rows (8
// tiles); it first converts the chunk's activations of all vectors to f16 in shared memory, laid
// out as the MMA's B operand. A lane owns one tile of its warp's unit and reads 16 bytes at a
// time (4 rows x 16 trits), coalesced in 64-byte runs; the tile's rows 0/1 form the rows g / g + 8
// of one 16-row MMA tile and rows 2/3 those of a second, so both share every B fragment. Loads
// run one step (512 trits) ahead in registers, across unit boundaries. A unit's int32 sums of a
// chunk go to an int32 workspace with atomics; the CTA that completes a unit group's last chunk
// applies the fp32 epilogue (as the other paths: fl(fl(acc) * s_w) * s_x) and clears the
// workspace and the group's counter for the next call.
#include <cuda_fp16.h>

#include <atomic>
#include <climits>

#include "nt_kernels.cuh"

namespace nt {
namespace {

constexpr int kMmaWarps = 8;
constexpr int kMmaThreads = 32 * kMmaWarps;
constexpr int kUnitRows = 32;            // rows per warp unit: 8 tiles, one per lane group
constexpr int kUnitsPerCta = kMmaWarps;  // one unit per warp
constexpr int kChunkK = 1024;            // trits of K per shared-memory activation buffer
constexpr int kChunkBlocks = kChunkK / 16;  // k16 blocks of the f16 MMA
constexpr int kStepSpans = 4;            // 64-trit spans per load step (a 16-byte load per lane each)
constexpr int kStepK = 64 * kStepSpans;
constexpr int kStepsPerChunk = kChunkK / kStepK;
// fp32 sums of integers stay exact below 2^24: 127 * 131072 < 2^24 trits of K per part
constexpr int64_t kMaxPartK = 131072;

// f16 pair-code pools: the tiled layout's codes select the high byte of +1 / -1 / 0 as 0x3C /
// 0xBC / 0x00 (the low byte of all three is 0). Code 14 (the pair (0, -1)) reads byte 6 in
// sign-replicate mode: pool A's 0x3C gives 0x00 as wanted, pool B's 0xBC gives 0xFF, which the
// AND with 0xBC turns into 0xBC.
constexpr uint32_t kH16PoolA_lo = 0x00BC3C00u;  // codes 0..3 -> 0, +1, -1, 0
constexpr uint32_t kH16PoolA_hi = 0xBC3CBC3Cu;  // codes 4..7 -> +1, -1, +1, -1
constexpr uint32_t kH16PoolB_lo = 0x3C000000u;  // codes 0..3 -> 0, 0, 0, +1
constexpr uint32_t kH16PoolB_hi = 0xBCBC3C3Cu;  // codes 4..7 -> +1, +1, -1, -1

// One tiled word (16 trits) as the f16 high bytes of trits 0-3, 4-7, 8-11 and 12-15.
__device__ __forceinline__ void word_hi_bytes(uint32_t w, uint32_t (&o)[4]) {
  const uint32_t hi = w >> 16;
  o[0] = prmt(kH16PoolA_lo, kH16PoolA_hi, w);
  o[1] = prmt(kH16PoolB_lo, kH16PoolB_hi, w) & 0xBCBCBCBCu;
  o[2] = prmt(kH16PoolA_lo, kH16PoolA_hi, hi);
  o[3] = prmt(kH16PoolB_lo, kH16PoolB_hi, hi) & 0xBCBCBCBCu;
}
// f16x2 of the high bytes 0, 1 (lo) or 2, 3 (hi) of a quad, low bytes zero.
__device__ __forceinline__ uint32_t f16x2_lo(uint32_t q) { return prmt(q, 0u, 0x1404u); }
__device__ __forceinline__ uint32_t f16x2_hi(uint32_t q) { return prmt(q, 0u, 0x3424u); }

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four int8 values as f16 (exact).
__device__ __forceinline__ uint2 f16x4(uint32_t x) {
  const __half2 lo = __halves2half2(__short2half_rn((short)(int8_t)(x & 0xFFu)), __short2half_rn((short)(int8_t)(x >> 8)));
  const __half2 hi = __halves2half2(__short2half_rn((short)(int8_t)(x >> 16)), __short2half_rn((short)(int8_t)(x >> 24)));
  return make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
}

// One 16-trit group of a tile: its 4 rows' words (streamed once, no L1 allocation).
__device__ __forceinline__ uint4 ld_group(const uint8_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// NT tiles of 8 vectors (B <= 8 NT). Grid: one CTA per (matrix, part of K, group of 8 units);
// a CTA walks its part chunk by chunk with the activations of the next chunk loaded while the
// current one is multiplied. Dynamic shared memory: two activation buffers.
template <int NT>
__global__ void __launch_bounds__(kMmaThreads, 2) gemv_mma_kernel(const MmaMat* __restrict__ mats, int n_mats,
                                                                 const uint16_t* __restrict__ cta_mat, const MmaMat one) {
  extern __shared__ __align__(16) uint2 sB[];  // [2][NT][kChunkBlocks][32]: per lane 4 f16 activations
  __shared__ int s_last;
  dependent_launch_wait();
  int lo = 0, hi = n_mats - 1;  // this CTA's matrix: from the table, else the last whose first CTA <= it
  if (cta_mat) {
    lo = __ldg(cta_mat + blockIdx.x);
  } else if (mats) {
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (mats[mid].cta_begin <= (int64_t)blockIdx.x) lo = mid; else hi = mid - 1;
    }
  }
  const MmaMat m = mats ? mats[lo] : one;  // a single matrix comes by value
  const int li = (int)(blockIdx.x - m.cta_begin);
  const int part = li / m.ugroups, ug = li - part * m.ugroups;
  const int64_t Kp = padded_k(m.K);
  const int c0 = part * m.cpp;                                // first chunk of the part
  const int nch = (m.kchunks - c0 < m.cpp ? m.kchunks - c0 : m.cpp);
  const int64_t tail = Kp - (int64_t)(c0 + nch - 1) * kChunkK;  // trits from the part's last chunk on
  const int last_steps = tail < kChunkK ? (int)(tail / kStepK) : kStepsPerChunk;  // 2 or 4

  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int u = ug * kUnitsPerCta + w;  // this warp's unit
  const int64_t T = (int64_t)(kUnitRows / 4) * u + g;  // this lane's tile
  const bool active = u < m.units32, okT = active && T < padded_rows(m.N) / 4;
  const int total = active ? (nch - 1) * kStepsPerChunk + last_steps : 0;  // even
  const uint8_t* wp = m.w + T * Kp + (int64_t)c0 * kChunkK + 16 * t;  // dereferenced only when okT

  // step s: trits c0 * 1024 + 256 s + 64 sp + 16 t .. + 15 of the tile's 4 rows, sp = 0..3
  auto load = [&](uint4 (&b)[kStepSpans], int s) {
    const bool ok = okT && s < total;
    const uint8_t* p = wp + (int64_t)kStepK * s;
#pragma unroll
    for (int sp = 0; sp < kStepSpans; ++sp) b[sp] = ok ? ld_group(p + 64 * sp) : make_uint4(0u, 0u, 0u, 0u);
  };
  // sums over the whole part stay exact in fp32: |sum| <= 127 * kMaxPartK < 2^24
  float c[2][NT][4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) c[mt][nt][e] = 0.0f;
  auto compute = [&](const uint4 (&b)[kStepSpans], int s, const uint2* sb) {
    const int sc = s & (kStepsPerChunk - 1);  // step within the chunk
#pragma unroll
    for (int sp = 0; sp < kStepSpans; ++sp) {
      uint32_t r0[4], r1[4], r2[4], r3[4];  // tile rows 0..3: trits 4 i .. 4 i + 3 of the group in [i]
      word_hi_bytes(b[sp].x, r0);
      word_hi_bytes(b[sp].y, r1);
      word_hi_bytes(b[sp].z, r2);
      word_hi_bytes(b[sp].w, r3);
#pragma unroll
      for (int i = 0; i < 4; ++i) {  // block i of the span: logical k 2t, 2t + 1 / 2t + 8, 2t + 9 are
        const int blk = (kStepK / 16) * sc + 4 * sp + i;  // the lane's trits 4 i, 4 i + 1 / 4 i + 2, 4 i + 3
        const uint32_t a0 = f16x2_lo(r0[i]), a1 = f16x2_lo(r1[i]), a2 = f16x2_hi(r0[i]), a3 = f16x2_hi(r1[i]);
        const uint32_t e0 = f16x2_lo(r2[i]), e1 = f16x2_lo(r3[i]), e2 = f16x2_hi(r2[i]), e3 = f16x2_hi(r3[i]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint2 bv = sb[(nt * kChunkBlocks + blk) * 32 + lane];
          mma_f16(c[0][nt], a0, a1, a2, a3, bv.x, bv.y);
          mma_f16(c[1][nt], e0, e1, e2, e3, bv.x, bv.y);
        }
      }
    }
  };

  // a chunk's activations of every vector as f16 in the B operand's order: 4 bytes k4 of vector
  // v (chunk trits 4 k4 .. 4 k4 + 3) are lane (v % 8, (k4 % 16) / 4)'s operand of block
  // 4 (k4 / 16) + k4 % 4 in vector tile v / 8
  constexpr int kActPerThread = NT * 8 * (kChunkK / 4) / kMmaThreads;
  uint32_t act[kActPerThread];
  auto fetch_act = [&](int chunk) {
#pragma unroll
    for (int r = 0; r < kActPerThread; ++r) {
      const int e = threadIdx.x + r * kMmaThreads;
      const int v = e / (kChunkK / 4), k = chunk * kChunkK + 4 * (e - v * (kChunkK / 4));
      act[r] = (v < m.B && k < m.K) ? __ldg(reinterpret_cast<const uint32_t*>(m.q + (int64_t)v * m.K + k)) : 0u;
    }
  };
  auto store_act = [&](int buf) {
#pragma unroll
    for (int r = 0; r < kActPerThread; ++r) {
      const int e = threadIdx.x + r * kMmaThreads;
      const int v = e / (kChunkK / 4), k4 = e - v * (kChunkK / 4);
      const int blk = 4 * (k4 >> 4) + (k4 & 3), ln = 4 * (v & 7) + ((k4 & 15) >> 2);
      sB[((buf * NT + (v >> 3)) * kChunkBlocks + blk) * 32 + ln] = f16x4(act[r]);
    }
  };

  // weight loads run one step ahead of the decode, across chunk boundaries
  uint4 ba[kStepSpans], bb[kStepSpans];
  load(ba, 0);
  fetch_act(c0);
  store_act(0);
  __syncthreads();
  int s = 0;
#pragma unroll 1
  for (int ci = 0; ci < nch; ++ci) {
    if (ci + 1 < nch) fetch_act(c0 + ci + 1);  // in flight during this chunk
    const uint2* sb = sB + (ci & 1) * NT * kChunkBlocks * 32;
    const int s_end = total < (ci + 1) * kStepsPerChunk ? total : (ci + 1) * kStepsPerChunk;
#pragma unroll 1
    for (; s < s_end; s += 2) {  // every chunk has an even number of steps
      load(bb, s + 1);
      compute(ba, s, sb);
      load(ba, s + 2);
      compute(bb, s + 1, sb);
    }
    if (ci + 1 < nch) store_act((ci + 1) & 1);  // the other buffer: its last readers passed the barrier below
    __syncthreads();
  }

  // lane (g, t) holds, per 16-row tile mt and vector tile nt, rows 4 g + 2 mt (+1) of its unit
  // and vectors 8 nt + 2 t (+1)
  if (m.nparts == 1) {  // the whole of K: the epilogue straight from the sums
    if (!active) return;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int64_t n = (int64_t)kUnitRows * u + 4 * g + 2 * mt + (e >> 1);
          const int v = 8 * nt + 2 * t + (e & 1);
          if (n >= m.N || v >= m.B) continue;
          const int sum = __float2int_rn(c[mt][nt][e]);
          m.y[(int64_t)v * m.N + n] = scale_out(sum, __ldg(m.s_w + n), __ldg(m.s_x + v));
          if (m.acc) m.acc[(int64_t)v * m.N + n] = sum;
        }
    return;
  }

  // K split over parts: partial sums into the int32 workspace; the CTA that completes a
  // group's last part applies the epilogue and clears the workspace and the counter
  if (active) {
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int sum = __float2int_rn(c[mt][nt][e]);
          const int64_t n = (int64_t)kUnitRows * u + 4 * g + 2 * mt + (e >> 1);
          const int v = 8 * nt + 2 * t + (e & 1);
          if (n < m.N && v < m.B && sum != 0) atomicAdd(m.acc_ws + (int64_t)v * m.N + n, sum);
        }
  }
  __threadfence();  // this thread's sums are visible before the group's counter moves
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(m.cnt + ug, 1u) == (unsigned)(m.nparts - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int64_t n = (int64_t)kUnitRows * kUnitsPerCta * ug + threadIdx.x;  // one row per thread
  static_assert(kUnitRows * kUnitsPerCta == kMmaThreads, "one row of the group per thread");
  if (n < m.N) {
    const float sw = __ldg(m.s_w + n);
    for (int v = 0; v < m.B; ++v) {
      int32_t* a = m.acc_ws + (int64_t)v * m.N + n;
      const int sum = __ldcg(a);
      m.y[(int64_t)v * m.N + n] = scale_out(sum, sw, __ldg(m.s_x + v));
      if (m.acc) m.acc[(int64_t)v * m.N + n] = sum;
      *a = 0;
    }
  }
  if (threadIdx.x == 0) m.cnt[ug] = 0u;
}

// ---------------------------------------------------------------------------------------
// Output projection (int8 table T [V][K] times int8 activations) for 2..16 vectors on the
// same f16 MMA: four table bytes become two f16x2 operands exactly (1024 + 128 + x, less 1152);
// a product is at most 127 * 128 in magnitude, so fp32 sums of a 1,024-element chunk stay
// exact and move into int32 registers once per chunk. A warp takes 32 rows of T (one 16-byte
// load per lane and row per 64-element span), a CTA 256 rows over the whole of K with the
// activations double-buffered per chunk as above; logits and each vector's arg-max (the largest
// logit, the lowest row on ties) follow from the int32 sums, the CTAs' arg-max candidates meet
// in the workspace and the last CTA to finish picks the winners.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t f16x2_sub(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;\n" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// int8 bytes 0, 1 (lo) and 2, 3 (hi) of x as f16x2 (exact)
__device__ __forceinline__ void i8x4_f16(uint32_t x, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = x ^ 0x80808080u;                         // x + 128 as unsigned bytes
  lo = f16x2_sub(prmt(u, 0x64646464u, 0x4140u), 0x64806480u);  // (1024 + u) - 1152
  hi = f16x2_sub(prmt(u, 0x64646464u, 0x4342u), 0x64806480u);
}
// 16 bytes global -> shared without registers (zero-filled when !ok); per-thread groups
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool ok) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src), "r"(ok ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }
// ring stages (64-element spans of 32 rows, 2 KB) per warp: with the activation buffers two
// CTAs fit an SM (8 warps x 4 x 2 KB + 32 KB; 8 x 3 x 2 KB + 64 KB)
constexpr int head_stages(int nt) { return nt == 1 ? 4 : 3; }
constexpr size_t head_smem(int nt) {
  return sizeof(uint2) * 2 * nt * kChunkBlocks * 32 + sizeof(uint4) * kMmaWarps * head_stages(nt) * 4 * 32;
}

__device__ __forceinline__ bool head_better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

template <int NT>
__global__ void __launch_bounds__(kMmaThreads, 2) head_mma_kernel(
    const int8_t* __restrict__ T, const float* __restrict__ s_T, int V, int K, const int8_t* __restrict__ q,
    const float* __restrict__ s_x, int B, float* __restrict__ logits, int32_t* __restrict__ argmax,
    HeadWs* __restrict__ ws) {
  extern __shared__ __align__(16) uint2 sB[];  // [2][NT][kChunkBlocks][32], then the warps' rings
  constexpr int kS = head_stages(NT);
  uint4* ring = reinterpret_cast<uint4*>(sB + 2 * NT * kChunkBlocks * 32) + (threadIdx.x >> 5) * kS * 4 * 32;
  // [kMmaWarps][8 NT] arg-max candidates, over the rings once every copy has landed
  HeadPartial* wbest = reinterpret_cast<HeadPartial*>(sB + 2 * NT * kChunkBlocks * 32);
  __shared__ int s_last;
  dependent_launch_wait();
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int kchunks = (K + kChunkK - 1) / kChunkK, nspans = (K + 63) / 64;
  const int groups = (V + kUnitRows * kUnitsPerCta - 1) / (kUnitRows * kUnitsPerCta);
  constexpr int kActPerThread = NT * 8 * (kChunkK / 4) / kMmaThreads;
  uint32_t act[kActPerThread];
  auto fetch_act = [&](int chunk) {
#pragma unroll
    for (int r = 0; r < kActPerThread; ++r) {
      const int e = threadIdx.x + r * kMmaThreads;
      const int v = e / (kChunkK / 4), k = chunk * kChunkK + 4 * (e - v * (kChunkK / 4));
      act[r] = (v < B && k < K) ? __ldg(reinterpret_cast<const uint32_t*>(q + (int64_t)v * K + k)) : 0u;
    }
  };
  auto store_act = [&](int buf) {
#pragma unroll
    for (int r = 0; r < kActPerThread; ++r) {
      const int e = threadIdx.x + r * kMmaThreads;
      const int v = e / (kChunkK / 4), k4 = e - v * (kChunkK / 4);
      const int blk = 4 * (k4 >> 4) + (k4 & 3), ln = 4 * (v & 7) + ((k4 & 15) >> 2);
      sB[((buf * NT + (v >> 3)) * kChunkBlocks + blk) * 32 + ln] = f16x4(act[r]);
    }
  };
  // running arg-max of this lane: vectors 8 nt + 2 t + j
  float bv[NT][2];
  int bi[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) { bv[nt][j] = -INFINITY; bi[nt][j] = INT_MAX; }

#pragma unroll 1
  for (int grp = blockIdx.x; grp < groups; grp += gridDim.x) {
    const int64_t r0 = (int64_t)kUnitRows * (kUnitsPerCta * (int64_t)grp + w) + g;  // rows r0 + 8 j
    float c[2][NT][4];
    int acc[2][NT][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) { c[mt][nt][e] = 0.0f; acc[mt][nt][e] = 0; }
    auto compute = [&](const uint4 (&b)[4], int s, const uint2* sb) {
      const uint32_t* w0 = reinterpret_cast<const uint32_t*>(&b[0]);
      const uint32_t* w1 = reinterpret_cast<const uint32_t*>(&b[1]);
      const uint32_t* w2 = reinterpret_cast<const uint32_t*>(&b[2]);
      const uint32_t* w3 = reinterpret_cast<const uint32_t*>(&b[3]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {  // block i: the lane's elements 16 t + 4 i .. + 3 of the span
        const int blk = 4 * (s & 15) + i;
        uint32_t a0, a1, a2, a3, e0, e1, e2, e3;
        i8x4_f16(w0[i], a0, a2);
        i8x4_f16(w1[i], a1, a3);
        i8x4_f16(w2[i], e0, e2);
        i8x4_f16(w3[i], e1, e3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint2 bb = sb[(nt * kChunkBlocks + blk) * 32 + lane];
          mma_f16(c[0][nt], a0, a1, a2, a3, bb.x, bb.y);
          mma_f16(c[1][nt], e0, e1, e2, e3, bb.x, bb.y);
        }
      }
    };
    // span s (16 elements k = 64 s + 16 t of rows r0 + 8 j, j = 0..3) streams into ring slot
    // s % S of this lane's own region, S - 1 spans ahead of the decode (zero-filled past K or V)
    auto issue = [&](int s) {
      uint4* slot = ring + (s % kS) * 4 * 32 + lane;
      const int k = 64 * s + 16 * t;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t r = r0 + 8 * j;
        const bool ok = s < nspans && k < K && r < V;
        cp_async16(slot + 32 * j, ok ? T + r * K + k : T, ok);
      }
      cp_async_commit();
    };
#pragma unroll
    for (int s = 0; s < kS - 1; ++s) issue(s);
    fetch_act(0);
    store_act(0);  // the buffer's last readers passed the previous group's final barrier
    __syncthreads();
    int s = 0;
#pragma unroll 1
    for (int ci = 0; ci < kchunks; ++ci) {
      if (ci + 1 < kchunks) fetch_act(ci + 1);  // in flight during this chunk
      const uint2* sb = sB + (ci & 1) * NT * kChunkBlocks * 32;
      const int s_end = nspans < 16 * (ci + 1) ? nspans : 16 * (ci + 1);
#pragma unroll 1
      for (; s < s_end; ++s) {
        issue(s + kS - 1);
        cp_async_wait<kS - 1>();  // span s has landed (this lane's own copies)
        const uint4* slot = ring + (s % kS) * 4 * 32 + lane;
        uint4 b[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) b[j] = slot[32 * j];
        compute(b, s, sb);
      }
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {  // the chunk's exact fp32 sums into int32
            acc[mt][nt][e] += __float2int_rn(c[mt][nt][e]);
            c[mt][nt][e] = 0.0f;
          }
      if (ci + 1 < kchunks) store_act((ci + 1) & 1);
      __syncthreads();
    }
    cp_async_wait<0>();  // the zero-filled copies past the end
    __syncthreads();     // every warp's ring is idle (the arg-max candidates reuse it)
    // lane (g, t) holds rows r0 + 8 (2 mt + e / 2) and vectors 8 nt + 2 t + e % 2
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int64_t n = r0 + 8 * (2 * mt + (e >> 1));
          const int v = 8 * nt + 2 * t + (e & 1);
          if (n >= V || v >= B) continue;
          const float lg = scale_out(acc[mt][nt][e], __ldg(s_T + n), __ldg(s_x + v));
          if (logits) logits[(int64_t)v * V + n] = lg;
          if (head_better(lg, (int)n, bv[nt][e & 1], bi[nt][e & 1])) { bv[nt][e & 1] = lg; bi[nt][e & 1] = (int)n; }
        }
  }

  // arg-max candidates: lanes of one t over the 8 row groups, then the CTA's warps
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv[nt][j], o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi[nt][j], o);
        if (head_better(ov, oi, bv[nt][j], bi[nt][j])) { bv[nt][j] = ov; bi[nt][j] = oi; }
      }
      if (g == 0) wbest[w * 8 * NT + 8 * nt + 2 * t + j] = HeadPartial{bv[nt][j], bi[nt][j]};
    }
  __syncthreads();
  if (threadIdx.x < B) {
    HeadPartial best = wbest[threadIdx.x];
    for (int i = 1; i < kMmaWarps; ++i) {
      const HeadPartial o = wbest[i * 8 * NT + threadIdx.x];
      if (head_better(o.val, o.idx, best.val, best.idx)) best = o;
    }
    ws->part[(int64_t)blockIdx.x * B + threadIdx.x] = best;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(&ws->done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int b = w; b < B; b += kMmaWarps) {
    float best_v = -INFINITY;
    int best_i = INT_MAX;
    for (int i = lane; i < (int)gridDim.x; i += 32) {
      const HeadPartial* pp = &ws->part[(int64_t)i * B + b];
      const float pv = __ldcg(&pp->val);
      const int pi = __ldcg(&pp->idx);
      if (head_better(pv, pi, best_v, best_i)) { best_v = pv; best_i = pi; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best_v, o);
      const int oi = __shfl_xor_sync(0xffffffffu, best_i, o);
      if (head_better(ov, oi, best_v, best_i)) { best_v = ov; best_i = oi; }
    }
    if (lane == 0) argmax[b] = best_i == INT_MAX ? 0 : best_i;
  }
  if (threadIdx.x == 0) ws->done = 0u;
}

}  // namespace

// Geometry of one matrix on the tensor-core batched path: its 32-row units, 1,024-trit chunks,
// groups of 8 units, and K in `parts` parts (at least enough that every part's fp32 sums stay
// exact; at most one per chunk). CTAs: one per part and group.
void mma_geometry(MmaMat& m, int parts) {
  const int64_t Kp = padded_k(m.K);
  m.units32 = (int)((padded_rows(m.N) + kUnitRows - 1) / kUnitRows);
  m.kchunks = (int)((Kp + kChunkK - 1) / kChunkK);
  m.ugroups = (m.units32 + kUnitsPerCta - 1) / kUnitsPerCta;
  const int64_t need = (Kp + kMaxPartK - 1) / kMaxPartK;
  int64_t p = parts > need ? parts : need;
  if (p > m.kchunks) p = m.kchunks;
  m.cpp = (int)((m.kchunks + p - 1) / p);
  m.nparts = (m.kchunks + m.cpp - 1) / m.cpp;
}
int64_t mma_ctas(const MmaMat& m) { return (int64_t)m.nparts * m.ugroups; }
size_t mma_ws_bytes(int64_t rows, int64_t groups, int B) {
  return sizeof(int32_t) * (size_t)(B * rows) + sizeof(unsigned int) * (size_t)groups;
}

// dynamic shared memory of gemv_mma_kernel<nt>: two activation buffers of 16 KB per vector tile
static size_t gemv_smem_bytes(int nt) { return sizeof(uint2) * 2 * nt * kChunkBlocks * 32; }
static nt_status gemv_mma_attrs() {
  static std::atomic<int> attr_set[64];  // per device: the buffers allowed for both tile counts
  int dev = 0;
  NT_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return set_error(NT_ERR_CUDA, "device index out of range");
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    NT_CUDA_TRY(cudaFuncSetAttribute(gemv_mma_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gemv_smem_bytes(1)));
    NT_CUDA_TRY(cudaFuncSetAttribute(gemv_mma_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gemv_smem_bytes(2)));
    attr_set[dev].store(1, std::memory_order_release);
  }
  return NT_OK;
}

nt_status launch_gemv_mma(const MmaMat* d_mats, int n_mats, const uint16_t* d_cta_mat, int64_t total_ctas, int max_B,
                          cudaStream_t st, bool pdl) {
  if (max_B < 1 || max_B > kMmaMaxBatch) return set_error(NT_ERR_INVALID_ARG, "batched tensor-core path: 1 <= B <= 16");
  const int nt = max_B <= 8 ? 1 : 2;
  NT_TRY(gemv_mma_attrs());
  auto kern = nt == 1 ? gemv_mma_kernel<1> : gemv_mma_kernel<2>;
  NT_CUDA_TRY(launch_kernel(kern, dim3((unsigned)total_ctas), dim3(kMmaThreads), gemv_smem_bytes(nt), st, pdl, d_mats,
                            n_mats, d_cta_mat, MmaMat{}));
  return check_launch("gemv_mma_kernel");
}

// One matrix per call (nt_ternary_gemm): the descriptor goes by value; K is split until the
// call has 8 waves of CTAs (or one chunk per part), the parts meeting in the caller's workspace.
size_t mma_single_ws_bytes(int N, int K, int B) {
  MmaMat m{};
  m.N = N;
  m.K = K;
  mma_geometry(m, 1);
  return kWsHeaderBytes + ((mma_ws_bytes(N, m.ugroups, B) + 15) & ~(size_t)15);  // status header first
}
nt_status launch_gemv_mma_single(const uint8_t* w, const float* s_w, int N, int K, const int8_t* q, const float* s_x,
                                 int B, float* y, int32_t* acc, void* ws, cudaStream_t st) {
  if (B < kMmaMinBatch || B > kMmaMaxBatch) return set_error(NT_ERR_INVALID_ARG, "batched tensor-core path: 2 <= B <= 16");
  MmaMat m{};
  m.w = w;
  m.s_w = s_w;
  m.q = q;
  m.s_x = s_x;
  m.y = y;
  m.acc = acc;
  m.N = N;
  m.K = K;
  m.B = B;
  mma_geometry(m, 1);
  for (int parts = 2; mma_ctas(m) < 8LL * device_sm_count() && parts <= 2 * m.kchunks; parts *= 2) mma_geometry(m, parts);
  m.acc_ws = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + kWsHeaderBytes);  // after the status header
  m.cnt = reinterpret_cast<unsigned int*>(m.acc_ws + (size_t)B * N);
  m.cta_begin = 0;
  const int nt = B <= 8 ? 1 : 2;
  NT_TRY(gemv_mma_attrs());
  auto kern = nt == 1 ? gemv_mma_kernel<1> : gemv_mma_kernel<2>;
  NT_CUDA_TRY(launch_kernel(kern, dim3((unsigned)mma_ctas(m)), dim3(kMmaThreads), gemv_smem_bytes(nt), st, false,
                            (const MmaMat*)nullptr, 0, (const uint16_t*)nullptr, m));
  return check_launch("gemv_mma_kernel");
}

nt_status launch_head_mma(const int8_t* T, const float* s_T, int V, int K, const int8_t* q, const float* s_x,
                          int B, float* logits, int32_t* argmax, HeadWs* ws, cudaStream_t st) {
  if (B < kMmaMinBatch || B > kMmaMaxBatch) return set_error(NT_ERR_INVALID_ARG, "tensor-core output projection: 2 <= B <= 16");
  const int nt = B <= 8 ? 1 : 2;
  const size_t smem = head_smem(nt);
  static std::atomic<int> attr_set[64];
  int dev = 0;
  NT_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return set_error(NT_ERR_CUDA, "device index out of range");
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    NT_CUDA_TRY(cudaFuncSetAttribute(head_mma_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)head_smem(1)));
    NT_CUDA_TRY(cudaFuncSetAttribute(head_mma_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)head_smem(2)));
    attr_set[dev].store(1, std::memory_order_release);
  }
  const int64_t groups = ((int64_t)V + kUnitRows * kUnitsPerCta - 1) / (kUnitRows * kUnitsPerCta);
  const int grid = (int)(groups < kHeadMaxCtas ? groups : kHeadMaxCtas);
  auto kern = nt == 1 ? head_mma_kernel<1> : head_mma_kernel<2>;
  NT_CUDA_TRY(launch_kernel(kern, dim3(grid), dim3(kMmaThreads), smem, st, false, T, s_T, V, K, q, s_x, B, logits,
                            argmax, ws));
  return check_launch("head_mma_kernel");
}

}  // namespace nt
