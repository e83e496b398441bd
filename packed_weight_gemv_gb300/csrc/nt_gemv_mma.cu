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

#include "nt_kernels.cuh"

namespace nt {
namespace {

constexpr int kMmaWarps = 8;
constexpr int kMmaThreads = 32 * kMmaWarps;
constexpr int kUnitRows = 32;            // rows per warp unit: 8 tiles, one per lane group
constexpr int kUnitsPerWarp = 2;         // units per warp and chunk
constexpr int kUnitsPerCta = kMmaWarps * kUnitsPerWarp;
constexpr int kChunkK = 1024;            // trits of K per CTA
constexpr int kChunkBlocks = kChunkK / 16;  // k16 blocks of the f16 MMA
constexpr int kStepSpans = 8;            // 64-trit spans per load step (a 16-byte load per lane each)
constexpr int kStepK = 64 * kStepSpans;

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

// Unit sums of one chunk into the workspace: lane (g, t) holds, per 16-row tile mt and vector
// tile nt, rows 4 g + 2 mt (+1) of its unit and vectors 8 nt + 2 t (+1).
template <int NT>
__device__ __forceinline__ void flush_unit(float (&c)[2][NT][4], const MmaMat& m, int u, int g, int t) {
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int acc = __float2int_rn(c[mt][nt][e]);
        c[mt][nt][e] = 0.0f;
        const int64_t n = (int64_t)kUnitRows * u + 4 * g + 2 * mt + (e >> 1);
        const int v = 8 * nt + 2 * t + (e & 1);
        if (n < m.N && v < m.B && acc != 0) atomicAdd(m.acc_ws + (int64_t)v * m.N + n, acc);
      }
}

// NT tiles of 8 vectors (B <= 8 NT). Grid: one CTA per (matrix, chunk, group of 16 units).
template <int NT>
__global__ void __launch_bounds__(kMmaThreads, 2) gemv_mma_kernel(const MmaMat* __restrict__ mats, int n_mats,
                                                                 const uint16_t* __restrict__ cta_mat) {
  __shared__ __align__(16) uint2 sB[NT][kChunkBlocks][32];  // per lane: 4 f16 activations
  __shared__ int s_last;
  dependent_launch_wait();
  int lo = 0, hi = n_mats - 1;  // this CTA's matrix: from the table, else the last whose first CTA <= it
  if (cta_mat) {
    lo = __ldg(cta_mat + blockIdx.x);
  } else {
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (mats[mid].cta_begin <= (int64_t)blockIdx.x) lo = mid; else hi = mid - 1;
    }
  }
  const MmaMat m = mats[lo];
  const int li = (int)(blockIdx.x - m.cta_begin);
  const int chunk = li / m.ugroups, ug = li - chunk * m.ugroups;
  const int64_t Kp = padded_k(m.K);
  const int k0 = chunk * kChunkK;
  const int steps = (int)(Kp - k0 < kChunkK ? Kp - k0 : kChunkK) / kStepK;  // 1 or 2 steps per unit

  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int64_t ntiles = padded_rows(m.N) / 4;
  const int ubase = ug * kUnitsPerCta + w;  // the warp's units: ubase + 8 j
  const int rem = m.units32 - ubase;
  const int items = rem <= 0 ? 0 : min(kUnitsPerWarp, (rem + kMmaWarps - 1) / kMmaWarps);
  const int sh = steps == 2 ? 1 : 0;
  const int total = items << sh;  // load steps of this warp: unit s >> sh, half s & (steps - 1)

  // step s: lane (g, t) reads tile 8 u + g at trits k0 + 512 half + 64 sp + 16 t, sp = 0..7
  auto load = [&](uint4 (&b)[kStepSpans], int s) {
    const int64_t T = (int64_t)(kUnitRows / 4) * (ubase + kMmaWarps * (s >> sh)) + g;
    const bool ok = s < total && T < ntiles;
    const uint8_t* p = m.w + T * Kp + k0 + kStepK * (s & (steps - 1)) + 16 * t;
#pragma unroll
    for (int sp = 0; sp < kStepSpans; ++sp) b[sp] = ok ? ld_group(p + 64 * sp) : make_uint4(0u, 0u, 0u, 0u);
  };
  // one chunk's sums stay exact in fp32: |sum| <= 127 * 1024
  float c[2][NT][4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) c[mt][nt][e] = 0.0f;
  auto compute = [&](const uint4 (&b)[kStepSpans], int s) {
    const int half = s & (steps - 1);
#pragma unroll
    for (int sp = 0; sp < kStepSpans; ++sp) {
      uint32_t r0[4], r1[4], r2[4], r3[4];  // tile rows 0..3: trits 4 i .. 4 i + 3 of the group in [i]
      word_hi_bytes(b[sp].x, r0);
      word_hi_bytes(b[sp].y, r1);
      word_hi_bytes(b[sp].z, r2);
      word_hi_bytes(b[sp].w, r3);
#pragma unroll
      for (int i = 0; i < 4; ++i) {  // block i of the span: logical k 2t, 2t + 1 / 2t + 8, 2t + 9 are
        const int blk = (kStepK / 16) * half + 4 * sp + i;  // the lane's trits 4 i, 4 i + 1 / 4 i + 2, 4 i + 3
        const uint32_t a0 = f16x2_lo(r0[i]), a1 = f16x2_lo(r1[i]), a2 = f16x2_hi(r0[i]), a3 = f16x2_hi(r1[i]);
        const uint32_t e0 = f16x2_lo(r2[i]), e1 = f16x2_lo(r3[i]), e2 = f16x2_hi(r2[i]), e3 = f16x2_hi(r3[i]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint2 bv = sB[nt][blk][lane];
          mma_f16(c[0][nt], a0, a1, a2, a3, bv.x, bv.y);
          mma_f16(c[1][nt], e0, e1, e2, e3, bv.x, bv.y);
        }
      }
    }
    if (half == steps - 1) flush_unit<NT>(c, m, ubase + kMmaWarps * (s >> sh), g, t);
  };
  // loads run one step ahead of the decode, across unit boundaries
  uint4 ba[kStepSpans], bb[kStepSpans];
  load(ba, 0);  // in flight while the activations are converted

  // the chunk's activations of every vector as f16 in the B operand's order: 4 bytes k4 of
  // vector v (chunk trits 4 k4 .. 4 k4 + 3) are lane (v % 8, (k4 % 16) / 4)'s operand of block
  // 4 (k4 / 16) + k4 % 4 in vector tile v / 8
#pragma unroll
  for (int r = 0; r < NT * 8 * (kChunkK / 4) / kMmaThreads; ++r) {
    const int e = threadIdx.x + r * kMmaThreads;
    const int v = e / (kChunkK / 4), k4 = e - v * (kChunkK / 4);
    const int k = k0 + 4 * k4;
    uint32_t qv = 0u;
    if (v < m.B && k < m.K) qv = __ldg(reinterpret_cast<const uint32_t*>(m.q + (int64_t)v * m.K + k));
    const int blk = 4 * (k4 >> 4) + (k4 & 3), ln = 4 * (v & 7) + ((k4 & 15) >> 2);
    sB[v >> 3][blk][ln] = f16x4(qv);
  }
  __syncthreads();

#pragma unroll 1
  for (int s = 0; s < total; s += 2) {
    load(bb, s + 1);
    compute(ba, s);
    if (s + 1 < total) {  // the same in every lane
      load(ba, s + 2);
      compute(bb, s + 1);
    }
  }

  // the group's epilogue by the CTA that completes its last chunk
  __threadfence();  // this thread's sums are visible before the group's counter moves
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(m.cnt + ug, 1u) == (unsigned)(m.kchunks - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int64_t n0 = (int64_t)kUnitRows * kUnitsPerCta * ug;
  const int64_t n1 = m.N < n0 + kUnitRows * kUnitsPerCta ? m.N : n0 + kUnitRows * kUnitsPerCta;
  for (int v = 0; v < m.B; ++v)
    for (int64_t n = n0 + threadIdx.x; n < n1; n += kMmaThreads) {
      int32_t* a = m.acc_ws + (int64_t)v * m.N + n;
      const int sum = __ldcg(a);
      m.y[(int64_t)v * m.N + n] = scale_out(sum, __ldg(m.s_w + n), __ldg(m.s_x + v));
      if (m.acc) m.acc[(int64_t)v * m.N + n] = sum;
      *a = 0;
    }
  if (threadIdx.x == 0) m.cnt[ug] = 0u;
}

}  // namespace

// Geometry of one matrix on the tensor-core batched path: its 32-row units, 1,024-trit chunks,
// groups of 32 units and CTAs (one per chunk and group).
void mma_geometry(MmaMat& m) {
  m.units32 = (int)((padded_rows(m.N) + kUnitRows - 1) / kUnitRows);
  m.kchunks = (int)((padded_k(m.K) + kChunkK - 1) / kChunkK);
  m.ugroups = (m.units32 + kUnitsPerCta - 1) / kUnitsPerCta;
}
int64_t mma_ctas(const MmaMat& m) { return (int64_t)m.kchunks * m.ugroups; }
size_t mma_ws_bytes(int64_t rows, int64_t groups, int B) {
  return sizeof(int32_t) * (size_t)(B * rows) + sizeof(unsigned int) * (size_t)groups;
}

nt_status launch_gemv_mma(const MmaMat* d_mats, int n_mats, const uint16_t* d_cta_mat, int64_t total_ctas, int max_B,
                          cudaStream_t st, bool pdl) {
  if (max_B < 1 || max_B > kMmaMaxBatch) return set_error(NT_ERR_INVALID_ARG, "batched tensor-core path: 1 <= B <= 16");
  auto kern = max_B <= 8 ? gemv_mma_kernel<1> : gemv_mma_kernel<2>;
  NT_CUDA_TRY(launch_kernel(kern, dim3((unsigned)total_ctas), dim3(kMmaThreads), 0, st, pdl, d_mats, n_mats, d_cta_mat));
  return check_launch("gemv_mma_kernel");
}

}  // namespace nt
