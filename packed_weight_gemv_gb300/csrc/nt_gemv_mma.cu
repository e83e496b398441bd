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
// Work: a warp takes 4 (16-row unit, 1,024-trit chunk) items, a CTA 32 units of one chunk. The
// CTA converts the chunk's activations of all vectors to f16 in shared memory, laid out as the
// MMA's B operand; each lane then reads the packed words of its two rows straight from the
// tiled layout (two 4-byte words per 64 trits, coalesced in 64-byte runs), decodes them with
// the pair-code pools into the f16 high bytes and spreads those into the A operand. Partial
// int32 sums of a chunk go to an int32 workspace with atomics; the warp that completes a
// unit's last chunk applies the fp32 epilogue (as the other paths: fl(fl(acc) * s_w) * s_x)
// and clears the workspace and its counter for the next call.
#include <cuda_fp16.h>

#include "nt_kernels.cuh"

namespace nt {
namespace {

constexpr int kMmaWarps = 8;
constexpr int kMmaThreads = 32 * kMmaWarps;
constexpr int kUnitsPerWarp = 4;         // 16-row units per warp and chunk
constexpr int kUnitsPerCta = kMmaWarps * kUnitsPerWarp;
constexpr int kChunkK = 1024;            // trits per work item
constexpr int kChunkBlocks = kChunkK / 16;  // k16 blocks of the f16 MMA

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

__device__ __forceinline__ uint32_t ld_word(const uint8_t* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];\n" : "=r"(v) : "l"(p));
  return v;
}

// NT tiles of 8 vectors (B <= 8 NT). Grid: one CTA per (matrix, chunk, 32 units).
template <int NT>
__global__ void __launch_bounds__(kMmaThreads) gemv_mma_kernel(const MmaMat* __restrict__ mats, int n_mats,
                                                              const uint16_t* __restrict__ cta_mat) {
  __shared__ __align__(16) uint2 sB[NT][kChunkBlocks][32];  // per lane: 4 f16 activations
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
  const int spans = (int)(Kp - k0 < kChunkK ? Kp - k0 : kChunkK) / 64;  // 8 or 16 spans of 64 trits

  // the chunk's activations of every vector as f16 in the B operand's order: 4 bytes k4 of
  // vector v (chunk trits 4 k4 .. 4 k4 + 3) are lane (v % 8, (k4 % 16) / 4)'s operand of block
  // 4 (k4 / 16) + k4 % 4 in vector tile v / 8
  for (int e = threadIdx.x; e < NT * 8 * (kChunkK / 4); e += kMmaThreads) {
    const int v = e / (kChunkK / 4), k4 = e - v * (kChunkK / 4);
    const int k = k0 + 4 * k4;
    uint32_t qv = 0u;
    if (v < m.B && k < m.K) qv = __ldg(reinterpret_cast<const uint32_t*>(m.q + (int64_t)v * m.K + k));
    const int blk = 4 * (k4 >> 4) + (k4 & 3), ln = 4 * (v & 7) + ((k4 & 15) >> 2);
    sB[v >> 3][blk][ln] = f16x4(qv);
  }
  __syncthreads();

  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int64_t ntiles = padded_rows(m.N) / 4;
#pragma unroll 1
  for (int j = 0; j < kUnitsPerWarp; ++j) {
    const int u = ug * kUnitsPerCta + j * kMmaWarps + w;
    if (u >= m.units16) return;
    const int64_t T0 = 4 * (int64_t)u + (g >> 2), T1 = T0 + 2;  // tiles of rows g and g + 8
    const uint8_t* r0 = m.w + T0 * Kp + 4 * (g & 3);
    const uint8_t* r1 = m.w + T1 * Kp + 4 * (g & 3);
    const bool ok0 = T0 < ntiles, ok1 = T1 < ntiles;

    // every load of the chunk first: span s, lane t: the 16 trits k0 + 64 s + 16 t .. of each row
    uint32_t w0[16], w1[16];
#pragma unroll
    for (int s = 0; s < 16; ++s) {
      const int64_t off = (int64_t)(k0 + 64 * s + 16 * t);  // a multiple of 16: the word's group
      w0[s] = (s < spans && ok0) ? ld_word(r0 + off) : 0u;
      w1[s] = (s < spans && ok1) ? ld_word(r1 + off) : 0u;
    }
    // one chunk's sums stay exact in fp32: |sum| <= 127 * 1024
    float c[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) c[nt][e] = 0.0f;
#pragma unroll
    for (int s = 0; s < 16; ++s) {
      if (s < spans) {  // the same in every lane
        uint32_t a[4], b[4];
        word_hi_bytes(w0[s], a);  // row g: trits 16 t + 4 i .. + 3 of the span in a[i]
        word_hi_bytes(w1[s], b);  // row g + 8
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // block 4 s + i: logical k 2t, 2t + 1 / 2t + 8, 2t + 9 are
          const int blk = 4 * s + i;   // the lane's trits 4 i, 4 i + 1 / 4 i + 2, 4 i + 3
          const uint32_t a0 = f16x2_lo(a[i]), a1 = f16x2_lo(b[i]), a2 = f16x2_hi(a[i]), a3 = f16x2_hi(b[i]);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const uint2 bv = sB[nt][blk][lane];
            mma_f16(c[nt], a0, a1, a2, a3, bv.x, bv.y);
          }
        }
      }
    }

    // the chunk's sums: lane (g, t) holds rows g, g + 8 x vectors 2t, 2t + 1 of each tile
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int acc = __float2int_rn(c[nt][e]);
        const int64_t n = 16 * (int64_t)u + g + 8 * (e >> 1);
        const int v = 8 * nt + 2 * t + (e & 1);
        if (n < m.N && v < m.B && acc != 0) atomicAdd(m.acc_ws + (int64_t)v * m.N + n, acc);
      }
    __syncwarp();
    unsigned int last = 0;
    if (lane == 0) {
      __threadfence();  // this warp's sums are visible before the unit's counter moves
      last = atomicAdd(m.cnt + u, 1u) == (unsigned)(m.kchunks - 1);
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) {
      __threadfence();
      for (int i = lane; i < 16 * m.B; i += 32) {  // the unit's epilogue, then clear for the next call
        const int64_t n = 16 * (int64_t)u + (i & 15);
        const int v = i >> 4;
        if (n >= m.N) continue;
        int32_t* a = m.acc_ws + (int64_t)v * m.N + n;
        const int total = __ldcg(a);
        m.y[(int64_t)v * m.N + n] = scale_out(total, __ldg(m.s_w + n), __ldg(m.s_x + v));
        if (m.acc) m.acc[(int64_t)v * m.N + n] = total;
        *a = 0;
      }
      if (lane == 0) m.cnt[u] = 0u;
    }
  }
}

}  // namespace

// Geometry of one matrix on the tensor-core batched path: its 16-row units, 1,024-trit chunks
// and CTAs (32 units of one chunk each).
void mma_geometry(MmaMat& m) {
  m.units16 = (int)((padded_rows(m.N) + 15) / 16);
  m.kchunks = (int)((padded_k(m.K) + kChunkK - 1) / kChunkK);
  m.ugroups = (m.units16 + kUnitsPerCta - 1) / kUnitsPerCta;
}
int64_t mma_ctas(const MmaMat& m) { return (int64_t)m.kchunks * m.ugroups; }
size_t mma_ws_bytes(int64_t rows, int64_t units16, int B) {
  return sizeof(int32_t) * (size_t)(B * rows) + sizeof(unsigned int) * (size_t)units16;
}

nt_status launch_gemv_mma(const MmaMat* d_mats, int n_mats, const uint16_t* d_cta_mat, int64_t total_ctas, int max_B,
                          cudaStream_t st, bool pdl) {
  if (max_B < 1 || max_B > kMmaMaxBatch) return set_error(NT_ERR_INVALID_ARG, "batched tensor-core path: 1 <= B <= 16");
  auto kern = max_B <= 8 ? gemv_mma_kernel<1> : gemv_mma_kernel<2>;
  NT_CUDA_TRY(launch_kernel(kern, dim3((unsigned)total_ctas), dim3(kMmaThreads), 0, st, pdl, d_mats, n_mats, d_cta_mat));
  return check_launch("gemv_mma_kernel");
}

}  // namespace nt
