// nt_gemv_tc8.cu -- batched ternary projections (2..16 activation vectors) on the 5th-generation
// tensor cores: tcgen05.mma kind::f8f6f4 with the decoded weights in tensor memory.
//
// A trit is exactly an e4m3 value (+1 = 0x38, -1 = 0xB8, 0 = 0) and an int8 activation code
// q is exactly 16 h + l with h = q >> 4 in [-8, 7] and l = q & 15 in [0, 15], both exact e4m3
// integers. The MMA therefore multiplies the weights (M side: 128 rows per CTA) with 2 B digit
// rows (N side, 16 or 32 with zero padding) and the fp32 sums of one digit row are integers of
// magnitude at most 15 K, exact below 2^24; the epilogue forms acc = 16 D_h + D_l in int32,
// bit for bit the integer dot product.
//
// Why the tensor memory: the decode (two byte permutes and one AND per 8 trits, against seven
// instructions for the f16 form of the older mma.sync) writes each row's e4m3 bytes straight
// into that row's tensor-memory lane with tcgen05.st, so the weights never pass through the
// shared-memory port a second time.
//
// Used by nt_ternary_gemm with a workspace (one matrix, gemv_tc8_kernel) and by independent
// decode plans on the graph / stream launchers (every matrix of the step in one launch,
// gemv_tc8_multi_kernel, after one launch that writes every matrix's digit rows).
//
// CTA (192 threads), one 128-row tile of the weights over a range of K ("part"):
//   warp 4 lane 0  -- TMA producer: per 128-trit K-block one 2-D box of the tiled weights
//                     (32 tiles x 128 bytes, 128-byte swizzle) and one box of the digit rows
//                     (N x 128 bytes) into a ring of 4 stages (full / empty mbarriers);
//   warps 0-3      -- decoders, one thread per weight row (tensor-memory lane = row): 8
//                     shared loads of its row's words per K-block (conflict-free thanks to the
//                     swizzle), decode to 32 e4m3 bytes, tcgen05.st into the A buffer once the
//                     previous block's MMAs have read it;
//   warp 5 lane 0  -- MMA issuer: 4 x tcgen05.mma (M 128, N 16/32, K 32) per K-block, commits
//                     release the stage and the A buffer;
//   epilogue       -- the decoders read the accumulator (tcgen05.ld), then y = fl(fl(acc) s_w) s_x
//                     straight (one part) or int32 partial sums to a workspace whose last part
//                     applies it (several parts, K split for small calls).
// Every wait is bounded (2 s); after a timeout the CTA stops issuing work, waits (bounded) for
// its own MMAs and frees its tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <mutex>
#include <vector>
#include <string>

#include "nt_kernels.cuh"

namespace nt {
namespace {

constexpr int kTc8Tiles = 32;                  // tiles (4 rows) per CTA: 128 weight rows (MMA M)
constexpr int kTc8KB = 128;                    // trits per K-block = bytes of one tile's block
// ring stages: few, so that more CTAs share an SM (measured: 4 stages, 64 tensor-memory columns
// and 56 registers per thread run six CTAs per SM and beat 8 stages with four)
constexpr int tc8_stages(int nn) { return nn <= 16 ? 4 : 4; }
constexpr int kTc8WBytes = kTc8Tiles * kTc8KB;  // weight box: 4 KB
constexpr int kTc8Threads = 192;
constexpr int kTc8MinBlocks = 6;               // CTAs per SM: registers capped at 56 (no spills)
constexpr int kTc8Decoders = 128;
constexpr int kTc8TmemCols = 64;               // D at column 0 (<= 32), the A buffer at 32
constexpr int kTc8ABufs = 1;                   // the decode of the next block overlaps the MMA
constexpr uint64_t kTc8TimeoutNs = 2000000000ull;
constexpr int64_t kTc8MaxPartK = 131072;       // |D| <= 15 K < 2^24
constexpr unsigned int kTc8ErrWait = 16;        // status code of a wait that ran out

// e4m3 pools of the pair codes: the same pools as the dp4a decode with +1 -> 0x38, -1 -> 0xB8.
// Code 14 (the pair (0, -1)) reads byte 6 in sign-replicate mode: 0x38 -> 0x00 in pool A,
// 0xB8 -> 0xFF in pool B, which the AND with 0xB8 turns into 0xB8.
constexpr uint32_t kE4PoolA_lo = 0x00B83800u;  // codes 0..3 -> 0, +1, -1, 0
constexpr uint32_t kE4PoolA_hi = 0xB838B838u;  // codes 4..7 -> +1, -1, +1, -1
constexpr uint32_t kE4PoolB_lo = 0x38000000u;  // codes 0..3 -> 0, 0, 0, +1
constexpr uint32_t kE4PoolB_hi = 0xB8B83838u;  // codes 4..7 -> +1, +1, -1, -1

__device__ __forceinline__ uint32_t s_u32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ void bar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void bar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool bar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// The same test, the thread suspended (up to 0.1 ms) until the phase completes.
__device__ __forceinline__ bool bar_try_sleep(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(100000u)
      : "memory");
  return ok != 0;
}
// Bounded wait; false after the timeout or once another role of the CTA has given up.
__device__ bool bar_wait(uint32_t bar, uint32_t parity, volatile int* fail, uint64_t timeout_ns) {
  if (bar_try(bar, parity)) return true;
  const uint64_t deadline = globaltimer_ns() + timeout_ns;
  for (;;) {
    if (bar_try_sleep(bar, parity)) return true;
    if (*fail || globaltimer_ns() > deadline) {
      *fail = 1;
      return false;
    }
  }
}
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// K-major operand in shared memory with the 128-byte swizzle (as the TMA writes it): rows of
// 128 bytes, 8-row groups 1,024 bytes apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;  // stride byte offset: 8-row group pitch
  d |= (uint64_t)1 << 46;                          // descriptor version
  d |= (uint64_t)2 << 61;                          // 128-byte swizzle
  return d;
}
// kind::f8f6f4, A = B = e4m3, D = fp32, K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_e4m3(int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

struct Tc8Params {
  const float* s_w;  // [N]
  const float* s_x;  // [B]
  float* y;          // [B][N]
  int32_t* acc;      // [B][N] or null
  int32_t* acc_ws;   // [B][N] partial sums (several parts), zero between calls
  unsigned int* cnt; // [mtiles] parts finished, zero between calls
  int N, B;
  int mtiles;        // 128-row tiles
  int kblocks;       // 128-trit blocks of padded K
  int kb_per_part, nparts;
  unsigned int* err;  // status word [code, CTA]: a decode plan's, or the call's workspace header
  uint64_t timeout_ns;  // bound on every wait
  int fault;           // tests of the timeout path: the producer issues no copies
};
struct Tc8Mat {
  CUtensorMap tmW;   // the tiles, box 128 bytes x 32 tiles
  CUtensorMap tmD;   // the digit rows, box 128 bytes x NN rows
  Tc8Params p;
  int64_t cta_begin;  // first CTA of this matrix in its launch
};

// One CTA's work: 128-row tile `cta % mtiles` over K part `cta / mtiles` of the matrix whose
// maps and parameters are given (kernel parameters for one call, global memory for a plan).
template <int NN>
__device__ __forceinline__ void tc8_cta(const CUtensorMap* tmW_, const CUtensorMap* tmD_, const Tc8Params& p, int cta,
                                        bool global_maps) {
  const CUtensorMap& tmW = *tmW_;
  const CUtensorMap& tmD = *tmD_;
  constexpr int kTc8Stages = tc8_stages(NN);
  constexpr int kStageBytes = kTc8WBytes + NN * kTc8KB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kTc8Stages * kStageBytes);
  const uint32_t full0 = s_u32(bars), empty0 = full0 + 8 * kTc8Stages;
  const uint32_t afull0 = empty0 + 8 * kTc8Stages, aempty0 = afull0 + 8 * kTc8ABufs, dfull = aempty0 + 8 * kTc8ABufs;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kTc8Stages + 2 * kTc8ABufs + 1);
  volatile int* fail = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_last = reinterpret_cast<int*>(tmem_slot + 2);

  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int mtile = cta % p.mtiles, part = cta / p.mtiles;
  const int kb0 = part * p.kb_per_part;
  const int nkb = (p.kblocks - kb0 < p.kb_per_part) ? p.kblocks - kb0 : p.kb_per_part;

  dependent_launch_wait();
  if (t == 0) {
    for (int s = 0; s < kTc8Stages; ++s) {
      bar_init(full0 + 8 * s, 1);
      bar_init(empty0 + 8 * s, kTc8Decoders + 1);  // the decoders' reads and the MMAs' commit
    }
    for (int b = 0; b < kTc8ABufs; ++b) {
      bar_init(afull0 + 8 * b, kTc8Decoders);
      bar_init(aempty0 + 8 * b, 1);
    }
    bar_init(dfull, 1);
    *fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 4) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(s_u32(tmem_slot)),
                 "r"(kTc8TmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ---- TMA producer: weight box and digit box of every K-block of the part ----
    if (lane == 0 && !p.fault) {
      if (global_maps) {  // maps written to global memory before the launch: make them visible to the TMA
        asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(tmW_) : "memory");
        asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(tmD_) : "memory");
      }
      for (int i = 0; i < nkb; ++i) {
        const int s = i % kTc8Stages;
        if (i >= kTc8Stages && !bar_wait(empty0 + 8 * s, ((i / kTc8Stages) - 1) & 1u, fail, p.timeout_ns)) break;
        uint8_t* st = smem + s * kStageBytes;
        bar_expect_tx(full0 + 8 * s, kStageBytes);
        const int x = (kb0 + i) * kTc8KB;  // byte (= trit) offset within a tile, a multiple of 128
        tma_2d(s_u32(st), &tmW, x, mtile * kTc8Tiles, full0 + 8 * s);
        tma_2d(s_u32(st + kTc8WBytes), &tmD, x, 0, full0 + 8 * s);
      }
    }
  } else if (warp == 5) {
    // ---- MMA issuer ----
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3(NN);
      for (int i = 0; i < nkb; ++i) {
        const int s = i % kTc8Stages, b = i % kTc8ABufs;
        if (!bar_wait(full0 + 8 * s, (i / kTc8Stages) & 1u, fail, p.timeout_ns)) break;
        if (!bar_wait(afull0 + 8 * b, (i / kTc8ABufs) & 1u, fail, p.timeout_ns)) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t bsm = s_u32(smem + s * kStageBytes + kTc8WBytes);
#pragma unroll
        for (int kk = 0; kk < kTc8KB / 32; ++kk) {
          const uint32_t a_tmem = tmem + 32u + 32u * (uint32_t)b + 8u * (uint32_t)kk;  // 8 columns = 32 e4m3
          asm volatile(
              "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
              " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}\n" ::"r"(tmem),
              "r"(a_tmem), "l"(desc_sw128(bsm + 32u * (uint32_t)kk)), "r"(idesc), "r"((uint32_t)((i | kk) != 0))
              : "memory");
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(empty0 + 8 * s)
                     : "memory");
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(aempty0 + 8 * b)
                     : "memory");
      }
      // the accumulator is final once every MMA issued above has completed (also after a failure)
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(dfull) : "memory");
    }
  } else {
    // ---- decoders: thread = weight row = tensor-memory lane ----
    const int row = 32 * warp + lane;
    const int T = row >> 2, j = row & 3;  // tile within the CTA's 32, row within the tile
    const uint32_t tl = tmem + ((uint32_t)(32 * warp) << 16);
    for (int i = 0; i < nkb; ++i) {
      const int s = i % kTc8Stages, b = i % kTc8ABufs;
      if (!bar_wait(full0 + 8 * s, (i / kTc8Stages) & 1u, fail, p.timeout_ns)) break;
      // the row's 8 words of the K-block: 16-byte chunk g of box row T sits at chunk g ^ (T % 8)
      const uint8_t* ws = smem + s * kStageBytes + T * kTc8KB + 4 * j;
      uint32_t w[8];
#pragma unroll
      for (int g = 0; g < 8; ++g) w[g] = *reinterpret_cast<const uint32_t*>(ws + ((g ^ (T & 7)) << 4));
      bar_arrive(empty0 + 8 * s);  // release: the reads above are ordered before it
      if (i >= kTc8ABufs && !bar_wait(aempty0 + 8 * b, ((i / kTc8ABufs) - 1) & 1u, fail, p.timeout_ns)) break;
      // e4m3 bytes of the block's trits 16 g .. 16 g + 15 into columns 4 g .. 4 g + 3 of the A buffer
      // two words (8 columns) per store: fewer store instructions than one per word, while
      // wider stores (16 or 32 columns) ran slower (they keep more registers live)
#pragma unroll
      for (int g = 0; g < 8; g += 2) {
        uint32_t r[8];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const uint32_t ww = w[g + j], hi = ww >> 16;
          r[4 * j + 0] = prmt(kE4PoolA_lo, kE4PoolA_hi, ww);
          r[4 * j + 1] = prmt(kE4PoolB_lo, kE4PoolB_hi, ww) & 0xB8B8B8B8u;
          r[4 * j + 2] = prmt(kE4PoolA_lo, kE4PoolA_hi, hi);
          r[4 * j + 3] = prmt(kE4PoolB_lo, kE4PoolB_hi, hi) & 0xB8B8B8B8u;
        }
        asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
                         tl + 32u + 32u * (uint32_t)b + 4u * (uint32_t)g),
                     "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                     : "memory");
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      bar_arrive(afull0 + 8 * b);
    }

    // ---- epilogue: wait for every issued MMA (bounded, also after a failure) ----
    bool drained = false;
    {
      const uint64_t deadline = globaltimer_ns() + kTc8TimeoutNs;
      for (uint32_t it = 0;; ++it) {
        if (bar_try(dfull, 0)) { drained = true; break; }
        if ((it & 255u) == 255u && globaltimer_ns() > deadline) break;
      }
    }
    if (!drained) *fail = 1;
    if (!*fail) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      uint32_t d[NN];
      if constexpr (NN == 16) {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
            : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3]), "=r"(d[4]), "=r"(d[5]), "=r"(d[6]), "=r"(d[7]),
              "=r"(d[8]), "=r"(d[9]), "=r"(d[10]), "=r"(d[11]), "=r"(d[12]), "=r"(d[13]), "=r"(d[14]), "=r"(d[15])
            : "r"(tl));
      } else {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
            "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
            : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3]), "=r"(d[4]), "=r"(d[5]), "=r"(d[6]), "=r"(d[7]),
              "=r"(d[8]), "=r"(d[9]), "=r"(d[10]), "=r"(d[11]), "=r"(d[12]), "=r"(d[13]), "=r"(d[14]), "=r"(d[15]),
              "=r"(d[16]), "=r"(d[17]), "=r"(d[18]), "=r"(d[19]), "=r"(d[20]), "=r"(d[21]), "=r"(d[22]),
              "=r"(d[23]), "=r"(d[24]), "=r"(d[25]), "=r"(d[26]), "=r"(d[27]), "=r"(d[28]), "=r"(d[29]),
              "=r"(d[30]), "=r"(d[31])
            : "r"(tl));
      }
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      const int64_t n = (int64_t)mtile * (4 * kTc8Tiles) + row;
      if (n < p.N) {
        const float sw = p.nparts == 1 ? __ldg(p.s_w + n) : 0.0f;
#pragma unroll
        for (int v = 0; v < NN / 2; ++v) {
          if (v >= p.B) break;
          // digit rows 2v (h) and 2v + 1 (l): exact integers in fp32
          const int sum = 16 * __float2int_rn(__uint_as_float(d[2 * v])) + __float2int_rn(__uint_as_float(d[2 * v + 1]));
          if (p.nparts == 1) {
            p.y[(int64_t)v * p.N + n] = scale_out(sum, sw, __ldg(p.s_x + v));
            if (p.acc) p.acc[(int64_t)v * p.N + n] = sum;
          } else if (sum != 0) {
            atomicAdd(p.acc_ws + (int64_t)v * p.N + n, sum);
          }
        }
      }
      __threadfence();  // this thread's partial sums are visible before the tile's counter moves
    }
  }

  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 4)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTc8TmemCols) : "memory");
  if (t == 0 && *fail && p.err && atomicCAS(p.err, 0u, kTc8ErrWait) == 0u) p.err[1] = blockIdx.x;
  if (p.nparts == 1 || *fail) return;
  // K split: the CTA that completes a tile's last part applies the epilogue and clears
  if (t == 0) *s_last = atomicAdd(p.cnt + mtile, 1u) == (unsigned)(p.nparts - 1);
  __syncthreads();
  if (!*s_last) return;
  __threadfence();
  if (t < 4 * kTc8Tiles) {
    const int64_t n = (int64_t)mtile * (4 * kTc8Tiles) + t;
    if (n < p.N) {
      const float sw = __ldg(p.s_w + n);
      for (int v = 0; v < p.B; ++v) {
        int32_t* a = p.acc_ws + (int64_t)v * p.N + n;
        const int sum = __ldcg(a);
        p.y[(int64_t)v * p.N + n] = scale_out(sum, sw, __ldg(p.s_x + v));
        if (p.acc) p.acc[(int64_t)v * p.N + n] = sum;
        *a = 0;
      }
    }
  }
  if (t == 0) p.cnt[mtile] = 0u;
}

template <int NN>
__global__ void __launch_bounds__(kTc8Threads, kTc8MinBlocks)
    gemv_tc8_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmD, const Tc8Params p) {
  tc8_cta<NN>(&tmW, &tmD, p, (int)blockIdx.x, false);
}

// Several matrices in one launch (a decode plan's stage): CTA -> matrix from the table; the
// matrices' tensor maps live in global memory (written before the plan's first launch).
template <int NN>
__global__ void __launch_bounds__(kTc8Threads, kTc8MinBlocks)
    gemv_tc8_multi_kernel(const Tc8Mat* __restrict__ mats, const uint16_t* __restrict__ cta_mat) {
  const Tc8Mat* m = mats + __ldg(cta_mat + blockIdx.x);
  const Tc8Params p = m->p;
  tc8_cta<NN>(&m->tmW, &m->tmD, p, (int)(blockIdx.x - m->cta_begin), true);
}

// e4m3 codes of the integers 0..15 (2^(e-7) (1 + m/8)); a negative digit sets bit 7
__constant__ uint8_t kE4Int[16] = {0x00, 0x38, 0x40, 0x44, 0x48, 0x4A, 0x4C, 0x4E,
                                   0x50, 0x51, 0x52, 0x53, 0x54, 0x55, 0x56, 0x57};

// Digit rows of the activations: row 2 v is h = q >> 4, row 2 v + 1 is l = q & 15 of vector v,
// as e4m3 bytes, K padded with zeros to Kd; rows of vectors >= B are zero.
__device__ __forceinline__ void tc8_digits_range(const int8_t* __restrict__ q, int B, int K, int Kd, int NN,
                                                 uint8_t* __restrict__ out, int64_t first, int64_t stride) {
  const int64_t n4 = (int64_t)NN * Kd / 4;
  for (int64_t i = first; i < n4; i += stride) {
    const int64_t e = 4 * i;
    const int n = (int)(e / Kd), k = (int)(e - (int64_t)n * Kd);
    const int v = n >> 1, hi = (n & 1) == 0;
    uint32_t o = 0;
    if (v < B && k < K) {
      const uint32_t x = __ldg(reinterpret_cast<const uint32_t*>(q + (int64_t)v * K + k));
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int c = (int8_t)(x >> (8 * b));
        const int dgt = hi ? (c >> 4) : (c & 15);
        const uint32_t code = dgt < 0 ? (0x80u | kE4Int[-dgt]) : kE4Int[dgt];
        o |= code << (8 * b);
      }
    }
    *reinterpret_cast<uint32_t*>(out + e) = o;
  }
}
__global__ void __launch_bounds__(256) tc8_digits_kernel(const int8_t* __restrict__ q, int B, int K, int Kd, int NN,
                                                         uint8_t* __restrict__ out) {
  dependent_launch_wait();
  tc8_digits_range(q, B, K, Kd, NN, out, blockIdx.x * (int64_t)blockDim.x + threadIdx.x,
                   (int64_t)gridDim.x * blockDim.x);
}
// one job per matrix of a plan (blockIdx.y)
struct Tc8DigitJob {
  const int8_t* q;
  uint8_t* out;
  int B, K, Kd, NN;
};
__global__ void __launch_bounds__(256) tc8_digits_multi_kernel(const Tc8DigitJob* __restrict__ jobs) {
  dependent_launch_wait();
  const Tc8DigitJob j = jobs[blockIdx.y];
  tc8_digits_range(j.q, j.B, j.K, j.Kd, j.NN, j.out, blockIdx.x * (int64_t)blockDim.x + threadIdx.x,
                   (int64_t)gridDim.x * blockDim.x);
}

// ---- host ----------------------------------------------------------------------------
std::mutex g_tc8_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_tc8_encode = nullptr;
bool g_tc8_attr[64] = {};

constexpr int tc8_nn(int B) { return B <= 8 ? 16 : 32; }
constexpr size_t tc8_smem(int nn) { return (size_t)tc8_stages(nn) * (kTc8WBytes + nn * kTc8KB) + 1024 + 256; }
int64_t tc8_kd(int K) { return ((int64_t)K + kTc8KB - 1) / kTc8KB * kTc8KB; }
int64_t tc8_mtiles(int N) { return (padded_rows(N) / 4 + kTc8Tiles - 1) / kTc8Tiles; }

nt_status tc8_setup(int dev) {
  std::lock_guard<std::mutex> lock(g_tc8_mu);
  if (!g_tc8_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult qr;
    NT_CUDA_TRY(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr));
    if (qr != cudaDriverEntryPointSuccess || !fn) return set_error(NT_ERR_CUDA, "cuTensorMapEncodeTiled not available");
    g_tc8_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  if (dev >= 0 && dev < 64 && !g_tc8_attr[dev]) {
    NT_CUDA_TRY(cudaFuncSetAttribute(gemv_tc8_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc8_smem(16)));
    NT_CUDA_TRY(cudaFuncSetAttribute(gemv_tc8_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc8_smem(32)));
    NT_CUDA_TRY(cudaFuncSetAttribute(gemv_tc8_multi_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)tc8_smem(16)));
    NT_CUDA_TRY(cudaFuncSetAttribute(gemv_tc8_multi_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)tc8_smem(32)));
    g_tc8_attr[dev] = true;
  }
  return NT_OK;
}

// 2-D uint8 map over [rows][width] bytes (row pitch = width), box 128 x box_rows, 128-byte swizzle
nt_status tc8_map(CUtensorMap* map, const void* base, int64_t rows, int64_t width, int box_rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)width};
  const cuuint32_t box[2] = {(cuuint32_t)kTc8KB, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_tc8_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(NT_ERR_CUDA, "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")");
  return NT_OK;
}

}  // namespace

bool tc8_supported(int N, int K, int B) {
  return B >= kMmaMinBatch && B <= kMmaMaxBatch && padded_rows(N) / 4 >= kTc8Tiles && K >= 16 && K % 16 == 0;
}

// workspace: the status header (kWsHeaderBytes), digit rows [NN][Kd], then int32 partial sums
// [B][N], then one counter per 128-row tile
size_t tc8_ws_bytes(int N, int K, int B) {
  const size_t digits = (size_t)tc8_nn(B) * (size_t)tc8_kd(K);
  return kWsHeaderBytes +
         ((digits + sizeof(int32_t) * (size_t)B * N + sizeof(unsigned int) * (size_t)tc8_mtiles(N) + 15) & ~(size_t)15);
}

// Maps and parameters of one matrix: K in `parts` parts (at least enough for exact fp32
// sums, at most one per K-block); digits: its digit rows [nn][Kd]; acc_ws / cnt: partial sums
// [B][N] and one counter per 128-row tile (used when K is split).
static nt_status tc8_matrix(const uint8_t* w, const float* s_w, int N, int K, const float* s_x, int B, float* y,
                            int32_t* acc, uint8_t* digits, int32_t* acc_ws, unsigned int* cnt, int64_t parts,
                            Tc8Mat* m) {
  const int nn = tc8_nn(B);
  const int64_t Kd = tc8_kd(K), Kp = padded_k(K);
  NT_TRY(tc8_map(&m->tmW, w, padded_rows(N) / 4, Kp, kTc8Tiles));
  NT_TRY(tc8_map(&m->tmD, digits, nn, Kd, nn));
  Tc8Params& p = m->p;
  p = Tc8Params{};
  p.s_w = s_w;
  p.s_x = s_x;
  p.y = y;
  p.acc = acc;
  p.acc_ws = acc_ws;
  p.cnt = cnt;
  p.N = N;
  p.B = B;
  p.mtiles = (int)tc8_mtiles(N);
  p.kblocks = (int)(Kp / kTc8KB);
  p.timeout_ns = kTc8TimeoutNs;
  parts = std::max<int64_t>(parts, (Kp + kTc8MaxPartK - 1) / kTc8MaxPartK);
  parts = std::min<int64_t>(parts, p.kblocks);
  p.kb_per_part = (int)((p.kblocks + parts - 1) / parts);
  p.nparts = (p.kblocks + p.kb_per_part - 1) / p.kb_per_part;
  return NT_OK;
}
// K parts for a launch of `mtiles` row tiles: doubled while there are fewer than eight CTAs per
// SM (six are resident) and every part keeps at least 8 K-blocks.
static int64_t tc8_parts(int64_t mtiles, int64_t min_kblocks) {
  int64_t parts = 1;
  while (mtiles * parts < 8LL * device_sm_count() && parts * 2 * 8 <= min_kblocks) parts *= 2;
  return parts;
}

nt_status launch_gemv_tc8(const uint8_t* w, const float* s_w, int N, int K, const int8_t* q, const float* s_x, int B,
                          float* y, int32_t* acc, void* ws, cudaStream_t st) {
  if (!tc8_supported(N, K, B)) return set_error(NT_ERR_INVALID_ARG, "tcgen05 batched path: 2 <= B <= 16, N >= 128");
  int dev = 0;
  NT_CUDA_TRY(cudaGetDevice(&dev));
  NT_TRY(tc8_setup(dev));
  const int nn = tc8_nn(B);
  const int64_t Kd = tc8_kd(K), mtiles = tc8_mtiles(N);
  uint8_t* digits = static_cast<uint8_t*>(ws) + kWsHeaderBytes;
  int32_t* acc_ws = reinterpret_cast<int32_t*>(digits + (size_t)nn * Kd);
  unsigned int* cnt = reinterpret_cast<unsigned int*>(acc_ws + (size_t)B * N);
  {
    const int64_t n4 = nn * Kd / 4;
    const int grid = (int)std::min<int64_t>((n4 + 255) / 256, 4LL * device_sm_count());
    NT_CUDA_TRY(launch_kernel(tc8_digits_kernel, dim3(grid), dim3(256), 0, st, false, q, B, K, (int)Kd, nn, digits));
  }
  Tc8Mat m;
  NT_TRY(tc8_matrix(w, s_w, N, K, s_x, B, y, acc, digits, acc_ws, cnt, tc8_parts(mtiles, padded_k(K) / kTc8KB), &m));
  m.p.err = static_cast<unsigned int*>(ws);  // the workspace's status header
  m.p.timeout_ns = test_fault_timeout_ns(kTc8TimeoutNs);
  m.p.fault = test_fault() == kFaultTc8;
  const dim3 grid((unsigned)(mtiles * m.p.nparts));
  if (nn == 16)
    NT_CUDA_TRY(launch_kernel(gemv_tc8_kernel<16>, grid, dim3(kTc8Threads), tc8_smem(16), st, true, m.tmW, m.tmD, m.p));
  else
    NT_CUDA_TRY(launch_kernel(gemv_tc8_kernel<32>, grid, dim3(kTc8Threads), tc8_smem(32), st, true, m.tmW, m.tmD, m.p));
  return check_launch("gemv_tc8_kernel");
}

// ---- decode plans: all matrices of one stage in one launch ----------------------------
bool tc8_plan_supported(const MatDesc* mats, int n, int B) {
  if (n < 1 || n > 65535) return false;
  for (int i = 0; i < n; ++i)
    if (!tc8_supported(mats[i].N, mats[i].K, B) || mats[i].B != B) return false;
  return true;
}

nt_status tc8_plan_create(const MatDesc* mats, int n, int B, unsigned int* err, uint64_t timeout_ns, int fault,
                          Tc8Plan* t) {
  *t = Tc8Plan{};
  int dev = 0;
  NT_CUDA_TRY(cudaGetDevice(&dev));
  NT_TRY(tc8_setup(dev));
  const int nn = tc8_nn(B);
  size_t digit_bytes = 0, ws_bytes = 0;
  int64_t mtiles = 0, min_kb = INT64_MAX, max_n4 = 0;
  for (int i = 0; i < n; ++i) {
    digit_bytes += (size_t)nn * tc8_kd(mats[i].K);
    ws_bytes += sizeof(int32_t) * (size_t)B * mats[i].N + sizeof(unsigned int) * (size_t)tc8_mtiles(mats[i].N);
    mtiles += tc8_mtiles(mats[i].N);
    min_kb = std::min<int64_t>(min_kb, padded_k(mats[i].K) / kTc8KB);
    max_n4 = std::max<int64_t>(max_n4, nn * tc8_kd(mats[i].K) / 4);
  }
  const size_t total = ((digit_bytes + 15) & ~(size_t)15) + ws_bytes;
  cudaError_t e;
  if ((e = cudaMalloc(&t->d_buf, total)) != cudaSuccess) return set_error(NT_ERR_CUDA, std::string("cudaMalloc: ") + cudaGetErrorString(e));
  if ((e = cudaMemset(t->d_buf, 0, total)) != cudaSuccess) return set_error(NT_ERR_CUDA, std::string("cudaMemset: ") + cudaGetErrorString(e));
  uint8_t* digits = static_cast<uint8_t*>(t->d_buf);
  uint8_t* ws = digits + ((digit_bytes + 15) & ~(size_t)15);
  const int64_t parts = tc8_parts(mtiles, min_kb);
  std::vector<Tc8Mat> mm(n);
  std::vector<Tc8DigitJob> jobs(n);
  std::vector<uint16_t> tab;
  int64_t ctas = 0;
  for (int i = 0; i < n; ++i) {
    const MatDesc& d = mats[i];
    int32_t* acc_ws = reinterpret_cast<int32_t*>(ws);
    unsigned int* cnt = reinterpret_cast<unsigned int*>(acc_ws + (size_t)B * d.N);
    ws = reinterpret_cast<uint8_t*>(cnt + tc8_mtiles(d.N));
    NT_TRY(tc8_matrix(d.w, d.s_w, d.N, d.K, d.s_x, B, d.y, d.acc, digits, acc_ws, cnt, parts, &mm[i]));
    mm[i].p.err = err;
    mm[i].p.timeout_ns = timeout_ns;
    mm[i].p.fault = fault;
    mm[i].cta_begin = ctas;
    const int64_t c = (int64_t)mm[i].p.mtiles * mm[i].p.nparts;
    ctas += c;
    tab.insert(tab.end(), (size_t)c, (uint16_t)i);
    jobs[i] = Tc8DigitJob{d.q, digits, B, d.K, (int)tc8_kd(d.K), nn};
    digits += (size_t)nn * tc8_kd(d.K);
  }
  if (ctas > INT32_MAX) return set_error(NT_ERR_INVALID_ARG, "tcgen05 batched path: too many row tiles in one stage");
  if ((e = cudaMalloc(&t->d_mats, sizeof(Tc8Mat) * n)) != cudaSuccess ||
      (e = cudaMemcpy(t->d_mats, mm.data(), sizeof(Tc8Mat) * n, cudaMemcpyHostToDevice)) != cudaSuccess ||
      (e = cudaMalloc(&t->d_tab, sizeof(uint16_t) * tab.size())) != cudaSuccess ||
      (e = cudaMemcpy(t->d_tab, tab.data(), sizeof(uint16_t) * tab.size(), cudaMemcpyHostToDevice)) != cudaSuccess ||
      (e = cudaMalloc(&t->d_jobs, sizeof(Tc8DigitJob) * n)) != cudaSuccess ||
      (e = cudaMemcpy(t->d_jobs, jobs.data(), sizeof(Tc8DigitJob) * n, cudaMemcpyHostToDevice)) != cudaSuccess)
    return set_error(NT_ERR_CUDA, std::string("tcgen05 plan setup: ") + cudaGetErrorString(e));
  t->n = n;
  t->nn = nn;
  t->ctas = ctas;
  t->buf_bytes = total;
  t->digit_grid = (int)std::min<int64_t>((max_n4 + 255) / 256, 64);
  return NT_OK;
}

nt_status tc8_plan_launch(const Tc8Plan& t, cudaStream_t st, bool pdl) {
  NT_CUDA_TRY(launch_kernel(tc8_digits_multi_kernel, dim3(t.digit_grid, t.n), dim3(256), 0, st, pdl,
                            static_cast<const Tc8DigitJob*>(t.d_jobs)));
  const Tc8Mat* mats = static_cast<const Tc8Mat*>(t.d_mats);
  if (t.nn == 16)
    NT_CUDA_TRY(launch_kernel(gemv_tc8_multi_kernel<16>, dim3((unsigned)t.ctas), dim3(kTc8Threads), tc8_smem(16), st,
                              true, mats, (const uint16_t*)t.d_tab));
  else
    NT_CUDA_TRY(launch_kernel(gemv_tc8_multi_kernel<32>, dim3((unsigned)t.ctas), dim3(kTc8Threads), tc8_smem(32), st,
                              true, mats, (const uint16_t*)t.d_tab));
  return check_launch("gemv_tc8_multi_kernel");
}

void tc8_plan_destroy(Tc8Plan* t) {
  cudaFree(t->d_mats);
  cudaFree(t->d_tab);
  cudaFree(t->d_jobs);
  cudaFree(t->d_buf);
  *t = Tc8Plan{};
}

}  // namespace nt
