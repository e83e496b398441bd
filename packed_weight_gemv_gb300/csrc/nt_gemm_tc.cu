// nt_gemm_tc.cu -- ternary projection of many activation vectors (prefill-shaped batches) on
// the 5th-generation tensor cores, reading the packed trits directly.
//
// Y[m][n] = fl(fl(acc[m][n] * s_w[n]) * s_x[m]),  acc = sum_k q[m][k] * t[n][k].
// Prefill pushes thousands of tokens through the same weights, so the work is a dense
// contraction (the MLxcel page measures prefill as compute-bound); batch-1 decode stays on
// the streaming kernels. This part has no int8 tensor-core MMA (ptxas rejects
// tcgen05.mma .kind::i8 for sm_103a), so the contraction runs on kind::f16.
//
// Exactness: ternary weights and int8 activations are exact in f16, each product is an
// integer of magnitude <= 127, and every partial sum stays below 127 * K < 2^24 for
// K <= 131072, so the fp32 accumulator in tensor memory holds the exact integer sum; the
// epilogue applies the same two rounded products as every other path.
//
// A call runs two kernels:
//   1. the activations as f16 [M][K] (once for every matrix of the call) into the caller's
//      workspace -- the weights stay in their packed tiled form, no copy of them is made;
//      both kernels are programmatic dependent launches;
//   2. a persistent GEMM over the tiles of all matrices, one CTA per SM, looping over tiles of
//      128 weight rows (MMA M) x TN tokens (MMA N; TN <= 224 picked per call so the tiles fill
//      whole waves of SMs):
//        warp 12 lane 0: per 64-trit K step, a 2-D TMA load of the 32 packed weight tiles
//          (32 x 64 bytes; its own mbarrier, so decoding starts before the activations land)
//          and of the step's f16 activations (TN rows x 128 bytes, 128-byte swizzle) into a
//          ring of stages;
//        warps 8-11: decoders, thread = weight row = tensor-memory lane: the row's four 16-trit
//          words become 64 f16 (pair-code pools -> f16 high bytes -> f16 pairs) stored with
//          tcgen05.st into one of two A buffers in tensor memory;
//        warp 13: allocates all 512 tensor-memory columns (two TN-column accumulators and the
//          two 32-column A buffers); lane 0 issues tcgen05.mma (A from tensor memory, B from
//          shared memory; M = 128, N = TN, K = 16; 4 per K step) and commits each stage's and
//          each A buffer's release and each finished accumulator;
//        warps 0-7: epilogue -- tcgen05.ld of a finished accumulator (lane = weight row,
//          column = token), scales, fp32 stores that are 128-byte coalesced per warp --
//          overlapping the next tile's MMAs in the other accumulator.
// Decoding in the kernel costs about 240 warp-instructions of the ALU pipe per K step of one
// tile, against ~500 cycles of MMA at N = 224: a quarter of the pipe, and the A operand never
// passes through shared memory. Every wait is bounded (2 s); a CTA that gives up still drains
// its own copies and MMAs, frees its tensor memory and records the code 17 in the workspace's
// status header.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <string>

#include "nt_kernels.cuh"

namespace nt {
namespace {

constexpr int kBM = 128;                    // weight rows per tile (MMA M) = 32 tiles of 4 rows
constexpr int kBN = 224;                    // largest token tile (MMA N); a call picks TN <= kBN
constexpr int kBK = 64;                     // trits of K per stage: 4 MMAs of K = 16
constexpr int kStages = 5;
constexpr int kBBytes = kBN * kBK * 2;      // f16 activations of a stage: 28 KB (1024-aligned)
constexpr int kABytes = 32 * kBK;           // packed trits of a stage: 32 tiles x 64 bytes
constexpr int kStageBytes = kBBytes + kABytes;
constexpr int kEpiThreads = 256;            // warps 0-7: two per tensor-memory lane quarter
constexpr int kDecoders = 128;              // warps 8-11
constexpr int kDecWarp0 = kEpiThreads / 32;
constexpr int kProducerWarp = kDecWarp0 + 4, kMmaWarp = kProducerWarp + 1;
constexpr int kThreadsTc = (kMmaWarp + 1) * 32;
constexpr int kTcMaxMats = 8;               // matrices per call sharing the activations
constexpr int kTmemCols = 512;              // accumulators at 0 and TN, A buffers at kACol
constexpr uint32_t kACol = 2 * kBN;         // 448: two 32-column f16 A buffers
constexpr int kABufs = 2;
constexpr uint64_t kTcTimeoutNs = 2000000000ull;
constexpr unsigned int kTcErrWait = 17;     // status code of a wait that ran out
constexpr int kSmemTc = kStages * kStageBytes + 1024 /* alignment */ + 2 * kBN * 4 /* token scales */ +
                        256 /* barriers */;
static_assert(kACol + kABufs * 32 <= kTmemCols, "tensor-memory columns");
static_assert(kBBytes % 1024 == 0 && kStageBytes % 1024 == 0, "stage alignment of the swizzled operand");

// f16 pair-code pools: the tiled layout's codes select the high byte of +1 / -1 / 0 as 0x3C /
// 0xBC / 0x00 (the low byte of all three is 0). Code 14 (the pair (0, -1)) reads byte 6 in
// sign-replicate mode: pool A's 0x3C gives 0x00, pool B's 0xBC gives 0xFF, which the AND
// with 0xBC turns into 0xBC.
constexpr uint32_t kPoolA_lo = 0x00BC3C00u;  // codes 0..3 -> 0, +1, -1, 0
constexpr uint32_t kPoolA_hi = 0xBC3CBC3Cu;  // codes 4..7 -> +1, -1, +1, -1
constexpr uint32_t kPoolB_lo = 0x3C000000u;  // codes 0..3 -> 0, 0, 0, +1
constexpr uint32_t kPoolB_hi = 0xBCBC3C3Cu;  // codes 4..7 -> +1, +1, -1, -1

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
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
// Bounded wait; false after the timeout or once another role of the CTA has given up.
__device__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* fail, uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t deadline = globaltimer_ns() + timeout_ns;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0u && (*fail || globaltimer_ns() > deadline)) {
      *fail = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major 16-bit operand with the 128-byte swizzle (the
// layout the TMA writes): rows of 128 bytes, 8-row groups 1024 bytes apart; version 1.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;  // stride byte offset: 8-row group pitch
  d |= (uint64_t)1 << 46;                          // descriptor version (sm_100)
  d |= (uint64_t)2 << 61;                          // layout: 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f16, A = B = f16, D = fp32, both K-major, M = 128, N = tn.
__host__ __device__ constexpr uint32_t idesc_f16(int tn) {
  return (1u << 4) | ((uint32_t)(tn >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
}

__device__ __forceinline__ void mma_f16_tmem_a(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// ---- activation conversion -------------------------------------------------------------
// int8 codes -> f16 [M][K], once per call for all its matrices, exactly: a code v biased to
// u = v + 128 under the exponent byte 0x64 is the f16 1024 + u, and one f16x2 subtraction of
// 1152 leaves v (both operands lie in [1024, 2048), so the difference is exact).
__device__ __forceinline__ uint2 int8x4_f16(uint32_t x) {
  const uint32_t u = x ^ 0x80808080u;
  uint32_t lo = prmt(u, 0x64646464u, 0x4140u), hi = prmt(u, 0x64646464u, 0x4342u);
  const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6480u));  // 1152
  const __half2 a = __hsub2(*reinterpret_cast<const __half2*>(&lo), bias);
  const __half2 b = __hsub2(*reinterpret_cast<const __half2*>(&hi), bias);
  return make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
}

// Launched as a programmatic dependent: waits for the previous kernel (which may still be
// reading the workspace it overwrites) before its first access.
__global__ void __launch_bounds__(256) act_f16_kernel(const uint4* __restrict__ q, int64_t groups,
                                                      uint4* __restrict__ out) {
  dependent_launch_wait();
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < groups; i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 v = __ldg(q + i);
    const uint2 c0 = int8x4_f16(v.x), c1 = int8x4_f16(v.y), c2 = int8x4_f16(v.z), c3 = int8x4_f16(v.w);
    out[2 * i] = make_uint4(c0.x, c0.y, c1.x, c1.y);
    out[2 * i + 1] = make_uint4(c2.x, c2.y, c3.x, c3.y);
  }
}

// ---- GEMM ------------------------------------------------------------------------------
// The weights are the MMA's M side (128 rows per tile) and the tokens its N side, so
// tensor-memory lane = weight row and column = token: each epilogue store of one column by a
// warp is 32 consecutive floats of one output row. Several matrices sharing the activations
// are one tile set: matrix i owns weight tiles [tile_start[i], tile_start[i + 1]).
struct TcParams {
  const float* s_x;  // [M]
  int M, K;
  int tiles_n, tiles_m;  // 128-row weight tiles (all matrices), tn-token tiles
  int tn;                // tokens per tile (MMA N): a multiple of 32, <= kBN
  int n_mats;
  int tile_start[kTcMaxMats + 1];
  int Nm[kTcMaxMats];
  const float* s_w[kTcMaxMats];  // [N_i]
  float* y[kTcMaxMats];          // [M][N_i]
  int32_t* acc[kTcMaxMats];      // [M][N_i] or null
  unsigned int* err;             // the workspace's status header [code, CTA]
  uint64_t timeout_ns;           // bound on every wait
  int fault;                     // tests of the timeout path: the producer issues no copies
  const uint8_t* w[kTcMaxMats];  // the packed weights (prefetched into L2 at the start)
  int64_t w_bytes[kTcMaxMats];
};
// The packed-weight maps (one per matrix: 4-row tiles of Kp bytes, box 64 bytes x 32 tiles)
// and the activations' map, as one kernel parameter.
struct TcMaps {
  CUtensorMap w[kTcMaxMats];
  CUtensorMap x;
};

__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
}

__device__ __forceinline__ int tile_matrix(const TcParams& p, int tn) {
  int mi = 0;
  while (mi + 1 < p.n_mats && tn >= p.tile_start[mi + 1]) ++mi;
  return mi;
}

__global__ void __launch_bounds__(kThreadsTc, 1)
    gemm_tc_kernel(const __grid_constant__ TcMaps maps, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* sxs = reinterpret_cast<float*>(smem + kStages * kStageBytes);  // [2][kBN] token scales
  uint64_t* bars = reinterpret_cast<uint64_t*>(sxs + 2 * kBN);
  // full: a stage's activations landed; wfull: its packed weights landed (the decoders start on
  // those without waiting for the larger activation tile); empty: both read
  const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * kStages, wfull0 = empty0 + 8 * kStages;
  const uint32_t afull0 = wfull0 + 8 * kStages, aempty0 = afull0 + 8 * kABufs;
  const uint32_t tfull0 = aempty0 + 8 * kABufs, tempty0 = tfull0 + 16, drain = tempty0 + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * kStages + 2 * kABufs + 5);
  volatile int* fail = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int n_tiles = p.tiles_n * p.tiles_m;
  const int ksteps = (p.K + kBK - 1) / kBK;
  const int TN = p.tn;

  if (t == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(wfull0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kDecoders + 1);  // the decoders' reads and the MMAs' commit
    }
    for (int b = 0; b < kABufs; ++b) {
      mbar_init(afull0 + 8 * b, kDecoders);
      mbar_init(aempty0 + 8 * b, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull0 + 8 * b, 1);
      mbar_init(tempty0 + 8 * b, kEpiThreads);
    }
    mbar_init(drain, 1);
    *fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  // The call's packed weights (at most a few MB) into L2, 1/grid of them per CTA: every token
  // tile re-reads them, and the first reads would otherwise wait on DRAM inside the MMA loop.
  // Weights are constant inputs, so this may run before the previous kernel has finished.
  if (warp == kProducerWarp && lane == 0) {
    int64_t total = 0;  // the matrices' bytes taken as one range; this CTA prefetches [lo, hi)
    for (int i = 0; i < p.n_mats; ++i) total += p.w_bytes[i];
    const int64_t per = (total / gridDim.x + 15) & ~(int64_t)15;
    const int64_t lo = (int64_t)blockIdx.x * per, hi = lo + per < total ? lo + per : total;
    int64_t start = 0;  // offset of matrix i in that range (every size is a multiple of 16)
    for (int i = 0; i < p.n_mats; ++i) {
      const int64_t b0 = lo > start ? lo : start, b1 = hi < start + p.w_bytes[i] ? hi : start + p.w_bytes[i];
      for (int64_t o = b0; o < b1; o += 65536) {
        const uint32_t n = (uint32_t)(b1 - o < 65536 ? b1 - o : 65536);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.w[i] + (o - start)), "r"(n) : "memory");
      }
      start += p.w_bytes[i];
    }
  }
  // Launched as a programmatic dependent of the activation conversion: the set-up above
  // overlaps it, and nothing below reads an input before it has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp == kProducerWarp) {
    // ---- TMA producer ----
    if (lane == 0) {
      uint32_t it = 0;
      for (int tile = blockIdx.x; tile < n_tiles && !*fail && !p.fault; tile += gridDim.x) {
        const int tn = tile % p.tiles_n, tm = tile / p.tiles_n;
        const int mi = tile_matrix(p, tn);
        const int wrow = (tn - p.tile_start[mi]) * (kBM / 4);  // first 4-row tile of the box
        for (int ks = 0; ks < ksteps; ++ks, ++it) {
          const uint32_t s = it % kStages;
          if (it >= kStages && !mbar_wait(empty0 + 8 * s, ((it / kStages) - 1) & 1u, fail, p.timeout_ns)) break;
          const uint32_t st = smem_u32(smem + s * kStageBytes);
          mbar_expect_tx(wfull0 + 8 * s, (uint32_t)kABytes);
          tma_load_2d(st + kBBytes, &maps.w[mi], ks * kBK, wrow, wfull0 + 8 * s);
          mbar_expect_tx(full0 + 8 * s, (uint32_t)(TN * kBK * 2));
          tma_load_2d(st, &maps.x, ks * kBK, tm * TN, full0 + 8 * s);
        }
      }
      // Drain: the last copy issued into each stage must land before the CTA may exit.
      for (uint32_t s = 0; s < kStages && s < it; ++s) {
        const uint32_t last = (it - 1 - s) / kStages * kStages + s;
        const uint64_t deadline = globaltimer_ns() + p.timeout_ns;
        while (!mbar_try_wait(full0 + 8 * s, (last / kStages) & 1u) || !mbar_try_wait(wfull0 + 8 * s, (last / kStages) & 1u))
          if (globaltimer_ns() > deadline) break;
      }
    }
  } else if (warp == kMmaWarp) {
    // ---- MMA issuer ----
    if (lane == 0) {
      uint32_t it = 0, j = 0;
      const uint32_t idesc = idesc_f16(TN);
      for (int tile = blockIdx.x; tile < n_tiles && !*fail; tile += gridDim.x, ++j) {
        const uint32_t buf = j & 1u;
        if (j >= 2 && !mbar_wait(tempty0 + 8 * buf, ((j >> 1) - 1) & 1u, fail, p.timeout_ns)) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t d = tmem + buf * (uint32_t)TN;
        bool ok = true;
        for (int ks = 0; ks < ksteps; ++ks, ++it) {
          const uint32_t s = it % kStages, b = it % kABufs;
          if (!mbar_wait(full0 + 8 * s, (it / kStages) & 1u, fail, p.timeout_ns) ||
              !mbar_wait(afull0 + 8 * b, (it / kABufs) & 1u, fail, p.timeout_ns)) {
            ok = false;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint32_t bsm = smem_u32(smem + s * kStageBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)  // 16 f16 = 8 tensor-memory columns of A, 32 bytes of B
            mma_f16_tmem_a(d, tmem + kACol + 32u * b + 8u * (uint32_t)kk, sdesc_sw128(bsm + 32u * (uint32_t)kk), idesc,
                           (ks | kk) != 0);
          mma_commit(empty0 + 8 * s);   // the stage is free once these MMAs have read it
          mma_commit(aempty0 + 8 * b);  // and so is the A buffer
        }
        if (!ok) break;
        mma_commit(tfull0 + 8 * buf);  // accumulator buf complete
      }
      mma_commit(drain);  // every MMA of this CTA done (waited below before the memory is freed)
      const uint64_t deadline = globaltimer_ns() + p.timeout_ns;
      while (!mbar_try_wait(drain, 0))
        if (globaltimer_ns() > deadline) break;
    }
  } else if (warp >= kDecWarp0) {
    // ---- decoders: thread = weight row of the tile = tensor-memory lane ----
    const int row = t - kEpiThreads;   // 0..127
    const int T = row >> 2, jr = row & 3;  // 4-row tile within the box, row within it
    const uint32_t tl = tmem + ((uint32_t)(32 * (warp - kDecWarp0)) << 16);
    uint32_t it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
      for (int ks = 0; ks < ksteps; ++ks, ++it) {
        const uint32_t s = it % kStages, b = it % kABufs;
        if (!mbar_wait(wfull0 + 8 * s, (it / kStages) & 1u, fail, p.timeout_ns)) { ok = false; break; }
        // the row's four words of the step: 16-byte group g of tile T holds one word per row
        const uint8_t* ws = smem + s * kStageBytes + kBBytes + T * kBK + 4 * jr;
        uint32_t w[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) w[g] = *reinterpret_cast<const uint32_t*>(ws + 16 * g);
        mbar_arrive(empty0 + 8 * s);  // release: the reads above are ordered before it
        uint32_t c[32];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const uint32_t hi = w[g] >> 16;
          const uint32_t o0 = prmt(kPoolA_lo, kPoolA_hi, w[g]);                // trits 0..3
          const uint32_t o1 = prmt(kPoolB_lo, kPoolB_hi, w[g]) & 0xBCBCBCBCu;  // trits 4..7
          const uint32_t o2 = prmt(kPoolA_lo, kPoolA_hi, hi);                  // trits 8..11
          const uint32_t o3 = prmt(kPoolB_lo, kPoolB_hi, hi) & 0xBCBCBCBCu;    // trits 12..15
          c[8 * g + 0] = prmt(o0, 0u, 0x1404u);  // f16 pair (trit 2i, trit 2i + 1), low half first
          c[8 * g + 1] = prmt(o0, 0u, 0x3424u);
          c[8 * g + 2] = prmt(o1, 0u, 0x1404u);
          c[8 * g + 3] = prmt(o1, 0u, 0x3424u);
          c[8 * g + 4] = prmt(o2, 0u, 0x1404u);
          c[8 * g + 5] = prmt(o2, 0u, 0x3424u);
          c[8 * g + 6] = prmt(o3, 0u, 0x1404u);
          c[8 * g + 7] = prmt(o3, 0u, 0x3424u);
        }
        if (it >= kABufs && !mbar_wait(aempty0 + 8 * b, ((it / kABufs) - 1) & 1u, fail, p.timeout_ns)) {
          ok = false;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
            "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(tl + kACol + 32u * b),
            "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(c[4]), "r"(c[5]), "r"(c[6]), "r"(c[7]), "r"(c[8]),
            "r"(c[9]), "r"(c[10]), "r"(c[11]), "r"(c[12]), "r"(c[13]), "r"(c[14]), "r"(c[15]), "r"(c[16]),
            "r"(c[17]), "r"(c[18]), "r"(c[19]), "r"(c[20]), "r"(c[21]), "r"(c[22]), "r"(c[23]), "r"(c[24]),
            "r"(c[25]), "r"(c[26]), "r"(c[27]), "r"(c[28]), "r"(c[29]), "r"(c[30]), "r"(c[31])
            : "memory");
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        mbar_arrive(afull0 + 8 * b);
      }
    }
  } else {
    // ---- epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. +31 (weight rows) and
    // columns (tokens) [TN/2 (w / 4), +TN/2) of the finished accumulator ----
    const int quarter = warp & 3, half = warp >> 2;
    uint32_t j = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++j) {
      const uint32_t buf = j & 1u;
      const int tn = tile % p.tiles_n, tm = tile / p.tiles_n;
      const int mi = tile_matrix(p, tn);
      const int Nm = p.Nm[mi];
      float* const y = p.y[mi];
      int32_t* const acc = p.acc[mi];
      const int n = (tn - p.tile_start[mi]) * kBM + quarter * 32 + lane, m0 = tm * TN;  // row of matrix mi
      if (t < kBN) sxs[buf * kBN + t] = (t < TN && m0 + t < p.M) ? __ldg(p.s_x + m0 + t) : 0.0f;
      const float sw = (n < Nm) ? __ldg(p.s_w[mi] + n) : 0.0f;
      epi_sync();  // token scales of this tile visible to every epilogue thread
      // After a failed wait the thread keeps walking the tiles (the named barrier above needs
      // every epilogue thread) and only skips the stores.
      const bool ok = mbar_wait(tfull0 + 8 * buf, (j >> 1) & 1u, fail, p.timeout_ns);
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t base = tmem + buf * (uint32_t)TN + half * (TN / 2) + ((uint32_t)(quarter * 32) << 16);
#pragma unroll 1
      for (int c0 = 0; c0 < TN / 2; c0 += 16) {
        uint32_t r0, r1, r2, r3, r4, r5, r6, r7, r8, r9, r10, r11, r12, r13, r14, r15;
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
            : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3), "=r"(r4), "=r"(r5), "=r"(r6), "=r"(r7), "=r"(r8), "=r"(r9),
              "=r"(r10), "=r"(r11), "=r"(r12), "=r"(r13), "=r"(r14), "=r"(r15)
            : "r"(base + (uint32_t)c0)
            : "memory");
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        const uint32_t r[16] = {r0, r1, r2, r3, r4, r5, r6, r7, r8, r9, r10, r11, r12, r13, r14, r15};
        const int mc = m0 + half * (TN / 2) + c0;
        if (ok && n < Nm) {
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const int m = mc + q;
            if (m < p.M) {
              const float a = __int_as_float((int)r[q]);  // an exact integer
              y[(int64_t)m * Nm + n] = __fmul_rn(__fmul_rn(a, sw), sxs[buf * kBN + half * (TN / 2) + c0 + q]);
              if (acc) acc[(int64_t)m * Nm + n] = __float2int_rn(a);
            }
          }
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      mbar_arrive(tempty0 + 8 * buf);
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == kMmaWarp)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  if (t == 0 && *fail && atomicCAS(p.err, 0u, kTcErrWait) == 0u) p.err[1] = blockIdx.x;
}

// ---- host ----------------------------------------------------------------------------
std::mutex g_tc_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
bool g_tc_attr[64] = {};

nt_status tc_setup(int dev) {
  std::lock_guard<std::mutex> lock(g_tc_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    NT_CUDA_TRY(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q));
    if (q != cudaDriverEntryPointSuccess || !fn) return set_error(NT_ERR_CUDA, "cuTensorMapEncodeTiled not available");
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  if (dev >= 0 && dev < 64 && !g_tc_attr[dev]) {
    NT_CUDA_TRY(cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTc));
    g_tc_attr[dev] = true;
  }
  return NT_OK;
}

// 2-D f16 tensor map over a row-major [rows][K] matrix, box 64 (K) x box_rows, 128B swizzle.
nt_status encode_act_map(CUtensorMap* map, const void* base, int rows, int K, int box_rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(NT_ERR_CUDA, "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")");
  return NT_OK;
}

// 2-D byte map over a tiled ternary matrix: [n_tiles][Kp] bytes (a 4-row tile per row), box
// 64 bytes (64 trits of each of the tile's 4 rows) x 32 tiles; tiles past the matrix read as 0.
nt_status encode_weight_map(CUtensorMap* map, const void* base, int N, int K) {
  const cuuint64_t dims[2] = {(cuuint64_t)padded_k(K), (cuuint64_t)(padded_rows(N) / 4)};
  const cuuint64_t strides[1] = {(cuuint64_t)padded_k(K)};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)(kBM / 4)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(NT_ERR_CUDA, "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")");
  return NT_OK;
}

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

// Tokens per tile: the multiple of 32 (<= kBN) that minimises (waves of tiles over the SMs) x
// (tile width + a fixed per-tile cost of about 48 columns), so the last wave is not left
// mostly empty.
int pick_token_tile(int M, int n_tiles_w, int sms) {
  int best = kBN / 32 * 32;
  int64_t best_cost = INT64_MAX;
  for (int tn = kBN / 32 * 32; tn >= 32; tn -= 32) {
    const int64_t tiles = (int64_t)n_tiles_w * ((M + tn - 1) / tn);
    const int64_t waves = (tiles + sms - 1) / sms;
    const int64_t cost = waves * (tn + 48);
    if (cost < best_cost) {
      best_cost = cost;
      best = tn;
    }
  }
  return best;
}

}  // namespace

bool tc_gemm_supported(int M, int K) { return M >= kTcMinBatch && K <= 131072; }

size_t tc_gemm_workspace_bytes(int M, int N, int K) { return tc_gemm_multi_workspace_bytes(M, 1, &N, K); }

// workspace: the status header (kWsHeaderBytes), then the f16 activations [M][K]; the weights
// are read in their packed form
size_t tc_gemm_multi_workspace_bytes(int M, int n, const int* N, int K) {
  (void)n;
  (void)N;
  return kWsHeaderBytes + align256((size_t)M * K * 2);
}

nt_status launch_gemm_tc(const uint8_t* w, const float* s_w, int N, int K, const int8_t* q, const float* s_x,
                         int M, float* y, int32_t* acc, void* ws, cudaStream_t st) {
  return launch_gemm_tc_multi(1, &w, &s_w, &N, K, q, s_x, M, &y, &acc, ws, st);
}

nt_status launch_gemm_tc_multi(int n, const uint8_t* const* w, const float* const* s_w, const int* N, int K,
                               const int8_t* q, const float* s_x, int M, float* const* y, int32_t* const* acc,
                               void* ws, cudaStream_t st) {
  if (n < 1 || n > kTcMaxMats) return set_error(NT_ERR_INVALID_ARG, "1 to 8 matrices per call");
  int dev = 0;
  NT_CUDA_TRY(cudaGetDevice(&dev));
  NT_TRY(tc_setup(dev));
  uint8_t* a_f16 = static_cast<uint8_t*>(ws) + kWsHeaderBytes;
  const int sms = device_sm_count();
  {
    const int64_t groups = (int64_t)M * K / 16;
    const int g = (int)std::min<int64_t>((groups + 255) / 256, (int64_t)sms * 8);
    NT_CUDA_TRY(launch_kernel(act_f16_kernel, dim3(g), dim3(256), 0, st, true, reinterpret_cast<const uint4*>(q),
                              groups, reinterpret_cast<uint4*>(a_f16)));
  }
  TcParams p{};
  p.err = static_cast<unsigned int*>(ws);
  p.timeout_ns = test_fault_timeout_ns(kTcTimeoutNs);
  p.fault = test_fault() == kFaultPrefill;
  p.s_x = s_x;
  p.M = M;
  p.K = K;
  p.n_mats = n;
  TcMaps maps;
  int tiles = 0;
  for (int i = 0; i < n; ++i) {  // each matrix's rows from a whole tile on
    p.tile_start[i] = tiles;
    p.Nm[i] = N[i];
    p.s_w[i] = s_w[i];
    p.y[i] = y[i];
    p.acc[i] = acc ? acc[i] : nullptr;
    NT_TRY(encode_weight_map(&maps.w[i], w[i], N[i], K));
    p.w[i] = w[i];
    p.w_bytes[i] = padded_rows(N[i]) / 4 * padded_k(K);
    tiles += (N[i] + kBM - 1) / kBM;
  }
  for (int i = n; i < kTcMaxMats; ++i) maps.w[i] = maps.w[0];
  p.tile_start[n] = tiles;
  p.tiles_n = tiles;
  const int tn = pick_token_tile(M, tiles, sms);
  NT_TRY(encode_act_map(&maps.x, a_f16, M, K, tn));  // tokens: MMA N side, tn-row boxes
  p.tn = tn;
  p.tiles_m = (M + tn - 1) / tn;
  const int n_tiles = p.tiles_m * p.tiles_n;
  NT_CUDA_TRY(launch_kernel(gemm_tc_kernel, dim3(std::min(n_tiles, sms)), dim3(kThreadsTc), kSmemTc, st, true, maps, p));
  return check_launch("gemm_tc_kernel");
}

}  // namespace nt
