// nt_gemm_tc.cu -- ternary projection of many activation vectors (prefill-shaped batches) on
// the 5th-generation tensor cores.
//
// Y[m][n] = fl(fl(acc[m][n] * s_w[n]) * s_x[m]),  acc = sum_k q[m][k] * t[n][k].
// Prefill pushes thousands of tokens through the same weights, so the work is a dense
// contraction (the MLxcel page measures prefill as compute-bound); batch-1 decode stays on
// the streaming kernels.
//
// Exactness: ternary weights and int8 activations are exact in bf16, each product is an
// integer of magnitude <= 127, and every partial sum stays below 127 * K < 2^24 for
// K <= 131072, so the fp32 accumulator in tensor memory holds the exact integer sum; the
// epilogue applies the same two rounded products as every other path.
//
// A call runs two kernels:
//   1. preparation: int8 activations -> bf16 [M][K] (once for every matrix of the call), each
//      matrix's tiled trits -> bf16 rows starting on a whole 128-row tile, zeros for the rows
//      that pad a matrix to whole tiles -- all into the caller's workspace (operands for this
//      call only; nothing is kept across calls);
//   2. a persistent GEMM over the tiles of all matrices, one CTA per SM, looping over tiles of
//      128 weight rows (MMA M) x TN tokens (MMA N; TN <= 256 picked per call so the tiles fill
//      whole waves of SMs):
//        warp 8 lane 0: 2-D TMA loads (128-byte swizzle) of both operands of each 64-wide K
//          step into a 4-stage ring (full/empty mbarriers);
//        warp 9: allocates 512 tensor-memory columns (two 256-column accumulators); lane 0
//          issues tcgen05.mma (M = 128, N = TN, K = 16; 4 per K step), commits each stage's
//          release and each finished accumulator;
//        warps 0-7: epilogue -- tcgen05.ld of a finished accumulator (lane = weight row,
//          column = token), scales, fp32 stores that are 128-byte coalesced per warp --
//          overlapping the next tile's MMAs in the other accumulator.
// Every wait is bounded (2 s); a CTA that gives up still drains its own copies and MMAs, frees
// its tensor memory and records the code 17 in the workspace's status header.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <string>

#include "nt_kernels.cuh"

namespace nt {
namespace {

constexpr int kBM = 128;             // weight rows per tile (MMA M)
constexpr int kBN = 256;             // largest token tile (MMA N); a call picks TN <= kBN
constexpr int kBK = 64;              // K per stage: one 128-byte row of bf16
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;   // 16 KB
constexpr int kBBytes = kBN * kBK * 2;   // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kEpiThreads = 256;         // warps 0-7: two per tensor-memory lane quarter
constexpr int kTcMaxMats = 8;            // matrices per call sharing the activations
constexpr int kThreadsTc = kEpiThreads + 64;
constexpr int kTmemCols = 2 * kBN;       // two accumulators
constexpr uint64_t kTcTimeoutNs = 2000000000ull;
constexpr unsigned int kTcErrWait = 17;  // status code of a wait that ran out
constexpr int kSmemTc = kStages * kStageBytes + 1024 /* alignment */ + 2 * kBN * 4 /* token scales */ +
                        256 /* barriers */;

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

// Shared-memory matrix descriptor of a K-major bf16 operand with the 128-byte swizzle (the
// layout the TMA writes): rows of 128 bytes, 8-row groups 1024 bytes apart; version 1.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;  // stride byte offset: 8-row group pitch
  d |= (uint64_t)1 << 46;                          // descriptor version (sm_100)
  d |= (uint64_t)2 << 61;                          // layout: 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f16, A = B = bf16, D = fp32, both K-major, M = 128, N = tn.
__host__ __device__ constexpr uint32_t idesc_for(int tn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(tn >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// 4 int8 trits (0x00 / 0x01 / 0xFF bytes) -> 4 bf16 (0, +1.0 = 0x3F80, -1.0 = 0xBF80).
__device__ __forceinline__ uint2 trits4_bf16(uint32_t x) {
  const uint32_t s = x & 0x80808080u, nz = x & 0x01010101u;
  const uint32_t hi = (nz * 0x3Fu) | s, lo = nz << 7;
  return make_uint2(prmt(lo, hi, 0x5140u), prmt(lo, hi, 0x7362u));
}

// 4 int8 -> 4 bf16, exactly: 0x4B0000XX with XX = v + 128 is 2^23 + v + 128 in fp32.
__device__ __forceinline__ uint2 int8x4_bf16(uint32_t x) {
  const uint32_t xx = x ^ 0x80808080u;
  const float f0 = __int_as_float((int)prmt(xx, 0x4B000000u, 0x7440u)) - 8388736.0f;
  const float f1 = __int_as_float((int)prmt(xx, 0x4B000000u, 0x7441u)) - 8388736.0f;
  const float f2 = __int_as_float((int)prmt(xx, 0x4B000000u, 0x7442u)) - 8388736.0f;
  const float f3 = __int_as_float((int)prmt(xx, 0x4B000000u, 0x7443u)) - 8388736.0f;
  const __nv_bfloat162 a = __floats2bfloat162_rn(f0, f1), b = __floats2bfloat162_rn(f2, f3);
  return make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
}

// ---- operand conversion --------------------------------------------------------------
// All operand preparation of one call in one launch: the activations, every matrix's trits,
// and zeros for the rows that pad each matrix to whole tiles (one grid-stride index space).
struct PrepArgs {
  const uint4* q;
  int64_t act_groups;   // 16-byte groups of activations
  uint4* a_out;
  int n, K;
  const uint8_t* w[kTcMaxMats];
  int N[kTcMaxMats];
  uint8_t* b_out[kTcMaxMats];        // bf16 rows of matrix i
  int64_t word_start[kTcMaxMats + 1];  // cumulative (row, 16-trit word) counts
  uint4* pad[kTcMaxMats];            // first padding row of matrix i
  int64_t pad_start[kTcMaxMats + 1];   // cumulative 16-byte zero stores
};

__global__ void __launch_bounds__(256) prep_kernel(const PrepArgs a) {
  const int64_t words = a.word_start[a.n], total = a.act_groups + words + a.pad_start[a.n];
  const int kg = a.K / 16;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    if (i < a.act_groups) {
      const uint4 v = __ldg(a.q + i);
      const uint2 c0 = int8x4_bf16(v.x), c1 = int8x4_bf16(v.y), c2 = int8x4_bf16(v.z), c3 = int8x4_bf16(v.w);
      a.a_out[2 * i] = make_uint4(c0.x, c0.y, c1.x, c1.y);
      a.a_out[2 * i + 1] = make_uint4(c2.x, c2.y, c3.x, c3.y);
      continue;
    }
    int64_t j = i - a.act_groups;
    if (j < words) {
      int mi = 0;
      while (j >= a.word_start[mi + 1]) ++mi;
      j -= a.word_start[mi];
      const int64_t r = j / kg, g = j % kg;
      const int64_t Kp = padded_k(a.K);
      const uint32_t word = __ldg(reinterpret_cast<const uint32_t*>(a.w[mi] + (r >> 2) * Kp + g * 16 + (r & 3) * 4));
      const Trits16 d = tiled_word_decode(word);
      const uint2 a0 = trits4_bf16(d.t0), a1 = trits4_bf16(d.t1), a2 = trits4_bf16(d.t2), a3 = trits4_bf16(d.t3);
      uint4* dst = reinterpret_cast<uint4*>(a.b_out[mi] + (r * a.K + g * 16) * 2);
      dst[0] = make_uint4(a0.x, a0.y, a1.x, a1.y);
      dst[1] = make_uint4(a2.x, a2.y, a3.x, a3.y);
      continue;
    }
    j -= words;
    int mi = 0;
    while (j >= a.pad_start[mi + 1]) ++mi;
    a.pad[mi][j - a.pad_start[mi]] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// ---- GEMM ------------------------------------------------------------------------------
// The weights are the MMA's M side (128 rows per tile) and the tokens its N side (256 per
// tile), so tensor-memory lane = weight row and column = token: each epilogue store of one
// column by a warp is 32 consecutive floats of one output row.
// Several matrices sharing the activations are one tile set: matrix i owns weight tiles
// [tile_start[i], tile_start[i + 1]) (its rows padded to whole tiles in the bf16 copy).
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
};

__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
}

__global__ void __launch_bounds__(kThreadsTc, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* sxs = reinterpret_cast<float*>(smem + kStages * kStageBytes);  // [2][kBN] token scales
  uint64_t* bars = reinterpret_cast<uint64_t*>(sxs + 2 * kBN);
  const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * kStages;
  const uint32_t tfull0 = empty0 + 8 * kStages, tempty0 = tfull0 + 16, drain = tempty0 + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 5);
  volatile int* fail = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int n_tiles = p.tiles_n * p.tiles_m;
  const int ksteps = (p.K + kBK - 1) / kBK;
  const int TN = p.tn;
  constexpr int kProducerWarp = kEpiThreads / 32, kMmaWarp = kProducerWarp + 1;

  if (t == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
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

  if (warp == kProducerWarp && lane == 0) {
    // ---- TMA producer ----
    uint32_t it = 0;
    for (int tile = blockIdx.x; tile < n_tiles && !*fail && !p.fault; tile += gridDim.x) {
      const int tn = tile % p.tiles_n, tm = tile / p.tiles_n;
      for (int ks = 0; ks < ksteps; ++ks, ++it) {
        const uint32_t s = it % kStages;
        if (it >= kStages && !mbar_wait(empty0 + 8 * s, ((it / kStages) - 1) & 1u, fail, p.timeout_ns)) break;
        const uint32_t a = smem_u32(smem + s * kStageBytes);
        mbar_expect_tx(full0 + 8 * s, kABytes + TN * kBK * 2);
        tma_load_2d(a, &tmW, ks * kBK, tn * kBM, full0 + 8 * s);
        tma_load_2d(a + kABytes, &tmX, ks * kBK, tm * TN, full0 + 8 * s);
      }
    }
    // Drain: the last copy issued into each stage must land before the CTA may exit.
    for (uint32_t s = 0; s < kStages && s < it; ++s) {
      const uint32_t last = (it - 1 - s) / kStages * kStages + s;
      const uint64_t deadline = globaltimer_ns() + p.timeout_ns;
      while (!mbar_try_wait(full0 + 8 * s, (last / kStages) & 1u))
        if (globaltimer_ns() > deadline) break;
    }
  } else if (warp == kMmaWarp && lane == 0) {
    // ---- MMA issuer ----
    uint32_t it = 0, j = 0;
    const uint32_t idesc = idesc_for(TN);
    for (int tile = blockIdx.x; tile < n_tiles && !*fail; tile += gridDim.x, ++j) {
      const uint32_t buf = j & 1u;
      if (j >= 2 && !mbar_wait(tempty0 + 8 * buf, ((j >> 1) - 1) & 1u, fail, p.timeout_ns)) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t d = tmem + buf * kBN;
      bool ok = true;
      for (int ks = 0; ks < ksteps; ++ks, ++it) {
        const uint32_t s = it % kStages;
        if (!mbar_wait(full0 + 8 * s, (it / kStages) & 1u, fail, p.timeout_ns)) { ok = false; break; }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t a = smem_u32(smem + s * kStageBytes), b = a + kABytes;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          mma_bf16(d, sdesc_sw128(a + kk * 32), sdesc_sw128(b + kk * 32), idesc, (ks | kk) != 0);
        mma_commit(empty0 + 8 * s);  // the stage is free once these MMAs have read it
      }
      if (!ok) break;
      mma_commit(tfull0 + 8 * buf);  // accumulator buf complete
    }
    mma_commit(drain);  // every MMA of this CTA done (waited below before the memory is freed)
    const uint64_t deadline = globaltimer_ns() + p.timeout_ns;
    while (!mbar_try_wait(drain, 0))
      if (globaltimer_ns() > deadline) break;
  } else if (warp < kProducerWarp) {
    // ---- epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. +31 (weight rows) and
    // columns (tokens) [128 (w / 4), +128) of the finished accumulator ----
    const int quarter = warp & 3, half = warp >> 2;
    uint32_t j = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++j) {
      const uint32_t buf = j & 1u;
      const int tn = tile % p.tiles_n, tm = tile / p.tiles_n;
      int mi = 0;
      while (mi + 1 < p.n_mats && tn >= p.tile_start[mi + 1]) ++mi;
      const int Nm = p.Nm[mi];
      float* const y = p.y[mi];
      int32_t* const acc = p.acc[mi];
      const int n = (tn - p.tile_start[mi]) * kBM + quarter * 32 + lane, m0 = tm * TN;  // row of matrix mi
      sxs[buf * kBN + t] = (t < TN && m0 + t < p.M) ? __ldg(p.s_x + m0 + t) : 0.0f;
      const float sw = (n < Nm) ? __ldg(p.s_w[mi] + n) : 0.0f;
      epi_sync();  // token scales of this tile visible to every epilogue thread
      // After a failed wait the thread keeps walking the tiles (the named barrier above needs
      // every epilogue thread) and only skips the stores.
      const bool ok = mbar_wait(tfull0 + 8 * buf, (j >> 1) & 1u, fail, p.timeout_ns);
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t base = tmem + buf * kBN + half * (TN / 2) + ((uint32_t)(quarter * 32) << 16);
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

// 2-D bf16 tensor map over a row-major [rows][K] matrix, box 64 (K) x box_rows, 128B swizzle.
nt_status encode_map(CUtensorMap* map, const void* base, int rows, int K, int box_rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(NT_ERR_CUDA, "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")");
  return NT_OK;
}

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

// Tokens per tile: the multiple of 32 (<= 256) that minimises (waves of tiles over the SMs) x
// (tile width + a fixed per-tile cost of about 48 columns), so the last wave is not left
// mostly empty (e.g. 8192 tokens x 3072 rows: 256-token tiles make 5.05 waves, 224 make 5.8).
int pick_token_tile(int M, int N, int sms) {
  const int64_t tiles_n = (N + kBM - 1) / kBM;
  int best = kBN;
  int64_t best_cost = INT64_MAX;
  for (int tn = kBN; tn >= 32; tn -= 32) {
    const int64_t tiles = tiles_n * ((M + tn - 1) / tn);
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

int64_t tc_weight_rows(int n, const int* N) {
  int64_t rows = 0;
  for (int i = 0; i < n; ++i) rows += (int64_t)(N[i] + kBM - 1) / kBM * kBM;
  return rows;
}

size_t tc_gemm_workspace_bytes(int M, int N, int K) { return tc_gemm_multi_workspace_bytes(M, 1, &N, K); }

// workspace: the status header (kWsHeaderBytes), bf16 activations, bf16 weight rows
size_t tc_gemm_multi_workspace_bytes(int M, int n, const int* N, int K) {
  return kWsHeaderBytes + align256((size_t)M * K * 2) + align256((size_t)tc_weight_rows(n, N) * K * 2);
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
  uint8_t* a_bf16 = static_cast<uint8_t*>(ws) + kWsHeaderBytes;
  uint8_t* b_bf16 = a_bf16 + align256((size_t)M * K * 2);
  const int sms = device_sm_count();
  PrepArgs pa{};
  pa.q = reinterpret_cast<const uint4*>(q);
  pa.act_groups = (int64_t)M * K / 16;  // the activations once for every matrix
  pa.a_out = reinterpret_cast<uint4*>(a_bf16);
  pa.n = n;
  pa.K = K;
  TcParams p{};
  p.err = static_cast<unsigned int*>(ws);
  p.timeout_ns = test_fault_timeout_ns(kTcTimeoutNs);
  p.fault = test_fault() == kFaultPrefill;
  p.s_x = s_x;
  p.M = M;
  p.K = K;
  p.n_mats = n;
  int64_t row = 0;
  for (int i = 0; i < n; ++i) {  // each matrix's rows from a whole tile on
    p.tile_start[i] = (int)(row / kBM);
    p.Nm[i] = N[i];
    p.s_w[i] = s_w[i];
    p.y[i] = y[i];
    p.acc[i] = acc ? acc[i] : nullptr;
    const int64_t padded = (int64_t)(N[i] + kBM - 1) / kBM * kBM;
    pa.w[i] = w[i];
    pa.N[i] = N[i];
    pa.b_out[i] = b_bf16 + row * K * 2;
    pa.word_start[i + 1] = pa.word_start[i] + (int64_t)N[i] * (K / 16);
    // rows past the matrix inside its last tile must read as zeros (garbage there corrupted
    // valid outputs on the tensor cores)
    pa.pad[i] = reinterpret_cast<uint4*>(b_bf16 + (row + N[i]) * K * 2);
    pa.pad_start[i + 1] = pa.pad_start[i] + (padded - N[i]) * K * 2 / 16;
    row += padded;
  }
  {
    const int64_t total = pa.act_groups + pa.word_start[n] + pa.pad_start[n];
    const int g = (int)std::min<int64_t>((total + 255) / 256, (int64_t)sms * 8);
    prep_kernel<<<g, 256, 0, st>>>(pa);
    NT_TRY(check_launch("prep_kernel"));
  }
  p.tile_start[n] = (int)(row / kBM);
  p.tiles_n = p.tile_start[n];
  const int tn = pick_token_tile(M, (int)row, sms);
  CUtensorMap mw, mx;
  NT_TRY(encode_map(&mw, b_bf16, (int)row, K, kBM));  // weights: MMA M side, 128-row boxes
  NT_TRY(encode_map(&mx, a_bf16, M, K, tn));          // tokens: MMA N side, tn-row boxes
  p.tn = tn;
  p.tiles_m = (M + tn - 1) / tn;
  const int tiles = p.tiles_m * p.tiles_n;
  gemm_tc_kernel<<<std::min(tiles, sms), kThreadsTc, kSmemTc, st>>>(mw, mx, p);
  return check_launch("gemm_tc_kernel");
}

}  // namespace nt
