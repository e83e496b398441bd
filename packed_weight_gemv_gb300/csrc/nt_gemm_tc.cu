// nt_gemm_tc.cu -- ternary projection of many activation vectors (prefill-shaped batches) on
// the 5th-generation tensor cores.
//
// Y[m][n] = fl(fl(acc[m][n] * s_w[n]) * s_x[m]),  acc = sum_k q[m][k] * t[n][k].
// Prefill pushes M >= 2048 tokens through the same weights, so the work is a dense contraction
// (the MLxcel page measures prefill as compute-bound); the batch-1 decode path stays on the
// streaming kernels.
//
// Exactness: ternary weights and int8 activations are exact in bf16, each product is an
// integer of magnitude <= 127, and every partial sum stays below 127 * K < 2^24 for
// K <= 131072, so the fp32 accumulator in tensor memory holds the exact integer sum; the
// epilogue applies the same two rounded products as every other path.
//
// CTA tile: 128 tokens (MMA M) x 256 weight rows (MMA N); K in steps of 64 through a
// 4-stage shared-memory pipeline; both operands K-major with the 128-byte swizzle.
//   warps 0-3 (converters): int8 activations -> bf16 and 2-bit tiled trits -> bf16, written
//     in the swizzled operand layout; then the epilogue (tensor memory -> scaled fp32 out);
//   warp 4: allocates the 256 tensor-memory columns; lane 0 issues tcgen05.mma (4 per
//     K-step, K = 16 each) and commits each stage's completion to its "empty" mbarrier.
// Every wait is bounded; after a timeout the CTA skips its remaining work (outputs are then
// invalid) but still frees its tensor memory and waits for its own MMAs.
#include <cuda_bf16.h>

#include "nt_kernels.cuh"

namespace nt {
namespace {

constexpr int kBM = 128;             // tokens per CTA (MMA M)
constexpr int kBN = 256;             // weight rows per CTA (MMA N)
constexpr int kBK = 64;              // K per pipeline stage (one 128-byte bf16 row segment)
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;   // 16 KB
constexpr int kBBytes = kBN * kBK * 2;   // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kConvThreads = 128;
constexpr int kThreadsTc = kConvThreads + 32;
constexpr int kTmemCols = 256;
constexpr uint64_t kTcTimeoutNs = 2000000000ull;  // 2 s per wait
constexpr int kSmemTc = kStages * kStageBytes + 1024 /* alignment */ + 256 /* barriers */;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
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
// Bounded wait; false after the timeout.
__device__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t deadline = globaltimer_ns() + kTcTimeoutNs;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0u && globaltimer_ns() > deadline) return false;
  }
}

// Shared-memory matrix descriptor of a K-major bf16 operand with the 128-byte swizzle: rows
// of 128 bytes (64 elements), 8-row groups 1024 bytes apart; sm_100 descriptor version 1.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  // leading byte offset: 0 (not used by a K-major operand with the 128-byte swizzle)
  d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;  // stride byte offset: 8-row group pitch
  d |= (uint64_t)1 << 46;                      // descriptor version (sm_100)
  d |= (uint64_t)2 << 61;                      // layout: 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f16, A = B = bf16, D = fp32, both K-major, M = 128, N = 256.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) |
                            ((uint32_t)(kBM >> 4) << 24);

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// Byte offset of 16-byte chunk c (0..7) of row r in a 128-byte-swizzled K-major tile.
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
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

struct TcParams {
  const uint8_t* w;   // tiled weights
  const float* s_w;   // [N]
  const int8_t* q;    // [M][K]
  const float* s_x;   // [M]
  float* y;           // [M][N]
  int32_t* acc;       // [M][N] or null
  int M, N, K;
};

// Converts K-step `ks` of the CTA's operands into stage buffers sa (A) and sb (B).
__device__ __forceinline__ void convert_stage(const TcParams& p, int m0, int n0, int ks, uint8_t* sa,
                                              uint8_t* sb, int t) {
  const int k0 = ks * kBK;
  // A: token row t (one per thread), 64 int8 -> 64 bf16 (8 swizzled chunks).
  {
    const int m = m0 + t;
    const int8_t* src = p.q + (int64_t)m * p.K + k0;
#pragma unroll
    for (int g = 0; g < 4; ++g) {  // 16 int8 per group -> chunks 2g, 2g+1
      uint4 v = make_uint4(0, 0, 0, 0);
      if (m < p.M && k0 + 16 * g < p.K) v = __ldg(reinterpret_cast<const uint4*>(src + 16 * g));
      const uint2 c0 = int8x4_bf16(v.x), c1 = int8x4_bf16(v.y), c2 = int8x4_bf16(v.z), c3 = int8x4_bf16(v.w);
      *reinterpret_cast<uint4*>(sa + swz(t, 2 * g)) = make_uint4(c0.x, c0.y, c1.x, c1.y);
      *reinterpret_cast<uint4*>(sa + swz(t, 2 * g + 1)) = make_uint4(c2.x, c2.y, c3.x, c3.y);
    }
  }
  // B: 64 tiles x 4 groups of 16 bytes (4 rows x 16 trits each); 2 groups per thread.
  {
    const int64_t Kp = padded_k(p.K), tiles_total = padded_rows(p.N) / 4;
    const int tl = t >> 1;                    // tile within the CTA's 256 rows
    const int64_t tile = (int64_t)(n0 >> 2) + tl;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int jj = (t & 1) * 2 + h;         // group within the K-step (0..3)
      uint4 v = make_uint4(0, 0, 0, 0);
      if (tile < tiles_total) v = __ldg(reinterpret_cast<const uint4*>(p.w + tile * Kp + (int64_t)(k0 / 16 + jj) * 16));
      const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const Trits16 d = tiled_word_decode(words[r]);
        const uint2 a0 = trits4_bf16(d.t0), a1 = trits4_bf16(d.t1);
        const uint2 a2 = trits4_bf16(d.t2), a3 = trits4_bf16(d.t3);
        const int row = tl * 4 + r;
        *reinterpret_cast<uint4*>(sb + swz(row, 2 * jj)) = make_uint4(a0.x, a0.y, a1.x, a1.y);
        *reinterpret_cast<uint4*>(sb + swz(row, 2 * jj + 1)) = make_uint4(a2.x, a2.y, a3.x, a3.y);
      }
    }
  }
}

__global__ void __launch_bounds__(kThreadsTc, 1) gemm_tc_kernel(const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  // Operand stages must sit on 1024-byte boundaries (swizzle atom).
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 1);
  volatile int* s_fail = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kStages), accbar = smem_u32(bars + 2 * kStages);

  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int m0 = blockIdx.x * kBM, n0 = blockIdx.y * kBN;
  const int ksteps = (int)(padded_k(p.K) / kBK);

  if (t == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8 * s, kConvThreads);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(accbar, 1);
    *s_fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 4) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    if (lane == 0) {  // MMA issuer
      for (int ks = 0; ks < ksteps; ++ks) {
        const int s = ks % kStages;
        if (!mbar_wait(full0 + 8 * s, (uint32_t)(ks / kStages) & 1u)) { *s_fail = 1; break; }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t a = smem_u32(smem + s * kStageBytes), b = a + kABytes;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          mma_bf16(tmem, sdesc_sw128(a + kk * 32), sdesc_sw128(b + kk * 32), (ks | kk) != 0);
        mma_commit(empty0 + 8 * s);  // stage s free once these MMAs have read it
      }
      mma_commit(accbar);  // accumulator complete (or, after a failure, MMAs drained)
    }
  } else {
    // Converters: fill stage s once the MMAs of K-step ks - kStages have released it.
    for (int ks = 0; ks < ksteps; ++ks) {
      const int s = ks % kStages;
      if (ks >= kStages && !mbar_wait(empty0 + 8 * s, (uint32_t)(ks / kStages - 1) & 1u)) { *s_fail = 1; }
      if (*s_fail) break;
      uint8_t* sa = smem + s * kStageBytes;
      convert_stage(p, m0, n0, ks, sa, sa + kABytes, t);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> tensor core
      mbar_arrive(full0 + 8 * s);
    }
    // Epilogue: thread t owns token row m0 + t (tensor-memory lane t).
    const bool ok = mbar_wait(accbar, 0);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const int m = m0 + t;
    const float sx = (m < p.M) ? p.s_x[m] : 0.0f;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    for (int c0 = 0; c0 < kBN; c0 += 16) {
      uint32_t r[16];
      asm volatile(
          "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
          : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
            "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
          : "r"(lane_base + (uint32_t)c0)
          : "memory");
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      if (!ok || *s_fail || m >= p.M) continue;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int n = n0 + c0 + j;
        if (n < p.N) {
          const float a = __int_as_float((int)r[j]);  // an exact integer
          p.y[(int64_t)m * p.N + n] = __fmul_rn(__fmul_rn(a, __ldg(p.s_w + n)), sx);
          if (p.acc) p.acc[(int64_t)m * p.N + n] = __float2int_rn(a);
        }
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 4)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

}  // namespace

bool tc_gemm_supported(int M, int K) { return M >= kTcMinBatch && K <= 131072; }

nt_status launch_gemm_tc(const uint8_t* w, const float* s_w, int N, int K, const int8_t* q, const float* s_x,
                         int M, float* y, int32_t* acc, cudaStream_t st) {
  static bool attr_set = false;
  if (!attr_set) {
    NT_CUDA_TRY(cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTc));
    attr_set = true;
  }
  TcParams p{w, s_w, q, s_x, y, acc, M, N, K};
  const dim3 grid((M + kBM - 1) / kBM, (N + kBN - 1) / kBN);
  gemm_tc_kernel<<<grid, kThreadsTc, kSmemTc, st>>>(p);
  return check_launch("gemm_tc_kernel");
}

}  // namespace nt
