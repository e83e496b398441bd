// nt_internal.cuh -- device helpers and host-side plumbing shared by the library's own
// translation units (never by the oracle).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "nt.h"

namespace nt {

// ---------------------------------------------------------------------------------------
// Host side: error reporting and argument checks.
// ---------------------------------------------------------------------------------------
nt_status set_error(nt_status s, const std::string& detail);
nt_status clear_error();
nt_status check_device(int* sm_count = nullptr);  // GB300 (cc 10.3) or NT_ERR_UNSUPPORTED
int device_sm_count();

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Test hook of the per-call timeout paths (nt_set_test_fault): the fault that is set (0 =
// none) and the bound on the per-call kernels' waits while it is set (`dflt` otherwise).
enum : int { kFaultNone = 0, kFaultHeadStream = 1, kFaultTc8 = 2, kFaultPrefill = 3 };
int test_fault();
uint64_t test_fault_timeout_ns(uint64_t dflt);

#define NT_TRY(expr)                         \
  do {                                       \
    nt_status _s = (expr);                   \
    if (_s != NT_OK) return _s;              \
  } while (0)

#define NT_CUDA_TRY(expr)                                                          \
  do {                                                                             \
    cudaError_t _e = (expr);                                                       \
    if (_e != cudaSuccess)                                                         \
      return ::nt::set_error(NT_ERR_CUDA, std::string(#expr) + ": " + cudaGetErrorString(_e)); \
  } while (0)

// Checks a kernel launch (configuration errors only; faults surface at the next sync).
nt_status check_launch(const char* what);

// Launches kern<<<grid, block, smem, st>>>(args...); with pdl the launch may begin while the
// previous kernel in the stream is still running (programmatic dependent launch). Every kernel
// launched this way starts with dependent_launch_wait(), so only its launch and scheduling
// overlap the previous kernel: none of its memory accesses do.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                          Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------------------------------
// Layout constants of the tiled ternary layout (see nt.h).
// ---------------------------------------------------------------------------------------
constexpr int kTileRows = 4;      // rows per tile
constexpr int kKAlign = 512;      // Kp = roundup(K, 512): one warp-wide 512-byte sweep
constexpr int kGroupBytes = 16;   // one 16-byte group = 4 rows x 16 trits

__host__ __device__ inline int64_t padded_rows(int N) { return ((int64_t)N + 3) / 4 * 4; }
__host__ __device__ inline int64_t padded_k(int K) { return ((int64_t)K + kKAlign - 1) / kKAlign * kKAlign; }
// Bytes of one tile (4 rows x Kp trits at 2 bits) = Kp.
__host__ __device__ inline int64_t tile_bytes(int K) { return padded_k(K); }

// ---------------------------------------------------------------------------------------
// Device side.
// ---------------------------------------------------------------------------------------
#ifdef __CUDACC__

// Byte permute, PTX prmt.b32 default mode: byte i of the result is byte (c >> 4i) & 7 of the
// 8-byte pool {b:a} (a = bytes 0..3), or that byte's sign replicated when bit 4i+3 of c is
// set. Only c[15:0] is read.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ int dp4a(uint32_t a, uint32_t b, int c) {
  return __dp4a((int)a, (int)b, c);
}

// Pair-code pools of the tiled layout: with a word's low 16 bits as the selector, pool A
// yields the first trit of each of the 4 pairs as int8 and pool B the second. Codes 0..7
// copy a pool byte; code 14 (the pair (0,-1)) selects byte 6 in sign-replicate mode, which
// gives 0 from pool A (0x01) and -1 from pool B (0xFF).
constexpr uint32_t kPoolA_lo = 0x00FF0100u;  // codes 0..3 -> 0, +1, -1, 0
constexpr uint32_t kPoolA_hi = 0xFF01FF01u;  // codes 4..7 -> +1, -1, +1, -1
constexpr uint32_t kPoolB_lo = 0x01000000u;  // codes 0..3 -> 0, 0, 0, +1
constexpr uint32_t kPoolB_hi = 0xFFFF0101u;  // codes 4..7 -> +1, +1, -1, -1

// One tiled word (16 trits) as four int8x4 words, trits 0-3, 4-7, 8-11 and 12-15.
struct Trits16 {
  uint32_t t0, t1, t2, t3;
};
__device__ __forceinline__ Trits16 tiled_word_decode(uint32_t w) {
  const uint32_t hi = w >> 16;
  return Trits16{prmt(kPoolA_lo, kPoolA_hi, w), prmt(kPoolB_lo, kPoolB_hi, w),
                 prmt(kPoolA_lo, kPoolA_hi, hi), prmt(kPoolB_lo, kPoolB_hi, hi)};
}
__device__ __forceinline__ int trits16_dot(const Trits16& t, uint32_t a0, uint32_t a1, uint32_t a2,
                                           uint32_t a3, int acc) {
  acc = dp4a(t.t0, a0, acc);
  acc = dp4a(t.t1, a1, acc);
  acc = dp4a(t.t2, a2, acc);
  acc = dp4a(t.t3, a3, acc);
  return acc;
}

// Dot product of one tiled word (16 trits) with its 16 activation bytes a0..a3.
__device__ __forceinline__ int tiled_word_dot(uint32_t w, uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, int acc) {
  return trits16_dot(tiled_word_decode(w), a0, a1, a2, a3, acc);
}

// Plain-layout decode: field codes 00, 01, 11 (10 reads as 0) through a 4-entry byte table.
constexpr uint32_t kPlainLut = 0xFF000100u;  // codes 0..3 -> 0, +1, 0, -1

// Dot product of one plain word (16 trits, fields LSB first) with activation bytes
// q[0..15] packed little-endian in a0..a3.
__device__ __forceinline__ int plain_word_dot(uint32_t w, uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, int acc) {
  const uint32_t m0 = w & 0x33333333u;          // even trits' codes, one per nibble
  const uint32_t m1 = (w >> 2) & 0x33333333u;   // odd trits' codes
  const uint32_t qe_lo = prmt(a0, a1, 0x6420u), qo_lo = prmt(a0, a1, 0x7531u);
  const uint32_t qe_hi = prmt(a2, a3, 0x6420u), qo_hi = prmt(a2, a3, 0x7531u);
  acc = dp4a(prmt(kPlainLut, 0u, m0), qe_lo, acc);
  acc = dp4a(prmt(kPlainLut, 0u, m1), qo_lo, acc);
  acc = dp4a(prmt(kPlainLut, 0u, m0 >> 16), qe_hi, acc);
  acc = dp4a(prmt(kPlainLut, 0u, m1 >> 16), qo_hi, acc);
  return acc;
}

// Epilogue: fp32(fp32(float(acc) * s_row) * s_vec), each step rounded to nearest, no FMA.
__device__ __forceinline__ float scale_out(int acc, float s_row, float s_vec) {
  return __fmul_rn(__fmul_rn(__int2float_rn(acc), s_row), s_vec);
}

// Verify-pass acceptance by one thread: positions 0..B-1 hold the last emitted token and the
// B-1 drafted tokens; with j drafts equal to the model's arg-max at the position before them
// (and every earlier draft accepted), emit draft[0..j-1] then argmax[j]; returns j + 1.
__device__ __forceinline__ int verify_accept_device(const int32_t* draft, const int32_t* argmax, int B,
                                                    int32_t* emit) {
  int j = 0;
  while (j < B - 1 && draft[j] == argmax[j]) {
    emit[j] = draft[j];
    ++j;
  }
  emit[j] = argmax[j];
  return j + 1;
}

// First statement of a kernel that may be launched as a programmatic dependent: waits until the
// previous kernel in the stream has completed and its writes are visible (returns at once when
// the launch had no such dependency), then lets the next kernel's launch begin.
__device__ __forceinline__ void dependent_launch_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

#endif  // __CUDACC__

}  // namespace nt
