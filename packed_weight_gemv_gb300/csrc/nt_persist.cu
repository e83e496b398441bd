// nt_persist.cu -- the persistent decode-step kernel.
//
// "The Neutrino Engine" (§ "A 104 microsecond floor inside a 694 microsecond step") reports
// that a decode step spent most of its time across ~120 kernel boundaries, and that a single
// fused kernel with software barriers brought similar waits back. Here one cooperative
// launch streams the whole step, and the weight stream never waits for a barrier: weights
// do not depend on activations, so the producer warp of every CTA keeps its shared-memory
// ring full across stage boundaries while the consumer warps wait.
//
// CTA layout (one CTA per SM): warps 0..15 consume, warp 16 produces.
//   producer (lane w feeds consumer warp w): walks the CTA's schedule and issues one
//     cp.async.bulk per chunk (<= 4 KB of a tile or of an output-table row) of the units warp
//     w owns (units are dealt round-robin) into w's ring, completing on the slot's mbarrier;
//   consumers: wait for a chunk, decode + dp4a it against the activation held in shared
//     memory, release the slot; per unit (4 rows of a tiled matrix, or one output-table row)
//     a warp reduction and the fp32 epilogue.
// Ordered mode puts a grid-wide barrier before each stage; only consumers wait at it.
// Every wait is bounded by a %globaltimer deadline; on expiry the CTA records an error code,
// stops, and the producer waits (bounded) for its own copies in flight before exiting.
#include <float.h>
#include <limits.h>
#include <math.h>

#include <algorithm>
#include <string>
#include <vector>

#include "nt_step.cuh"

namespace nt {
namespace {

constexpr int kConsumerWarps = 16;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreadsP = kConsumerThreads + 32;
constexpr int kSlots = 3;
constexpr int kSlotBytes = 4096;
constexpr int kRingBytes = kConsumerWarps * kSlots * kSlotBytes;  // 192 KB
constexpr int kBars = kConsumerWarps * kSlots;                     // full (and empty) barriers
constexpr int kConsumerBarrier = 1;                                // named barrier id

enum : unsigned int { kErrFullWait = 1, kErrEmptyWait = 2, kErrGridBarrier = 3, kErrDrain = 4 };

struct PersistParams {
  const MatDesc* mats;
  const WorkItem* items;
  const int* item_off;  // [grid + 1]
  const QuantJob* qjobs;
  int n_qjobs;
  int n_barriers;
  StepCtrl* ctrl;
  const int8_t* head_T;
  const float* head_s;
  const int8_t* head_q;
  const float* head_sx;
  float* head_logits;
  int32_t* head_argmax;
  HeadWs* head_ws;
  int head_V, head_K;
  int has_head;
  int act_stride;
  uint32_t launch_idx;
  uint32_t barrier_extra;  // added to the first grid barrier's target (timeout-path tests)
  uint64_t timeout_ns;
};

// ---- PTX wrappers --------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
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
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                          uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync %0, %1;" ::"n"(kConsumerBarrier), "n"(kConsumerThreads) : "memory");
}
__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ unsigned int ld_acquire(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add(unsigned int* p, unsigned int v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ void record_error(StepCtrl* ctrl, unsigned int code, volatile int* s_abort) {
  *s_abort = 1;
  if (atomicCAS(&ctrl->error, 0u, code) == 0u) ctrl->error_cta = blockIdx.x;
}

// Bounded wait for the phase of `bar` with parity `parity` to complete.
__device__ bool wait_phase(uint32_t bar, uint32_t parity, uint64_t timeout_ns, StepCtrl* ctrl,
                           volatile int* s_abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t deadline = globaltimer_ns() + timeout_ns;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0u) {
      if (*s_abort) return false;  // this CTA gave up (shared flag, cheap to poll)
      if ((it & 1023u) == 0u) {    // rarely: the clock, and other CTAs' errors in L2
        if (globaltimer_ns() > deadline) return false;
        if (*reinterpret_cast<volatile unsigned int*>(&ctrl->error)) {
          *s_abort = 1;
          return false;
        }
      }
    }
  }
}

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum of 4 per-lane values across the warp; row r's total lands in lane 8r.
__device__ __forceinline__ int warp_sum4(int a0, int a1, int a2, int a3, int lane) {
  const bool h16 = lane & 16;
  int k0 = h16 ? a2 : a0, k1 = h16 ? a3 : a1;
  const int s0 = h16 ? a0 : a2, s1 = h16 ? a1 : a3;
  k0 += __shfl_xor_sync(0xffffffffu, s0, 16);
  k1 += __shfl_xor_sync(0xffffffffu, s1, 16);
  const bool h8 = lane & 8;
  int k = h8 ? k1 : k0;
  k += __shfl_xor_sync(0xffffffffu, h8 ? k0 : k1, 8);
  k += __shfl_xor_sync(0xffffffffu, k, 4);
  k += __shfl_xor_sync(0xffffffffu, k, 2);
  k += __shfl_xor_sync(0xffffffffu, k, 1);
  return k;
}

// Unit geometry of a work item: bytes per unit and the source base address.
__device__ __forceinline__ void unit_geometry(const PersistParams& P, const WorkItem& it,
                                              const uint8_t*& base, int& unit_bytes) {
  if (it.kind == kItemTernary) {
    const MatDesc& m = P.mats[it.mat];
    base = m.w;
    unit_bytes = (int)padded_k(m.K);
  } else {
    base = reinterpret_cast<const uint8_t*>(P.head_T);
    unit_bytes = P.head_K;
  }
}

// ---- producer ------------------------------------------------------------------------
// Lane w of the producer warp feeds consumer warp w's ring: it walks the CTA's schedule and
// issues the chunks of the units that warp w owns (units are dealt round-robin), so the 8
// lanes issue copies independently of each other.
__device__ void producer(const PersistParams& P, const WorkItem* items, int n_items, uint8_t* ring,
                         uint32_t full0, uint32_t empty0, volatile int* s_abort, int w) {
  const uint64_t pol = evict_first_policy();
  const uint32_t ring_w = smem_addr(ring) + (uint32_t)w * kSlots * kSlotBytes;
  const uint32_t full_w = full0 + 8u * w * kSlots, empty_w = empty0 + 8u * w * kSlots;
  uint32_t cnt = 0, seq = 0;
  bool ok = true;
  for (int i = 0; i < n_items && ok; ++i) {
    const WorkItem it = items[i];
    const uint8_t* base;
    int ub;
    unit_geometry(P, it, base, ub);
    const int64_t first = it.begin + (int64_t)((w - (int)(seq % kConsumerWarps) + kConsumerWarps) % kConsumerWarps);
    for (int64_t u = first; u < it.end && ok; u += kConsumerWarps) {
      const uint8_t* src = base + u * (int64_t)ub;
      for (int off = 0; off < ub; off += kSlotBytes) {
        const uint32_t bytes = (uint32_t)min(kSlotBytes, ub - off);
        const uint32_t slot = cnt % kSlots, phase = (cnt / kSlots) & 1u;
        if (!wait_phase(empty_w + 8 * slot, phase ^ 1u, P.timeout_ns, P.ctrl, s_abort)) {
          if (!*s_abort) record_error(P.ctrl, kErrEmptyWait, s_abort);
          ok = false;
          break;
        }
        mbar_expect_tx(full_w + 8 * slot, bytes);
        bulk_load(ring_w + slot * kSlotBytes, src + off, bytes, full_w + 8 * slot, pol);
        ++cnt;
      }
    }
    seq += (uint32_t)(it.end - it.begin);
  }
  // Drain: every slot's last copy must have landed before this thread (and so the CTA)
  // may exit, whatever happened to the consumers.
  for (uint32_t s = 0; s < kSlots; ++s) {
    if (cnt <= s) continue;
    const uint32_t last = (cnt - 1 - s) / kSlots * kSlots + s;
    const uint32_t bar = full_w + 8 * s;
    if (mbar_try_wait(bar, (last / kSlots) & 1u)) continue;
    const uint64_t deadline = globaltimer_ns() + P.timeout_ns;
    while (!mbar_try_wait(bar, (last / kSlots) & 1u)) {
      if (globaltimer_ns() > deadline) {
        record_error(P.ctrl, kErrDrain, s_abort);
        break;
      }
    }
  }
}

// ---- consumers -----------------------------------------------------------------------
struct ConsumerState {
  uint32_t cnt;  // chunks this warp consumed
  uint32_t seq;  // units seen by the CTA (for the round-robin owner)
  float best_v;  // output projection: this warp's best logit / row (lane 0)
  int best_i;
};

// Quantize one fp32 vector with the 256 consumer threads.
__device__ void quantize_consumers(const QuantJob& j, float* red) {
  const int t = threadIdx.x;
  float m = 0.0f;
  for (int k = t; k < j.K; k += kConsumerThreads) m = fmaxf(m, fabsf(j.x[k]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((t & 31) == 0) red[t >> 5] = m;
  consumer_sync();
  m = red[0];
#pragma unroll
  for (int i = 1; i < kConsumerWarps; ++i) m = fmaxf(m, red[i]);
  const float s = (m == 0.0f) ? 0.0f : __fdiv_rn(m, 127.0f);
  if (t == 0) *j.s = s;
  for (int k = t; k < j.K; k += kConsumerThreads) {
    int v = 0;
    if (m != 0.0f) {
      v = __float2int_rn(__fdiv_rn(j.x[k], s));
      v = v > 127 ? 127 : (v < -127 ? -127 : v);
    }
    j.q[k] = (int8_t)v;
  }
  consumer_sync();  // red[] reuse
}

// Grid-wide barrier among the consumers of all CTAs; `target` counts arrivals modulo 2^32.
__device__ bool grid_barrier(const PersistParams& P, uint32_t target, volatile int* s_abort) {
  target += P.barrier_extra;
  consumer_sync();
  if (threadIdx.x == 0 && !*s_abort) {
    __threadfence();
    red_release_add(&P.ctrl->arrive, 1u);
    const uint64_t deadline = globaltimer_ns() + P.timeout_ns;
    for (uint32_t it = 0;; ++it) {
      if ((int)(ld_acquire(&P.ctrl->arrive) - target) >= 0) break;
      if ((it & 63u) == 63u) {
        if (*reinterpret_cast<volatile unsigned int*>(&P.ctrl->error)) { *s_abort = 1; break; }
        if (globaltimer_ns() > deadline) { record_error(P.ctrl, kErrGridBarrier, s_abort); break; }
      }
    }
  }
  consumer_sync();
  return !*s_abort;
}

// Copies K activation bytes (K % 16 == 0) into shared memory, synchronously or with cp.async.
__device__ void load_act(uint8_t* dst, const int8_t* src, int K, bool async) {
  for (int o = threadIdx.x * 16; o < K; o += kConsumerThreads * 16) {
    if (async) cp_async16(smem_addr(dst + o), src + o);
    else *reinterpret_cast<uint4*>(dst + o) = __ldcg(reinterpret_cast<const uint4*>(src + o));
  }
  if (async) cp_async_commit();
}

__device__ __forceinline__ const int8_t* item_act(const PersistParams& P, const WorkItem& it, int& K) {
  if (it.kind == kItemTernary) {
    K = P.mats[it.mat].K;
    return P.mats[it.mat].q;
  }
  K = P.head_K;
  return P.head_q;
}

// A consumer warp's wait for one chunk: every lane waits (each observes the mbarrier phase,
// which makes the bulk copy's bytes visible to it) and the outcome is made warp-uniform, so
// no lane leaves while others go on to warp-wide shuffles.
__device__ __forceinline__ bool wait_chunk(uint32_t bar, uint32_t phase, const PersistParams& P,
                                           int lane, volatile int* s_abort) {
  const bool ok = __all_sync(0xffffffffu, wait_phase(bar, phase, P.timeout_ns, P.ctrl, s_abort));
  if (!ok && lane == 0 && !*s_abort) record_error(P.ctrl, kErrFullWait, s_abort);
  return ok;
}

// 16 bytes of one lane in one 512-byte piece: 4 rows x 16 trits against 16 activations.
__device__ __forceinline__ void tile_piece(const uint8_t* sb, const uint8_t* ab, int& a0, int& a1,
                                           int& a2, int& a3) {
  const uint4 wv = lds128(sb);
  const uint4 a = lds128(ab);
  a0 = tiled_word_dot(wv.x, a.x, a.y, a.z, a.w, a0);
  a1 = tiled_word_dot(wv.y, a.x, a.y, a.z, a.w, a1);
  a2 = tiled_word_dot(wv.z, a.x, a.y, a.z, a.w, a2);
  a3 = tiled_word_dot(wv.w, a.x, a.y, a.z, a.w, a3);
}

// One tile (4 rows) of a tiled ternary matrix. The row scale is loaded before the first
// chunk so its latency hides behind the chunk work; sx is the item's activation scale.
__device__ bool consume_tile(const PersistParams& P, const MatDesc& m, float sx, int64_t tile,
                             const uint8_t* act, uint8_t* ring, uint32_t full0, uint32_t empty0,
                             ConsumerState& st, int cw, int lane, volatile int* s_abort) {
  constexpr int kPieces = kSlotBytes / 512;
  const int pieces = (int)(padded_k(m.K) / 512);
  const int64_t n = tile * 4 + (lane >> 3);
  const float sw = ((lane & 7) == 0 && n < m.N) ? __ldg(m.s_w + n) : 0.0f;
  int a0 = 0, a1 = 0, a2 = 0, a3 = 0;
  for (int p0 = 0; p0 < pieces; p0 += kPieces) {
    const uint32_t slot = st.cnt % kSlots, phase = (st.cnt / kSlots) & 1u;
    const uint32_t idx = (uint32_t)cw * kSlots + slot;
    if (!wait_chunk(full0 + 8 * idx, phase, P, lane, s_abort)) return false;
    const uint8_t* sb = ring + idx * kSlotBytes + lane * 16;
    const uint8_t* ab = act + (p0 * 32 + lane) * 16;
    if (pieces - p0 >= kPieces) {
#pragma unroll
      for (int p = 0; p < kPieces; ++p) tile_piece(sb + p * 512, ab + p * 512, a0, a1, a2, a3);
    } else {
      for (int p = 0; p < pieces - p0; ++p) tile_piece(sb + p * 512, ab + p * 512, a0, a1, a2, a3);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * idx);
    ++st.cnt;
  }
  const int total = warp_sum4(a0, a1, a2, a3, lane);
  if ((lane & 7) == 0 && n < m.N) m.y[n] = scale_out(total, sw, sx);
  return true;
}

// One row of the int8 output table.
__device__ __forceinline__ void row_piece(const uint8_t* sb, const uint8_t* ab, int& acc) {
  const uint4 t = lds128(sb);
  const uint4 a = lds128(ab);
  acc = dp4a(t.x, a.x, acc);
  acc = dp4a(t.y, a.y, acc);
  acc = dp4a(t.z, a.z, acc);
  acc = dp4a(t.w, a.w, acc);
}

__device__ bool consume_head_row(const PersistParams& P, float sx, int64_t v, const uint8_t* act,
                                 uint8_t* ring, uint32_t full0, uint32_t empty0, ConsumerState& st,
                                 int cw, int lane, volatile int* s_abort) {
  const float sv = lane == 0 ? __ldg(P.head_s + v) : 0.0f;
  int acc = 0, acc2 = 0;
  for (int off = 0; off < P.head_K; off += kSlotBytes) {
    const int cb = min(kSlotBytes, P.head_K - off);
    const uint32_t slot = st.cnt % kSlots, phase = (st.cnt / kSlots) & 1u;
    const uint32_t idx = (uint32_t)cw * kSlots + slot;
    if (!wait_chunk(full0 + 8 * idx, phase, P, lane, s_abort)) return false;
    const uint8_t* sb = ring + idx * kSlotBytes + lane * 16;
    const uint8_t* ab = act + off + lane * 16;
    if (cb == kSlotBytes) {
#pragma unroll
      for (int o = 0; o < kSlotBytes; o += 1024) {
        row_piece(sb + o, ab + o, acc);
        row_piece(sb + o + 512, ab + o + 512, acc2);
      }
    } else {
      for (int o = 0; o + lane * 16 < cb; o += 512) row_piece(sb + o, ab + o, acc);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * idx);
    ++st.cnt;
  }
  const int total = warp_sum(acc + acc2);
  if (lane == 0) {
    const float lg = scale_out(total, sv, sx);
    if (P.head_logits) P.head_logits[v] = lg;
    if (lg > st.best_v) { st.best_v = lg; st.best_i = (int)v; }  // rows rise per warp
  }
  return true;
}

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

__global__ void __launch_bounds__(kThreadsP, 1) persist_kernel(const PersistParams P) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  uint8_t* act = smem + kRingBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(act + 2 * P.act_stride);
  HeadPartial* hbest = reinterpret_cast<HeadPartial*>(bars + 2 * kBars);
  float* red = reinterpret_cast<float*>(hbest + kConsumerWarps);
  volatile int* s_abort = reinterpret_cast<volatile int*>(red + kConsumerWarps);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full0 = smem_addr(bars), empty0 = smem_addr(bars + kBars);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kBars; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, 1);
    }
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  const int i0 = P.item_off[blockIdx.x], n_items = P.item_off[blockIdx.x + 1] - i0;
  const WorkItem* items = P.items + i0;

  if (warp == kConsumerWarps) {
    if (lane < kConsumerWarps) producer(P, items, n_items, ring, full0, empty0, s_abort, lane);
    return;
  }

  // ---- consumers ----
  // Every consumer warp walks the same sequence of named and grid barriers whatever
  // happens; after an abort (s_abort) they only skip the work, so no barrier is left short.
  const int cw = warp;
  ConsumerState st{0u, 0u, -INFINITY, INT_MAX};
  const uint32_t barrier_base = P.launch_idx * (uint32_t)P.n_barriers * gridDim.x;
  uint32_t barriers = 0;

  if (P.n_qjobs > 0) {  // quantize the step's fp32 inputs, then wait for every CTA
    for (int j = blockIdx.x; j < P.n_qjobs; j += gridDim.x) quantize_consumers(P.qjobs[j], red);
    ++barriers;
    grid_barrier(P, barrier_base + barriers * gridDim.x, s_abort);
  }

  int buf = 0;
  bool prefetched = false;
  for (int i = 0; i < n_items; ++i) {
    const WorkItem it = items[i];
    if (it.flags & kFlagStage) {
      ++barriers;
      grid_barrier(P, barrier_base + barriers * gridDim.x, s_abort);
    }
    int K;
    const int8_t* q = item_act(P, it, K);
    uint8_t* abuf = act + buf * P.act_stride;
    if (prefetched) cp_async_wait_all();
    else load_act(abuf, q, K, false);
    consumer_sync();  // act[buf] complete; every warp is past the previous item
    prefetched = false;
    if (i + 1 < n_items && !(items[i + 1].flags & kFlagStage)) {
      int K2;
      const int8_t* q2 = item_act(P, items[i + 1], K2);
      load_act(act + (buf ^ 1) * P.act_stride, q2, K2, true);
      prefetched = true;
    }
    // The abort flag is read by lane 0 and broadcast, so the whole warp takes one branch.
    const int64_t first = it.begin + (int64_t)((cw - (int)(st.seq % kConsumerWarps) + kConsumerWarps) % kConsumerWarps);
    if (it.kind == kItemTernary) {
      const MatDesc m = P.mats[it.mat];
      const float sx = __ldcg(m.s_x);
      for (int64_t u = first; u < it.end; u += kConsumerWarps)
        if (!__shfl_sync(0xffffffffu, *s_abort, 0))
          consume_tile(P, m, sx, u, abuf, ring, full0, empty0, st, cw, lane, s_abort);
    } else {
      const float sx = __ldcg(P.head_sx);
      for (int64_t u = first; u < it.end; u += kConsumerWarps)
        if (!__shfl_sync(0xffffffffu, *s_abort, 0))
          consume_head_row(P, sx, u, abuf, ring, full0, empty0, st, cw, lane, s_abort);
    }
    st.seq += (uint32_t)(it.end - it.begin);
    buf ^= 1;
  }
  if (prefetched) cp_async_wait_all();

  if (P.has_head) {  // CTA best, then the last CTA reduces all CTAs
    if (lane == 0) hbest[cw] = HeadPartial{st.best_v, st.best_i};
    consumer_sync();
    if (threadIdx.x == 0 && !*s_abort) {
      HeadPartial b = hbest[0];
      for (int w = 1; w < kConsumerWarps; ++w)
        if (better(hbest[w].val, hbest[w].idx, b.val, b.idx)) b = hbest[w];
      P.head_ws->part[blockIdx.x] = b;
      __threadfence();
      if (atomicAdd(&P.ctrl->head_done, 1u) == gridDim.x - 1) {
        __threadfence();
        float bv = -INFINITY;
        int bi = INT_MAX;
        for (int c = 0; c < (int)gridDim.x; ++c) {
          const float pv = __ldcg(&P.head_ws->part[c].val);
          const int pi = __ldcg(&P.head_ws->part[c].idx);
          if (better(pv, pi, bv, bi)) { bv = pv; bi = pi; }
        }
        P.head_argmax[0] = bi == INT_MAX ? 0 : bi;
        P.ctrl->head_done = 0u;
      }
    }
  }
}

// ---- host: schedule --------------------------------------------------------------------
struct Unitset {
  int kind, mat;
  int64_t units;
  int64_t unit_bytes;
};

// Splits one stage's units into `grid` contiguous byte ranges and appends each CTA's items.
void partition_stage(const std::vector<Unitset>& sets, int grid, bool barrier_before,
                     std::vector<std::vector<WorkItem>>& per_cta) {
  int64_t total = 0;
  for (const Unitset& s : sets) total += s.units * s.unit_bytes;
  std::vector<bool> flagged(grid, false);
  auto push = [&](int c, const WorkItem& w) {
    WorkItem x = w;
    if (barrier_before && !flagged[c]) { x.flags |= kFlagStage; flagged[c] = true; }
    per_cta[c].push_back(x);
  };
  int64_t start = 0;  // byte offset of the current unit within the stage
  for (const Unitset& s : sets) {
    int64_t u = 0;
    while (u < s.units) {
      // owner of unit u: the CTA whose byte range holds the unit's first byte
      const int c = (int)std::min<int64_t>(grid - 1, (start + u * s.unit_bytes) * grid / std::max<int64_t>(total, 1));
      const int64_t end_byte = (int64_t)(c + 1) * total / grid;  // first byte of CTA c+1
      int64_t v = u + 1;
      while (v < s.units && start + v * s.unit_bytes < end_byte) ++v;
      push(c, WorkItem{s.kind, s.mat, 0, 0, u, v});
      u = v;
    }
    start += s.units * s.unit_bytes;
  }
  if (barrier_before)  // every CTA takes part in the barrier, with or without work
    for (int c = 0; c < grid; ++c)
      if (!flagged[c]) push(c, WorkItem{kItemTernary, 0, 0, 0, 0, 0});
}

}  // namespace

nt_status persist_prepare(nt_decode_plan* p) {
  if (p->B != 1)
    return set_error(NT_ERR_INVALID_ARG, "the persistent launcher runs batch 1; use NT_LAUNCH_GRAPH for batch > 1");
  int kmax = p->has_head ? p->head_K : 0;
  for (const MatDesc& m : p->mats) kmax = std::max<int>(kmax, (int)padded_k(m.K));
  p->act_stride = (int)padded_k(kmax);
  p->smem_bytes = kRingBytes + 2 * (size_t)p->act_stride + 2 * kBars * 8 +
                  kConsumerWarps * sizeof(HeadPartial) + kConsumerWarps * 4 + 16;
  int optin = 0;
  NT_CUDA_TRY(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, p->device));
  if (p->smem_bytes > (size_t)optin)
    return set_error(NT_ERR_INVALID_ARG, "persistent launcher: K too large for the shared-memory budget (K <= 16384)");
  NT_CUDA_TRY(cudaFuncSetAttribute(persist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p->smem_bytes));
  int per_sm = 0;
  NT_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, persist_kernel, kThreadsP, p->smem_bytes));
  if (per_sm < 1) return set_error(NT_ERR_CUDA, "persistent kernel cannot be resident on an SM");
  const int grid = p->sm_count;
  p->grid = grid;

  std::vector<std::vector<WorkItem>> per_cta(grid);
  const int n_proj = (int)p->mats.size();
  auto ternary = [&](int mi) {
    return Unitset{kItemTernary, mi, padded_rows(p->mats[mi].N) / 4, padded_k(p->mats[mi].K)};
  };
  const Unitset head{kItemHead, 0, p->head_V, p->head_K};
  int barriers = p->n_qjobs > 0 ? 1 : 0;
  if (p->mode == NT_STEP_INDEPENDENT) {
    // Each CTA gets 1/grid of the ternary bytes and 1/grid of the output table, so every
    // CTA has the same mix of decode-heavy and decode-free work.
    std::vector<Unitset> all;
    for (int i = 0; i < n_proj; ++i) all.push_back(ternary(i));
    partition_stage(all, grid, false, per_cta);
    if (p->has_head) partition_stage({head}, grid, false, per_cta);
  } else {
    bool first = true;
    for (int l = 0; l < p->n_layers; ++l) {
      const int b = l * kProjPerLayer;
      const int groups[4][2] = {{b, 3}, {b + 3, 1}, {b + 4, 2}, {b + 6, 1}};
      for (const auto& g : groups) {
        std::vector<Unitset> sets;
        for (int i = 0; i < g[1]; ++i) sets.push_back(ternary(g[0] + i));
        partition_stage(sets, grid, !first, per_cta);
        barriers += first ? 0 : 1;
        first = false;
      }
    }
    if (p->has_head) {
      partition_stage({head}, grid, true, per_cta);
      ++barriers;
    }
  }
  p->n_barriers = barriers;

  std::vector<WorkItem> items;
  std::vector<int> off(grid + 1, 0);
  for (int c = 0; c < grid; ++c) {
    off[c] = (int)items.size();
    items.insert(items.end(), per_cta[c].begin(), per_cta[c].end());
  }
  off[grid] = (int)items.size();
  const size_t item_bytes = sizeof(WorkItem) * std::max<size_t>(items.size(), 1);
  NT_CUDA_TRY(cudaMalloc(&p->d_sched, item_bytes + sizeof(int) * off.size()));
  if (!items.empty()) NT_CUDA_TRY(cudaMemcpy(p->d_sched, items.data(), sizeof(WorkItem) * items.size(), cudaMemcpyHostToDevice));
  NT_CUDA_TRY(cudaMemcpy(reinterpret_cast<uint8_t*>(p->d_sched) + item_bytes, off.data(), sizeof(int) * off.size(),
                         cudaMemcpyHostToDevice));
  p->sched_item_bytes = item_bytes;
  return NT_OK;
}

nt_status persist_launch(nt_decode_plan* p, cudaStream_t st) {
  PersistParams P{};
  P.mats = p->d_mats;
  P.items = p->d_sched;
  P.item_off = reinterpret_cast<const int*>(reinterpret_cast<const uint8_t*>(p->d_sched) + p->sched_item_bytes);
  P.qjobs = p->d_qjobs;
  P.n_qjobs = p->n_qjobs;
  P.n_barriers = p->n_barriers;
  P.ctrl = p->d_ctrl;
  P.head_T = p->head_T;
  P.head_s = p->head_s;
  P.head_q = p->head_q;
  P.head_sx = p->head_sx;
  P.head_logits = p->head_logits;
  P.head_argmax = p->head_argmax;
  P.head_ws = p->d_head_ws;
  P.head_V = p->head_V;
  P.head_K = p->head_K;
  P.has_head = p->has_head ? 1 : 0;
  P.act_stride = p->act_stride;
  P.launch_idx = (uint32_t)p->launches;
  P.barrier_extra = p->test_fault == 1 ? 1u : 0u;
  P.timeout_ns = p->timeout_ns;
  void* args[] = {&P};
  const cudaError_t e = cudaLaunchCooperativeKernel((const void*)persist_kernel, dim3(p->grid), dim3(kThreadsP), args,
                                                    p->smem_bytes, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return set_error(NT_ERR_CUDA, std::string("persistent launch: ") + cudaGetErrorString(e));
  }
  ++p->launches;
  return NT_OK;
}

}  // namespace nt
