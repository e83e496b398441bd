// nt_persist.cu -- the persistent streaming kernel: the decode step, and the standalone output
// projection.
//
// "The Neutrino Engine" (§ "A 104 microsecond floor inside a 694 microsecond step") reports
// that a decode step spent most of its time across ~120 kernel boundaries, and that a single
// fused kernel with software barriers brought similar waits back. Here one launch streams the
// whole step, and the weight stream never waits for a barrier: weights do not depend on
// activations, so the producer warp of every CTA keeps its shared-memory ring full across
// stage boundaries while only the consumer warps wait.
//
// CTA layout (one CTA per SM): CW consumer warps (16 for batch 1, 15 for batched plans) and
// one producer warp after them.
//   producer (lane w feeds consumer warp w): walks the CTA's schedule and issues one
//     cp.async.bulk per chunk (<= 4 KB of a tile or of an output-table row) of the units warp
//     w owns (units are dealt round-robin) into w's ring, completing on the slot's mbarrier;
//   consumers: wait for a chunk, decode it once and dp4a it against up to 4 activation
//     vectors held in shared memory, release the slot; per unit (4 rows of a tiled matrix, or
//     one output-table row) a warp reduction and the fp32 epilogue.
// Batches above 4 vectors take several passes over the weights (the decode + dp4a work, not
// the memory, bounds those batches). Ordered mode puts a grid-wide barrier before each stage;
// only consumers wait at it. Every wait is bounded by a %globaltimer deadline; on expiry the
// CTA records an error code, consumers walk the remaining barriers without work, and the
// producer waits (bounded) for its own copies in flight before exiting.
#include <float.h>
#include <limits.h>
#include <math.h>

#include <algorithm>
#include <mutex>
#include <string>
#include <vector>

#include "nt_step.cuh"

namespace nt {
namespace {

constexpr int kMaxSlots = 3;
constexpr int kSlotBytes = 4096;
constexpr int kPiecesPerSlot = kSlotBytes / 512;
constexpr int kChunkBatch = 4;                       // activation vectors per pass (batched)
constexpr int kConsumerBarrier = 1;                  // named barrier id
constexpr int kMaxSmem = 232448;                     // 227 KB per CTA on sm_103

// Kernel configuration: CW consumer warps and up to NBMAX activation vectors per pass. Batch 1
// runs 16 consumer warps (17 warps, registers capped at 96 by the 5 warps one SM
// sub-partition holds); batched plans need more registers for 4 vectors' accumulators and run
// 15 (16 warps, up to 128 registers), and so do chained batch-1 plans, which hold a stage input
// of up to 28 values per thread in registers while they quantize it.
template <int CW_, int NBMAX_, bool CHAINED_ = false>
struct KCfg {
  static constexpr bool CHAINED = CHAINED_;  // NT_STEP_CHAINED plans (a separate instance)
  static constexpr int CW = CW_;
  static constexpr int CT = CW * 32;       // consumer threads
  static constexpr int THREADS = CT + 32;  // + the producer warp
  static constexpr int NBMAX = NBMAX_;
  static constexpr int BARS = CW * kMaxSlots;
};
using Cfg1 = KCfg<16, 1>;
using CfgB = KCfg<15, kChunkBatch>;
using Cfg1C = KCfg<15, 1, true>;
using CfgBC = KCfg<15, kChunkBatch, true>;

enum : unsigned int { kErrFullWait = 1, kErrEmptyWait = 2, kErrGridBarrier = 3, kErrDrain = 4 };

struct PersistParams {
  const MatDesc* mats;
  const WorkItem* items;  // NULL: implicit schedule (standalone output projection)
  const int* item_off;    // [grid + 1]
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
  unsigned int* head_next;  // kItemHeadDyn: counter of handed-out rows after the fixed ones
  int head_fixed;           // kItemHeadDyn: rows each CTA takes before the counter (its own block)
  int head_dyn;             // the implicit schedule (standalone call) uses kItemHeadDyn
  int head_V, head_K;
  int has_head;
  int B;         // activation vectors
  int chunk_b;   // vectors per pass (<= kChunkBatch)
  int nslots;    // ring slots per consumer warp (<= kMaxSlots)
  int act_k;     // bytes per activation vector in shared memory
  uint32_t barrier_base;    // grid-barrier arrivals of all earlier launches on this plan (mod 2^32)
  int reset_barriers;       // single-launch steps: the barrier targets start at 0 and the CTA that
                            // finishes last zeroes the arrival counter, so every launch of the step
                            // takes the same parameters (the launch can be captured in a CUDA graph)
  uint32_t barrier_extra;  // added to every grid barrier's target (timeout-path tests)
  int no_copies;           // timeout-path tests: the producer issues nothing, so consumers time out
  uint64_t timeout_ns;
  unsigned long long* trace;  // optional timeline: [grid][n_barriers + 1][4]
  // input-table gather before quantization (embed_T == NULL: none)
  const int8_t* embed_T;
  const float* embed_s;
  int embed_V, embed_K;
  const int32_t* tokens;
  float* embed_x;
  // verify-pass acceptance after the arg-max (verify_emit == NULL: none)
  const int32_t* verify_draft;
  int32_t* verify_emit;
  int32_t* verify_n;
  // chained steps: every stage quantizes its input from the previous stages' outputs
  ChainSrc head_src;  // the output projection's input (the residual stream)
};

// One timeline stamp (thread 0 of the consumers only).
__device__ __forceinline__ void stamp(const PersistParams& P, int b, int i) {
  if (P.trace && threadIdx.x == 0)
    P.trace[((int64_t)blockIdx.x * (P.n_barriers + 1) + b) * 4 + i] = globaltimer_ns();
}

struct SmemLayout {
  int ring, act, bars, hbest, red, abort_flag, chain_s, slot_row, rec_state, total;
};

template <class C>
__host__ __device__ inline SmemLayout smem_layout(int nslots, int chunk_b, int act_k) {
  SmemLayout L;
  L.ring = 0;
  L.act = L.ring + C::CW * nslots * kSlotBytes;
  L.bars = L.act + 2 * chunk_b * act_k;
  L.hbest = L.bars + 2 * C::BARS * 8;
  L.red = L.hbest + C::CW * kStepMaxBatch * (int)sizeof(HeadPartial);
  L.abort_flag = L.red + 2 * C::CW * 4 + (C::CHAINED ? 16 : 0);  // chained: the norm factor after the warps' values
  L.chain_s = L.abort_flag + 16;
  L.slot_row = L.chain_s + kStepMaxBatch * 4;   // kItemHeadDyn: the row each ring slot holds
  // chained: CTA 0's recorded stage input still to be written out (see flush_record)
  L.rec_state = (L.slot_row + C::CW * kMaxSlots * 4 + 7) & ~7;
  L.total = L.rec_state + (C::CHAINED ? 32 : 0);
  return L;
}

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
template <class C>
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync %0, %1;" ::"n"(kConsumerBarrier), "n"(C::CT) : "memory");
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

// Sum of 4 per-lane values across the warp; row r's total lands in lanes 8r..8r+7.
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

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// ---- schedule --------------------------------------------------------------------------
__device__ __forceinline__ int item_count(const PersistParams& P) {
  if (P.items) return P.item_off[blockIdx.x + 1] - P.item_off[blockIdx.x];
  return (P.B + P.chunk_b - 1) / P.chunk_b;  // implicit: one item per pass
}

// Item i of this CTA. The implicit schedule (standalone output projection) gives CTA c the
// rows [c V / grid, (c+1) V / grid) once per pass of chunk_b vectors.
__device__ __forceinline__ WorkItem get_item(const PersistParams& P, int i) {
  if (P.items) return P.items[P.item_off[blockIdx.x] + i];
  WorkItem w;
  w.kind = P.head_dyn ? kItemHeadDyn : kItemHead;
  w.mat = 0;
  w.flags = 0;
  w.b0 = i * P.chunk_b;
  w.begin = P.head_dyn ? 0 : (int64_t)blockIdx.x * P.head_V / gridDim.x;
  w.end = P.head_dyn ? P.head_V : (int64_t)(blockIdx.x + 1) * P.head_V / gridDim.x;
  return w;
}

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

// First unit of an item that consumer warp w owns (units are dealt round-robin by their
// sequence number within the CTA).
template <class C>
__device__ __forceinline__ int64_t first_unit(const WorkItem& it, uint32_t seq, int w) {
  return it.begin + (int64_t)((w - (int)(seq % C::CW) + C::CW) % C::CW);
}

// ---- producer ------------------------------------------------------------------------
// Lane w of the producer warp feeds consumer warp w's ring.
template <class C>
__device__ void producer(const PersistParams& P, int n_items, uint8_t* ring, uint32_t full0,
                         uint32_t empty0, volatile int* s_abort, int* slot_row, int w) {
  const uint64_t pol = evict_first_policy();
  const uint32_t ring_w = smem_addr(ring) + (uint32_t)(w * P.nslots * kSlotBytes);
  const uint32_t full_w = full0 + 8u * w * kMaxSlots, empty_w = empty0 + 8u * w * kMaxSlots;
  int* rows_w = slot_row + w * kMaxSlots;
  uint32_t slot = 0, phase = 0, issued = 0, seq = 0;
  bool ok = !P.no_copies;
  // Copies unit u (ub bytes at base + u * ub) chunk by chunk into this lane's ring; with a row
  // index (kItemHeadDyn) the consumer learns which row each slot holds from rows_w.
  auto issue_unit = [&](const uint8_t* base, int ub, int64_t u, int row) {
    const uint8_t* src = base + u * (int64_t)ub;
    for (int off = 0; off < ub && ok; off += kSlotBytes) {
      const uint32_t bytes = (uint32_t)min(kSlotBytes, ub - off);
      if (!wait_phase(empty_w + 8 * slot, phase ^ 1u, P.timeout_ns, P.ctrl, s_abort)) {
        if (!*s_abort) record_error(P.ctrl, kErrEmptyWait, s_abort);
        ok = false;
        break;
      }
      rows_w[slot] = row;  // ordered before the consumer's wait by the arrive's release
      mbar_expect_tx(full_w + 8 * slot, bytes);
      bulk_load(ring_w + slot * kSlotBytes, src + off, bytes, full_w + 8 * slot, pol);
      ++issued;
      if (++slot == (uint32_t)P.nslots) { slot = 0; phase ^= 1u; }
    }
  };
  for (int i = 0; i < n_items && ok; ++i) {
    const WorkItem it = get_item(P, i);
    const uint8_t* base;
    int ub;
    unit_geometry(P, it, base, ub);
    if (it.kind == kItemHeadDyn) {  // always a CTA's last item
      // this CTA's own block of fixed rows first (issued before the previous kernel has finished,
      // for the standalone call), then CW rows per grab, one per lane, until the table is done
      const int64_t f0 = (int64_t)blockIdx.x * P.head_fixed;
      for (int64_t r = f0 + w; r < f0 + P.head_fixed && ok; r += C::CW) issue_unit(base, ub, r, (int)r);
      asm volatile("griddepcontrol.wait;" ::: "memory");  // the counter is the previous call's until it ends
      const int64_t dyn0 = (int64_t)gridDim.x * P.head_fixed;
      constexpr unsigned int kLanes = (1u << C::CW) - 1u;
      for (;;) {
        unsigned int g = 0;
        if (w == 0) g = atomicAdd(P.head_next, (unsigned int)C::CW);
        g = __shfl_sync(kLanes, g, 0);
        if (dyn0 + (int64_t)g >= it.end || !__all_sync(kLanes, ok)) break;
        const int64_t r = dyn0 + (int64_t)g + w;
        if (r < it.end) issue_unit(base, ub, r, (int)r);
      }
      // end of the stream: a slot whose row is -1, its phase completed by a plain arrival
      if (ok && wait_phase(empty_w + 8 * slot, phase ^ 1u, P.timeout_ns, P.ctrl, s_abort)) {
        rows_w[slot] = -1;
        mbar_arrive(full_w + 8 * slot);
        ++issued;  // the drain below treats it as this slot's last use (its phase is complete)
        if (++slot == (uint32_t)P.nslots) { slot = 0; phase ^= 1u; }
      } else if (ok) {
        if (!*s_abort) record_error(P.ctrl, kErrEmptyWait, s_abort);
        ok = false;
      }
      continue;
    }
    for (int64_t u = first_unit<C>(it, seq, w); u < it.end && ok; u += C::CW) issue_unit(base, ub, u, 0);
    seq += (uint32_t)(it.end - it.begin);
  }
  // Drain: every slot's last copy must have landed before this thread (and so the CTA)
  // may exit, whatever happened to the consumers.
  for (uint32_t s = 0; s < (uint32_t)P.nslots; ++s) {
    if (issued <= s) continue;
    const uint32_t parity = ((issued - 1 - s) / (uint32_t)P.nslots) & 1u;
    const uint32_t bar = full_w + 8 * s;
    if (mbar_try_wait(bar, parity)) continue;
    const uint64_t deadline = globaltimer_ns() + P.timeout_ns;
    while (!mbar_try_wait(bar, parity)) {
      if (globaltimer_ns() > deadline) {
        record_error(P.ctrl, kErrDrain, s_abort);
        break;
      }
    }
  }
}

// ---- consumers -----------------------------------------------------------------------
struct Ring {
  uint8_t* base;  // this warp's first slot
  uint32_t full, empty;
  uint32_t slot, phase;
  int nslots;
};

// A consumer warp's wait for its next chunk: every lane waits (each observes the mbarrier
// phase, which makes the bulk copy's bytes visible to it) and the outcome is made
// warp-uniform, so no lane leaves while others go on to warp-wide shuffles.
__device__ __forceinline__ const uint8_t* wait_chunk(const PersistParams& P, Ring& r, int lane,
                                                     volatile int* s_abort) {
  const bool ok = __all_sync(0xffffffffu, wait_phase(r.full + 8 * r.slot, r.phase, P.timeout_ns,
                                                     P.ctrl, s_abort));
  if (!ok) {
    if (lane == 0 && !*s_abort) record_error(P.ctrl, kErrFullWait, s_abort);
    return nullptr;
  }
  return r.base + r.slot * kSlotBytes;
}

__device__ __forceinline__ void release_chunk(Ring& r, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(r.empty + 8 * r.slot);
  if (++r.slot == (uint32_t)r.nslots) { r.slot = 0; r.phase ^= 1u; }
}

// Quantize one fp32 vector with the consumer threads: s = fl(max|x| / 127), q[k] =
// clamp(rint(fl(x[k] / s)), -127, 127), in two passes over x (the second from L2). x is read
// through L2: the input-table rows that other CTAs wrote earlier in the same launch are
// quantized here.
template <class C>
__device__ void quantize_consumers(const float* x, int K, int8_t* q, float* s_out, float* red) {
  const int t = threadIdx.x;
  float m = 0.0f;
  for (int k = t; k < K; k += C::CT) m = fmaxf(m, fabsf(__ldcg(x + k)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((t & 31) == 0) red[t >> 5] = m;
  consumer_sync<C>();
  m = red[0];
#pragma unroll
  for (int i = 1; i < C::CW; ++i) m = fmaxf(m, red[i]);
  const bool nz = m != 0.0f;
  const float s = nz ? __fdiv_rn(m, 127.0f) : 0.0f;
  if (t == 0) *s_out = s;
  for (int k = t; k < K; k += C::CT) q[k] = (int8_t)quant_byte(__ldcg(x + k), s, nz);
  consumer_sync<C>();  // red[] reuse
}

// Register-resident vectors of the first phase: up to 4 * kPer * CT values (at least 12,288),
// thread t holding the float4 groups at 4t + 4 CT i.
template <class C>
struct QRegs {
  static constexpr int kPer = (12288 + 4 * C::CT - 1) / (4 * C::CT);
  float4 v[kPer];
};
template <class C>
__device__ __forceinline__ bool qregs_fit(const QuantJob& j) {
  return j.B == 1 && j.K <= 4 * QRegs<C>::kPer * C::CT &&
         ((reinterpret_cast<uintptr_t>(j.x) & 15) | (reinterpret_cast<uintptr_t>(j.q) & 3) | (j.K & 3)) == 0;
}
template <class C>
__device__ __forceinline__ void qregs_load(const QuantJob& j, QRegs<C>& r) {
#pragma unroll
  for (int i = 0; i < QRegs<C>::kPer; ++i) {
    const int k = 4 * threadIdx.x + 4 * C::CT * i;
    r.v[i] = k < j.K ? __ldcg(reinterpret_cast<const float4*>(j.x + k)) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}
// The scale and codes of one register-resident vector; red2 holds CW floats and is reused two
// vectors later, so one consumer barrier per vector suffices.
template <class C>
__device__ __forceinline__ void qregs_quantize(const QuantJob& j, const QRegs<C>& r, float* red2) {
  const int t = threadIdx.x;
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < QRegs<C>::kPer; ++i)
    m = fmaxf(fmaxf(m, fmaxf(fabsf(r.v[i].x), fabsf(r.v[i].y))), fmaxf(fabsf(r.v[i].z), fabsf(r.v[i].w)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((t & 31) == 0) red2[t >> 5] = m;
  consumer_sync<C>();
  m = red2[0];
#pragma unroll
  for (int i = 1; i < C::CW; ++i) m = fmaxf(m, red2[i]);
  const bool nz = m != 0.0f;
  const float s = nz ? __fdiv_rn(m, 127.0f) : 0.0f;
  if (t == 0) *j.s = s;
#pragma unroll
  for (int i = 0; i < QRegs<C>::kPer; ++i) {
    const int k = 4 * t + 4 * C::CT * i;
    if (k < j.K) *reinterpret_cast<uint32_t*>(j.q + k) = quant4(r.v[i], s, nz);
  }
}

// The step's first phase: this CTA's quantization jobs j = blockIdx.x + r * gridDim.x (a job
// with B = 0 ends the list), one vector each; vectors that do not fit the registers take the
// two-pass path. (Loading the next vector into a second register set while one is converted
// shortened this phase by ~1 us but made the rest of the kernel's code slower in ordered
// steps, ~28 us per token.)
template <class C>
__device__ void quantize_phase(const PersistParams& P, float* red) {
  int par = 0;
  for (int j = blockIdx.x; j < P.n_qjobs; j += gridDim.x) {
    const QuantJob cur = P.qjobs[j];
    if (cur.B == 0) break;
    if (qregs_fit<C>(cur)) {
      QRegs<C> a;
      qregs_load<C>(cur, a);
      qregs_quantize<C>(cur, a, red + par * C::CW);
      par ^= 1;
    } else {
      consumer_sync<C>();  // red[] may still be read for the previous vector
      for (int v = 0; v < cur.B; ++v)
        quantize_consumers<C>(cur.x + (int64_t)v * cur.K, cur.K, cur.q + (int64_t)v * cur.K, cur.s + v, red);
    }
  }
  consumer_sync<C>();
}

// Input-table row of token b, dequantized into embed_x[b] by the consumer threads:
// x[k] = fl((float)T[tok][k] * s[tok]); a token outside [0, V) gives a zero row.
template <class C>
__device__ void embed_row_consumers(const PersistParams& P, int b) {
  const int t = P.tokens[b];
  const bool ok = t >= 0 && t < P.embed_V;
  const float sc = ok ? P.embed_s[t] : 0.0f;
  float4* out = reinterpret_cast<float4*>(P.embed_x + (int64_t)b * P.embed_K);
  for (int g = threadIdx.x; g < P.embed_K / 16; g += C::CT) {
    uint4 v = make_uint4(0, 0, 0, 0);
    if (ok) v = __ldg(reinterpret_cast<const uint4*>(P.embed_T + (int64_t)t * P.embed_K) + g);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int8_t* c = reinterpret_cast<const int8_t*>(&w[i]);
      out[4 * g + i] = make_float4(__fmul_rn((float)c[0], sc), __fmul_rn((float)c[1], sc),
                                   __fmul_rn((float)c[2], sc), __fmul_rn((float)c[3], sc));
    }
  }
}

// Chained steps: quantizes the stage input of vectors b0 .. b0+nb-1 straight into this CTA's
// activation buffer; every CTA computes the same codes from the same fp32 values, read
// through L2. The scales go to s_chain. With `record` (CTA 0) the codes and scales are also
// written to the q / s_x of the stage's matrices (rec[0..n_rec)) or of the output projection.
template <class C>
__device__ void chain_prologue(const ChainSrc& cs, int b0, int nb, int act_k, uint8_t* abuf, float* s_chain,
                               float* red, bool record, const MatDesc* rec, int n_rec, int8_t* hq, float* hs) {
  const int t = threadIdx.x;
  // the value quantized at k: the stage input, RMS-normalised with gamma when the source has
  // one (fl(fl(v * r) * gamma[k]), r = fl32(1 / sqrt(mean(v^2) + eps)): the squares summed in
  // fp32 within each warp, the warps' sums added and r formed in double by one thread)
  auto value4 = [&](int b, int k, float r) {
    float4 v = chain_load4(cs, b, k);
    if (cs.gamma) {
      const float4 g = __ldg(reinterpret_cast<const float4*>(cs.gamma + k));
      v = make_float4(__fmul_rn(__fmul_rn(v.x, r), g.x), __fmul_rn(__fmul_rn(v.y, r), g.y),
                      __fmul_rn(__fmul_rn(v.z, r), g.z), __fmul_rn(__fmul_rn(v.w, r), g.w));
    }
    return v;
  };
  // Vectors of up to 4 * kPer * CT values (13,440 at batch 1) stay in registers: one pass of
  // loads through L2, the reductions and the codes from the registers.
  constexpr int kPer = C::NBMAX == 1 ? 7 : 2;
  if (cs.K <= 4 * kPer * C::CT) {
    for (int b = 0; b < nb; ++b) {
      float4 v[kPer];
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int k = 4 * t + 4 * C::CT * i;
        v[i] = k < cs.K ? chain_load4(cs, b0 + b, k) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      if (cs.gamma) {
        float sf = 0.0f;
#pragma unroll
        for (int i = 0; i < kPer; ++i)
          sf = fmaf(v[i].x, v[i].x, fmaf(v[i].y, v[i].y, fmaf(v[i].z, v[i].z, fmaf(v[i].w, v[i].w, sf))));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sf += __shfl_xor_sync(0xffffffffu, sf, o);
        if ((t & 31) == 0) red[t >> 5] = sf;
        consumer_sync<C>();
        if (t == 0) {  // the warps' sums added in double by one thread; r broadcast in red[CW]
          double tot = 0.0;
          for (int i = 0; i < C::CW; ++i) tot += red[i];
          red[C::CW] = (float)(1.0 / sqrt(tot / cs.K + (double)cs.eps));
        }
        consumer_sync<C>();
        const float r = red[C::CW];
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int k = 4 * t + 4 * C::CT * i;
          if (k < cs.K) {
            const float4 g = __ldg(reinterpret_cast<const float4*>(cs.gamma + k));
            v[i] = make_float4(__fmul_rn(__fmul_rn(v[i].x, r), g.x), __fmul_rn(__fmul_rn(v[i].y, r), g.y),
                               __fmul_rn(__fmul_rn(v[i].z, r), g.z), __fmul_rn(__fmul_rn(v[i].w, r), g.w));
          }
        }
      }
      float m = 0.0f;
#pragma unroll
      for (int i = 0; i < kPer; ++i)
        m = fmaxf(fmaxf(m, fmaxf(fabsf(v[i].x), fabsf(v[i].y))), fmaxf(fabsf(v[i].z), fabsf(v[i].w)));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if ((t & 31) == 0) red[t >> 5] = m;
      consumer_sync<C>();
      m = red[0];
#pragma unroll
      for (int i = 1; i < C::CW; ++i) m = fmaxf(m, red[i]);
      const bool nz = m != 0.0f;
      const float s = nz ? __fdiv_rn(m, 127.0f) : 0.0f;
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int k = 4 * t + 4 * C::CT * i;
        if (k < cs.K) {
          const uint32_t c = quant4(v[i], s, nz);
          *reinterpret_cast<uint32_t*>(abuf + b * act_k + k) = c;
          if (record) {
            const int64_t o = (int64_t)(b0 + b) * cs.K + k;
            if (cs.cap) *reinterpret_cast<float4*>(cs.cap + o) = v[i];
            if (hq) *reinterpret_cast<uint32_t*>(hq + o) = c;
            for (int rr = 0; rr < n_rec; ++rr) *reinterpret_cast<uint32_t*>(const_cast<int8_t*>(rec[rr].q) + o) = c;
          }
        }
      }
      if (t == 0) {
        s_chain[b] = s;
        if (record) {
          if (hs) hs[b0 + b] = s;
          for (int rr = 0; rr < n_rec; ++rr) const_cast<float*>(rec[rr].s_x)[b0 + b] = s;
        }
      }
      consumer_sync<C>();  // red[] is reused by the next vector
    }
    return;
  }
  for (int b = 0; b < nb; ++b) {
    float r = 1.0f;
    if (cs.gamma) {
      float sf = 0.0f;  // this thread's few squares in fp32 (FP64 is slow on this part)
      for (int k = 4 * t; k < cs.K; k += 4 * C::CT) {
        const float4 v = chain_load4(cs, b0 + b, k);
        sf = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, sf))));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sf += __shfl_xor_sync(0xffffffffu, sf, o);
      if ((t & 31) == 0) red[t >> 5] = sf;
      consumer_sync<C>();
      if (t == 0) {  // the warps' sums added in double by one thread; r broadcast in red[CW]
        double tot = 0.0;
        for (int i = 0; i < C::CW; ++i) tot += red[i];
        red[C::CW] = (float)(1.0 / sqrt(tot / cs.K + (double)cs.eps));
      }
      consumer_sync<C>();
      r = red[C::CW];
    }
    float m = 0.0f;
    for (int k = 4 * t; k < cs.K; k += 4 * C::CT) {
      const float4 v = value4(b0 + b, k, r);
      m = fmaxf(fmaxf(m, fmaxf(fabsf(v.x), fabsf(v.y))), fmaxf(fabsf(v.z), fabsf(v.w)));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((t & 31) == 0) red[t >> 5] = m;
    consumer_sync<C>();
    m = red[0];
#pragma unroll
    for (int i = 1; i < C::CW; ++i) m = fmaxf(m, red[i]);
    const bool nz = m != 0.0f;
    const float s = nz ? __fdiv_rn(m, 127.0f) : 0.0f;
    for (int k = 4 * t; k < cs.K; k += 4 * C::CT) {
      const float4 v = value4(b0 + b, k, r);
      const uint32_t c = quant4(v, s, nz);
      *reinterpret_cast<uint32_t*>(abuf + b * act_k + k) = c;
      if (record) {
        const int64_t o = (int64_t)(b0 + b) * cs.K + k;
        if (cs.cap) *reinterpret_cast<float4*>(cs.cap + o) = v;
        if (hq) *reinterpret_cast<uint32_t*>(hq + o) = c;
        for (int r = 0; r < n_rec; ++r) *reinterpret_cast<uint32_t*>(const_cast<int8_t*>(rec[r].q) + o) = c;
      }
    }
    if (t == 0) {
      s_chain[b] = s;
      if (record) {
        if (hs) hs[b0 + b] = s;
        for (int r = 0; r < n_rec; ++r) const_cast<float*>(rec[r].s_x)[b0 + b] = s;
      }
    }
    consumer_sync<C>();  // red[] is reused by the next vector
  }
}

// Grid-wide barrier among the consumers of all CTAs; `target` counts arrivals modulo 2^32.
template <class C>
__device__ void grid_barrier(const PersistParams& P, uint32_t target, int b, volatile int* s_abort) {
  target += P.barrier_extra;
  consumer_sync<C>();
  stamp(P, b, 0);
  if (threadIdx.x == 0 && !*s_abort) {
    // the consumer barrier above orders every thread's writes before this release (cumulative)
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
  stamp(P, b, 1);
  consumer_sync<C>();
}

// Copies nb activation vectors of K bytes (vector b at src + b*K) into shared memory at
// stride act_k, synchronously or with cp.async.
template <class C>
__device__ void load_act(uint8_t* dst, const int8_t* src, int K, int nb, int act_k, bool async) {
  const int per = K / 16;
  for (int i = threadIdx.x; i < per * nb; i += C::CT) {
    const int b = i / per, o = (i - b * per) * 16;
    if (async) cp_async16(smem_addr(dst + b * act_k + o), src + (int64_t)b * K + o);
    else *reinterpret_cast<uint4*>(dst + b * act_k + o) = __ldcg(reinterpret_cast<const uint4*>(src + (int64_t)b * K + o));
  }
  if (async) cp_async_commit();
}

__device__ __forceinline__ const int8_t* item_act(const PersistParams& P, const WorkItem& it, int& K, int& nb) {
  nb = min(P.chunk_b, P.B - it.b0);
  if (it.kind == kItemTernary) {
    K = P.mats[it.mat].K;
    return P.mats[it.mat].q + (int64_t)it.b0 * K;
  }
  K = P.head_K;
  return P.head_q + (int64_t)it.b0 * K;
}

// 16 bytes of one lane in one 512-byte piece (4 rows x 16 trits), decoded once and dotted
// with NB activation vectors (stride act_k in shared memory).
template <int NB>
__device__ __forceinline__ void tile_piece(const uint8_t* sb, const uint8_t* ab, int act_k, int (&acc)[NB][4]) {
  const uint4 wv = lds128(sb);
  const Trits16 d0 = tiled_word_decode(wv.x), d1 = tiled_word_decode(wv.y);
  const Trits16 d2 = tiled_word_decode(wv.z), d3 = tiled_word_decode(wv.w);
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const uint4 a = lds128(ab + b * act_k);
    acc[b][0] = trits16_dot(d0, a.x, a.y, a.z, a.w, acc[b][0]);
    acc[b][1] = trits16_dot(d1, a.x, a.y, a.z, a.w, acc[b][1]);
    acc[b][2] = trits16_dot(d2, a.x, a.y, a.z, a.w, acc[b][2]);
    acc[b][3] = trits16_dot(d3, a.x, a.y, a.z, a.w, acc[b][3]);
  }
}

// 16 bytes of one lane of an output-table row against NB activation vectors.
template <int NB>
__device__ __forceinline__ void row_piece(const uint8_t* sb, const uint8_t* ab, int act_k, int (&acc)[NB][2], int h) {
  const uint4 t = lds128(sb);
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const uint4 a = lds128(ab + b * act_k);
    int s = acc[b][h];
    s = dp4a(t.x, a.x, s);
    s = dp4a(t.y, a.y, s);
    s = dp4a(t.z, a.z, s);
    s = dp4a(t.w, a.w, s);
    acc[b][h] = s;
  }
}

// One tile (4 rows) of a tiled ternary matrix against NB activation vectors. The row scale
// is loaded before the first chunk so its latency hides behind the chunk work.
// The fields of a matrix descriptor a tile's consumer needs. Chained steps load them before
// the stage's grid barrier, so the load's latency overlaps the wait (9 us per token); the
// other instances load the descriptor after it (doing the same there compiled into slower
// stage code for ordered steps).
struct TileDesc {
  const float* s_w;
  float* y;
  const float* res_in;
  float* res_out;
  int N, K;
};
template <int NB, bool CH, class M>
__device__ __forceinline__ void consume_tile(const PersistParams& P, const M& m, const float (&sx)[NB], int b0,
                             int64_t tile, const uint8_t* act, Ring& ring, int lane, volatile int* s_abort) {
  const int pieces = (int)(padded_k(m.K) / 512);
  const int64_t n = tile * 4 + (lane >> 3);
  const float sw = ((lane & 7) == 0 && n < m.N) ? __ldg(m.s_w + n) : 0.0f;
  float rin[NB];  // chained: the residual stream's values, loaded early like the row scale
  if constexpr (CH) {
#pragma unroll
    for (int b = 0; b < NB; ++b)
      rin[b] = (m.res_out && (lane & 7) == 0 && n < m.N) ? __ldcg(m.res_in + (int64_t)(b0 + b) * m.N + n) : 0.0f;
  }
  int acc[NB][4];
#pragma unroll
  for (int b = 0; b < NB; ++b) acc[b][0] = acc[b][1] = acc[b][2] = acc[b][3] = 0;
  for (int p0 = 0; p0 < pieces; p0 += kPiecesPerSlot) {
    const uint8_t* slot = wait_chunk(P, ring, lane, s_abort);
    if (!slot) return;
    const uint8_t* sb = slot + lane * 16;
    const uint8_t* ab = act + (p0 * 32 + lane) * 16;
    if (pieces - p0 >= kPiecesPerSlot) {  // full chunk: branch-free, so loads can run ahead
#pragma unroll
      for (int p = 0; p < kPiecesPerSlot; ++p) tile_piece<NB>(sb + p * 512, ab + p * 512, P.act_k, acc);
    } else {
      for (int p = 0; p < pieces - p0; ++p) tile_piece<NB>(sb + p * 512, ab + p * 512, P.act_k, acc);
    }
    release_chunk(ring, lane);
  }
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const int total = warp_sum4(acc[b][0], acc[b][1], acc[b][2], acc[b][3], lane);
    if ((lane & 7) == 0 && n < m.N) {
      const int64_t o = (int64_t)(b0 + b) * m.N + n;
      const float yv = scale_out(total, sw, sx[b]);
      m.y[o] = yv;
      if constexpr (CH) {  // chained: the residual stream
        if (m.res_out) m.res_out[o] = __fadd_rn(rin[b], yv);
      }
    }
  }
}

// One row of the int8 output table against NB activation vectors; lane 0 keeps each
// vector's best (logit, row) for this warp in shared memory.
template <int NB>
__device__ __forceinline__ void consume_head_row(const PersistParams& P, const float (&sx)[NB], int b0, int64_t v,
                                 const uint8_t* act, Ring& ring, HeadPartial* wbest, int lane,
                                 volatile int* s_abort) {
  const float sv = lane == 0 ? __ldg(P.head_s + v) : 0.0f;
  int acc[NB][2];
#pragma unroll
  for (int b = 0; b < NB; ++b) acc[b][0] = acc[b][1] = 0;
  for (int off = 0; off < P.head_K; off += kSlotBytes) {
    const int cb = min(kSlotBytes, P.head_K - off);
    const uint8_t* slot = wait_chunk(P, ring, lane, s_abort);
    if (!slot) return;
    const uint8_t* sb = slot + lane * 16;
    const uint8_t* ab = act + off + lane * 16;
    if (cb == kSlotBytes) {  // full chunk: branch-free
#pragma unroll
      for (int p = 0; p < kPiecesPerSlot; ++p) row_piece<NB>(sb + p * 512, ab + p * 512, P.act_k, acc, p & 1);
    } else {
      for (int p = 0; p * 512 + lane * 16 < cb; ++p) row_piece<NB>(sb + p * 512, ab + p * 512, P.act_k, acc, 0);
    }
    release_chunk(ring, lane);
  }
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const int total = warp_sum(acc[b][0] + acc[b][1]);
    if (lane == 0) {
      const float lg = scale_out(total, sv, sx[b]);
      if (P.head_logits) P.head_logits[(int64_t)(b0 + b) * P.head_V + v] = lg;
      HeadPartial& hb = wbest[b0 + b];
      if (better(lg, (int)v, hb.val, hb.idx)) hb = HeadPartial{lg, (int)v};
    }
  }
}

template <class C, int NB>
__device__ __forceinline__ void consume_item(const PersistParams& P, const WorkItem& it, uint32_t seq, const uint8_t* act,
                             Ring& ring, HeadPartial* wbest, int cw, int lane, volatile int* s_abort,
                             const float* s_chain, const int* slot_row, const TileDesc& pre, float sx_pre) {
  float sx[NB];
  const float* sxp = it.kind == kItemTernary ? P.mats[it.mat].s_x : P.head_sx;
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    if constexpr (C::CHAINED) sx[b] = s_chain[b];
    else if (C::NBMAX == 1 && it.kind == kItemTernary) sx[b] = sx_pre;
    else sx[b] = __ldcg(sxp + it.b0 + b);
  }
  const int64_t first = first_unit<C>(it, seq, cw);
  // The abort flag is read by lane 0 and broadcast, so the whole warp takes one branch.
  if (it.kind == kItemTernary) {
    if constexpr (C::CHAINED) {
      for (int64_t u = first; u < it.end; u += C::CW)
        if (!__shfl_sync(0xffffffffu, *s_abort, 0))
          consume_tile<NB, C::CHAINED>(P, pre, sx, it.b0, u, act, ring, lane, s_abort);
    } else {
      const MatDesc m = P.mats[it.mat];
      for (int64_t u = first; u < it.end; u += C::CW)
        if (!__shfl_sync(0xffffffffu, *s_abort, 0))
          consume_tile<NB, C::CHAINED>(P, m, sx, it.b0, u, act, ring, lane, s_abort);
    }
  } else if (it.kind == kItemHeadDyn) {
    // rows in the order the producer lane handed them out; the slot of a row's first chunk
    // names it, and a slot naming row -1 ends the stream
    const int* rows = slot_row + cw * kMaxSlots;
    for (;;) {
      if (__shfl_sync(0xffffffffu, *s_abort, 0)) break;
      if (wait_chunk(P, ring, lane, s_abort) == nullptr) break;  // a wait ran out
      const int r = rows[ring.slot];
      if (r < 0) break;
      consume_head_row<NB>(P, sx, it.b0, r, act, ring, wbest, lane, s_abort);  // its first wait returns at once
    }
  } else {
    for (int64_t u = first; u < it.end; u += C::CW)
      if (!__shfl_sync(0xffffffffu, *s_abort, 0))
        consume_head_row<NB>(P, sx, it.b0, u, act, ring, wbest, lane, s_abort);
  }
}

// Chained steps: CTA 0 writes the codes and scales of a stage input it quantized (still in its
// activation buffer and s_chain) to the q / s_x of the stage's matrices or of the output
// projection once its own share of the stage is done, so the writes do not delay the work
// that every other CTA waits for at the next grid barrier (written in the prologue, they made
// CTA 0 the last to arrive at most barriers: chained batch-1 steps 1,122 -> 1,103 us per token).
template <class C>
__device__ void flush_record(const uint8_t* abuf, const float* s_chain, int act_k, int K, int b0, int nb,
                             const MatDesc* rec, int n_rec, int8_t* hq, float* hs) {
  for (int b = 0; b < nb; ++b) {
    for (int k = 4 * (int)threadIdx.x; k < K; k += 4 * C::CT) {
      const uint32_t c = *reinterpret_cast<const uint32_t*>(abuf + b * act_k + k);
      const int64_t o = (int64_t)(b0 + b) * K + k;
      if (hq) *reinterpret_cast<uint32_t*>(hq + o) = c;
      for (int rr = 0; rr < n_rec; ++rr) *reinterpret_cast<uint32_t*>(const_cast<int8_t*>(rec[rr].q) + o) = c;
    }
    if (threadIdx.x == 0) {
      const float sv = s_chain[b];
      if (hs) hs[b0 + b] = sv;
      for (int rr = 0; rr < n_rec; ++rr) const_cast<float*>(rec[rr].s_x)[b0 + b] = sv;
    }
  }
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1) persist_kernel(const __grid_constant__ PersistParams P) {
  extern __shared__ __align__(128) uint8_t smem[];
  const SmemLayout L = smem_layout<C>(P.nslots, P.chunk_b, P.act_k);
  uint8_t* ring = smem + L.ring;
  uint8_t* act = smem + L.act;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  HeadPartial* hbest = reinterpret_cast<HeadPartial*>(smem + L.hbest);  // [warp][kStepMaxBatch]
  float* red = reinterpret_cast<float*>(smem + L.red);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L.abort_flag);
  float* s_chain = reinterpret_cast<float*>(smem + L.chain_s);
  int* slot_row = reinterpret_cast<int*>(smem + L.slot_row);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full0 = smem_addr(bars), empty0 = smem_addr(bars + C::BARS);
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::BARS; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, 1);
    }
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int i = threadIdx.x; i < C::CW * kStepMaxBatch; i += blockDim.x)
    hbest[i] = HeadPartial{-INFINITY, INT_MAX};
  __syncthreads();

  const int n_items = item_count(P);
  stamp(P, 0, 0);
  if (warp == C::CW) {
    if (lane < C::CW) producer<C>(P, n_items, ring, full0, empty0, s_abort, slot_row, lane);
    return;
  }

  // ---- consumers ----
  // Every consumer warp walks the same sequence of named and grid barriers whatever
  // happens; after an abort (s_abort) they only skip the work, so no barrier is left short.
  // Launched as a programmatic dependent (the standalone output projection), the producer
  // streams weights at once while the consumers wait here for the previous kernel: nothing
  // below reads an input or writes an output before this point.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the standalone call lets the next kernel's CTAs take each SM as this kernel's CTA leaves it
  if (!P.items) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0 && *reinterpret_cast<volatile unsigned int*>(&P.ctrl->error))
    *s_abort = 1;  // an earlier wait that ran out poisons the control word until it is cleared
  consumer_sync<C>();
  const int cw = warp;
  Ring rg{ring + cw * P.nslots * kSlotBytes, full0 + 8u * cw * kMaxSlots, empty0 + 8u * cw * kMaxSlots,
          0u, 0u, P.nslots};
  HeadPartial* wbest = hbest + cw * kStepMaxBatch;
  const uint32_t barrier_base = P.barrier_base;
  uint32_t barriers = 0, seq = 0;

  if (P.embed_T) {  // input-table rows of the step's tokens; quantization may read them
    for (int b = blockIdx.x; b < P.B; b += gridDim.x) embed_row_consumers<C>(P, b);
    if (P.n_qjobs > 0 || C::CHAINED) {
      ++barriers;
      grid_barrier<C>(P, barrier_base + barriers * gridDim.x, (int)barriers, s_abort);
      stamp(P, (int)barriers, 2);
    }
  }

  if (!C::CHAINED && P.n_qjobs > 0) {  // quantize the step's fp32 inputs, then wait for every CTA
    if constexpr (!C::CHAINED) quantize_phase<C>(P, red);
    ++barriers;
    grid_barrier<C>(P, barrier_base + barriers * gridDim.x, (int)barriers, s_abort);
    stamp(P, (int)barriers, 2);
  }

  const int act_buf = P.chunk_b * P.act_k;
  int buf = 0;
  bool prefetched = false;
  const float* chain_in0 = nullptr;  // chained: the stage input now in act[buf]
  int chain_b0 = -1;
  // chained, CTA 0: the recorded stage input waiting to be written out, in shared memory
  // (K, b0, nb, buffer, matrix count, output projection?; then the first matrix; K = 0: none)
  volatile int* s_rec = reinterpret_cast<volatile int*>(smem + L.rec_state);
  const MatDesc** s_rec_mats = reinterpret_cast<const MatDesc**>(smem + L.rec_state + 24);
  if (C::CHAINED && threadIdx.x == 0) s_rec[0] = 0;
  auto flush = [&]() {
    if constexpr (C::CHAINED && C::NBMAX == 1) {  // (the batched instance spilled registers with it)
      if (blockIdx.x == 0 && s_rec[0] > 0) {
        const bool hd = s_rec[5] != 0;
        flush_record<C>(act + s_rec[3] * act_buf, s_chain, P.act_k, s_rec[0], s_rec[1], s_rec[2], *s_rec_mats,
                        s_rec[4], hd ? const_cast<int8_t*>(P.head_q) : nullptr,
                        hd ? const_cast<float*>(P.head_sx) : nullptr);
        consumer_sync<C>();  // every thread has read the state before thread 0 clears it
        if (threadIdx.x == 0) s_rec[0] = 0;
      }
    }
  };
  for (int i = 0; i < n_items; ++i) {
    const WorkItem it = get_item(P, i);
    const bool staged = (it.flags & kFlagStage) != 0;
    TileDesc pre{};
    if constexpr (C::CHAINED) {
      if (it.kind == kItemTernary) {
        const MatDesc* md = P.mats + it.mat;
        pre = TileDesc{md->s_w, md->y, md->res_in, md->res_out, md->N, md->K};
      }
    }
    // supplied inputs: where the next item's activations come from (its work item and matrix
    // descriptor, two dependent loads), read before this item's barrier so that the prefetch
    // below is issued as soon as the item starts (ordered steps 847 -> 825 us per token; the
    // activation scale read early as well: 829 -> 794)
    int K2 = 0, nb2 = 0;
    const int8_t* q2 = nullptr;
    float sx_pre = 0.0f;  // batch 1: this item's activation scale, read before the barrier too
    if constexpr (!C::CHAINED && C::NBMAX == 1) {  // (the batched instance ran slower with it)
      if (i + 1 < n_items) q2 = item_act(P, get_item(P, i + 1), K2, nb2);
      if (it.kind == kItemTernary) sx_pre = __ldcg(P.mats[it.mat].s_x + it.b0);
    }
    if (staged) {
      flush();
      ++barriers;
      grid_barrier<C>(P, barrier_base + barriers * gridDim.x, (int)barriers, s_abort);
    }
    int K, nb;
    const int8_t* q = item_act(P, it, K, nb);
    const uint8_t* abuf;
    const float* sc = nullptr;  // chained: the scales of the vectors in act[buf]
    if constexpr (C::CHAINED) {  // the stage's matrices share one input: quantize it once per stage and pass
      const ChainSrc cs = it.kind == kItemTernary ? P.mats[it.mat].src : P.head_src;
      if ((staged || cs.in0 != chain_in0 || it.b0 != chain_b0) && (it.begin < it.end || blockIdx.x == 0)) {
        flush();  // this prologue replaces s_chain
        buf ^= 1;
        const bool rec = blockIdx.x == 0;
        if constexpr (C::NBMAX != 1) {  // the codes go out from the prologue itself
          if (it.kind == kItemTernary) {
            const int rf = P.mats[it.mat].rec_first, rn = P.mats[it.mat].rec_count;
            chain_prologue<C>(cs, it.b0, nb, P.act_k, act + buf * act_buf, s_chain, red, rec, P.mats + rf, rn,
                              nullptr, nullptr);
          } else {
            chain_prologue<C>(cs, it.b0, nb, P.act_k, act + buf * act_buf, s_chain, red, rec, nullptr, 0,
                              const_cast<int8_t*>(P.head_q), const_cast<float*>(P.head_sx));
          }
        } else {  // here only the capture buffer (tests); the codes: flush()
          chain_prologue<C>(cs, it.b0, nb, P.act_k, act + buf * act_buf, s_chain, red, rec, nullptr, 0, nullptr,
                            nullptr);
        }
        if (C::NBMAX == 1 && rec && threadIdx.x == 0) {
          const bool hd = it.kind != kItemTernary;
          s_rec[1] = it.b0;
          s_rec[2] = nb;
          s_rec[3] = buf;
          s_rec[4] = hd ? 0 : P.mats[it.mat].rec_count;
          s_rec[5] = hd ? 1 : 0;
          *s_rec_mats = hd ? nullptr : P.mats + P.mats[it.mat].rec_first;
          s_rec[0] = cs.K;
        }
        chain_in0 = cs.in0;
        chain_b0 = it.b0;
      }
      consumer_sync<C>();
      if (staged) stamp(P, (int)barriers, 2);
      abuf = act + buf * act_buf;
      sc = s_chain;
    } else {
      uint8_t* ab = act + buf * act_buf;
      if (prefetched) cp_async_wait_all();
      else load_act<C>(ab, q, K, nb, P.act_k, false);
      consumer_sync<C>();  // act[buf] complete; every warp is past the previous item
      if (staged) stamp(P, (int)barriers, 2);
      prefetched = false;
      if (i + 1 < n_items) {  // supplied inputs were quantized before any stage: prefetch across barriers too
        if constexpr (C::NBMAX != 1) q2 = item_act(P, get_item(P, i + 1), K2, nb2);
        load_act<C>(act + (buf ^ 1) * act_buf, q2, K2, nb2, P.act_k, true);
        prefetched = true;
      }
      abuf = ab;
    }
    if constexpr (C::NBMAX == 1) {
      consume_item<C, 1>(P, it, seq, abuf, rg, wbest, cw, lane, s_abort, sc, slot_row, pre, sx_pre);
    } else {
      switch (nb) {
        case 1: consume_item<C, 1>(P, it, seq, abuf, rg, wbest, cw, lane, s_abort, sc, slot_row, pre, sx_pre); break;
        case 2: consume_item<C, 2>(P, it, seq, abuf, rg, wbest, cw, lane, s_abort, sc, slot_row, pre, sx_pre); break;
        case 3: consume_item<C, 3>(P, it, seq, abuf, rg, wbest, cw, lane, s_abort, sc, slot_row, pre, sx_pre); break;
        default: consume_item<C, 4>(P, it, seq, abuf, rg, wbest, cw, lane, s_abort, sc, slot_row, pre, sx_pre); break;
      }
    }
    seq += (uint32_t)(it.end - it.begin);
    if constexpr (!C::CHAINED) buf ^= 1;
  }
  if (prefetched) cp_async_wait_all();
  flush();
  consumer_sync<C>();
  stamp(P, 0, 1);
  if (P.reset_barriers && !P.has_head && threadIdx.x == 0) {
    // this CTA is past its last grid barrier; the last one to get here (all others are past
    // theirs too) zeroes the arrival counter for the next launch
    __threadfence();
    if (atomicAdd(&P.ctrl->exit_done, 1u) == gridDim.x - 1) {
      P.ctrl->arrive = 0u;
      P.ctrl->exit_done = 0u;
    }
  }

  if (P.has_head) {  // CTA best per vector, then the last CTA to finish reduces all CTAs
    volatile int& s_last = *reinterpret_cast<volatile int*>(smem + L.abort_flag + 4);
    volatile int& s_fail = *reinterpret_cast<volatile int*>(smem + L.abort_flag + 8);
    consumer_sync<C>();
    if (threadIdx.x < P.B && !*s_abort) {
      HeadPartial b = hbest[threadIdx.x];
      for (int w = 1; w < C::CW; ++w) {
        const HeadPartial c = hbest[w * kStepMaxBatch + threadIdx.x];
        if (better(c.val, c.idx, b.val, b.idx)) b = c;
      }
      P.head_ws->part[(int64_t)blockIdx.x * P.B + threadIdx.x] = b;
    }
    consumer_sync<C>();
    if (threadIdx.x == 0) {
      // Every CTA counts itself, also one that gave up, so the counter always returns to zero.
      // The fence orders this CTA's partials and any error it recorded before its arrival.
      __threadfence();
      const bool last = atomicAdd(&P.ctrl->head_done, 1u) == gridDim.x - 1;
      if (last) __threadfence();
      s_fail = last && (*s_abort || *reinterpret_cast<volatile unsigned int*>(&P.ctrl->error) != 0u);
      s_last = last;
    }
    consumer_sync<C>();
    if (s_last) {
      // warp w picks the winner of vector w (w + CW, ...): its lanes walk the CTAs' partials,
      // then a shuffle reduction; a step in which some wait ran out reports -1 instead
      const bool failed = s_fail;
      for (int b = warp; b < P.B; b += C::CW) {
        float bv = -INFINITY;
        int bi = INT_MAX;
        for (int c = lane; c < (int)gridDim.x && !failed; c += 32) {
          const HeadPartial* pp = &P.head_ws->part[(int64_t)c * P.B + b];
          const float pv = __ldcg(&pp->val);
          const int pi = __ldcg(&pp->idx);
          if (better(pv, pi, bv, bi)) { bv = pv; bi = pi; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
          if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) P.head_argmax[b] = failed ? -1 : (bi == INT_MAX ? 0 : bi);
      }
      if (threadIdx.x == 0) {
        P.ctrl->head_done = 0u;
        if (P.head_next) *P.head_next = 0u;  // every producer's last grab came before its CTA arrived
        if (P.reset_barriers) P.ctrl->arrive = 0u;  // every CTA arrived after its last grid barrier
      }
      if (P.verify_emit && !failed) {  // accept the longest agreeing draft prefix on the device
        consumer_sync<C>();
        if (threadIdx.x == 0) *P.verify_n = verify_accept_device(P.verify_draft, P.head_argmax, P.B, P.verify_emit);
      }
    }
  }
}

// ---- host ------------------------------------------------------------------------------
struct Unitset {
  int kind, mat;
  int64_t units;
  int64_t unit_bytes;
};

// Splits one stage's units into `grid` contiguous byte ranges and appends each CTA's items
// for the pass starting at vector b0. With `one_item` (stages between grid barriers) every
// CTA gets units of one set only: the sets get whole CTAs in proportion to their bytes
// (largest remainder, at least one each while there are CTAs left) and split their units
// evenly among them (so CTA 0, which records a chained stage's codes, always has an item of
// the stage). A CTA whose range straddled two sets would run them one after the other
// -- its warps meet at the switch, since the second set's activations replace the first's --
// and so hold the whole stage back by a tile's latency.
void partition_stage(const std::vector<Unitset>& sets, int grid, int b0, bool barrier_before,
                     std::vector<std::vector<WorkItem>>& per_cta, bool one_item = false) {
  int64_t total = 0;
  for (const Unitset& s : sets) total += s.units * s.unit_bytes;
  std::vector<bool> flagged(grid, false);
  auto push = [&](int c, const WorkItem& w) {
    WorkItem x = w;
    if (barrier_before && !flagged[c]) { x.flags |= kFlagStage; flagged[c] = true; }
    per_cta[c].push_back(x);
  };
  const int ns = (int)sets.size();
  if (one_item && ns > 1 && ns <= grid && total > 0) {
    std::vector<int64_t> n(ns);
    std::vector<std::pair<int64_t, int>> rem;  // (remainder of share * total, set)
    int64_t given = 0;
    for (int i = 0; i < ns; ++i) {
      const int64_t b = sets[i].units * sets[i].unit_bytes;
      n[i] = std::max<int64_t>(1, b * grid / total);
      rem.push_back({b * grid - (b * grid / total) * total, i});
      given += n[i];
    }
    std::sort(rem.begin(), rem.end(), [](const auto& a, const auto& b) { return a.first > b.first; });
    for (size_t r = 0; given < grid; r = (r + 1) % rem.size(), ++given) ++n[rem[r].second];
    for (int i = ns - 1; given > grid; i = (i + ns - 1) % ns)  // the max(1, .) above overshot
      if (n[i] > 1) { --n[i]; --given; }
    int c0 = 0;
    for (int i = 0; i < ns; ++i) {
      const Unitset& st = sets[i];
      for (int64_t j = 0; j < n[i]; ++j) {  // rounded up: the set's first CTA always gets units
        const int64_t u = (st.units * j + n[i] - 1) / n[i], v = (st.units * (j + 1) + n[i] - 1) / n[i];
        if (u < v) push(c0 + (int)j, WorkItem{st.kind, st.mat, 0, b0, u, v});
      }
      c0 += (int)n[i];
    }
  } else {
  int64_t start = 0;  // byte offset of the current unit set within the stage
  for (const Unitset& s : sets) {
    int64_t u = 0;
    while (u < s.units) {
      // owner of unit u: the CTA whose byte range holds the unit's first byte
      const int c = (int)std::min<int64_t>(grid - 1, (start + u * s.unit_bytes) * grid / std::max<int64_t>(total, 1));
      const int64_t end_byte = (int64_t)(c + 1) * total / grid;
      int64_t v = u + 1;
      while (v < s.units && start + v * s.unit_bytes < end_byte) ++v;
      push(c, WorkItem{s.kind, s.mat, 0, b0, u, v});
      u = v;
    }
    start += s.units * s.unit_bytes;
  }
  }
  if (barrier_before)  // every CTA takes part in the barrier, with or without work
    for (int c = 0; c < grid; ++c)
      if (!flagged[c]) push(c, WorkItem{sets.front().kind, sets.front().mat, 0, b0, 0, 0});
}

// Chained stages: CTA 0 quantizes each stage input like every CTA and also writes its codes
// out, so it takes no units; the stage is split over CTAs 1 .. grid - 1 and CTA 0 gets an
// empty item of the stage (its prologue runs for CTA 0 with or without units).
void partition_stage_chained(const std::vector<Unitset>& sets, int grid, int b0, bool barrier_before,
                             std::vector<std::vector<WorkItem>>& per_cta) {
  std::vector<std::vector<WorkItem>> rest(grid - 1);
  partition_stage(sets, grid - 1, b0, barrier_before, rest, true);
  for (int c = 1; c < grid; ++c) per_cta[c].insert(per_cta[c].end(), rest[c - 1].begin(), rest[c - 1].end());
  per_cta[0].push_back(WorkItem{sets.front().kind, sets.front().mat, barrier_before ? kFlagStage : 0, b0, 0, 0});
}

// Ring depth and vectors per pass that fit the shared-memory budget for activations of
// act_k bytes: 3 slots when possible (deeper ring), else 2; then fewer vectors per pass.
template <class C>
bool pick_config_for(int B, int act_k, int* nslots, int* chunk_b, size_t* smem) {
  int dev = 0, optin = kMaxSmem;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  const int limit = std::min(kMaxSmem, optin);
  for (int cb = std::min(B, C::NBMAX); cb >= 1; --cb)
    for (int ns = kMaxSlots; ns >= 2; --ns) {
      const SmemLayout L = smem_layout<C>(ns, cb, act_k);
      if (L.total <= limit) {
        *nslots = ns;
        *chunk_b = cb;
        *smem = (size_t)L.total;
        return true;
      }
    }
  return false;
}

// Rows of the output table each CTA takes before it starts drawing rows from the counter
// (kItemHeadDyn): as many as every producer lane's ring holds at once, so the standalone call
// issues them without waiting for a slot, and never more than the table has for every CTA.
int head_fixed_rows(int cw, int nslots, int K, int V, int grid) {
  const int per_row = (int)((K + kSlotBytes - 1) / kSlotBytes);
  const int fixed = cw * (nslots / per_row);
  return std::min(fixed, V / std::max(grid, 1));
}

bool pick_config(int B, int act_k, int* nslots, int* chunk_b, size_t* smem, bool chained = false) {
  if (chained)
    return B == 1 ? pick_config_for<Cfg1C>(B, act_k, nslots, chunk_b, smem)
                  : pick_config_for<CfgBC>(B, act_k, nslots, chunk_b, smem);
  return B == 1 ? pick_config_for<Cfg1>(B, act_k, nslots, chunk_b, smem)
                : pick_config_for<CfgB>(B, act_k, nslots, chunk_b, smem);
}

std::mutex g_attr_mu;
bool g_attr_set[64] = {};

nt_status configure_kernel(int device) {
  std::lock_guard<std::mutex> lock(g_attr_mu);
  if (device >= 0 && device < 64 && g_attr_set[device]) return NT_OK;
  NT_CUDA_TRY(cudaFuncSetAttribute(persist_kernel<Cfg1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem));
  NT_CUDA_TRY(cudaFuncSetAttribute(persist_kernel<CfgB>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem));
  NT_CUDA_TRY(cudaFuncSetAttribute(persist_kernel<Cfg1C>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem));
  NT_CUDA_TRY(cudaFuncSetAttribute(persist_kernel<CfgBC>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem));
  if (device >= 0 && device < 64) g_attr_set[device] = true;
  return NT_OK;
}

// Consumer warps of the kernel instance for a batch and step mode.
int kernel_cw(int B, bool chained) {
  if (chained) return B == 1 ? Cfg1C::CW : CfgBC::CW;
  return B == 1 ? Cfg1::CW : CfgB::CW;
}

// The kernel instance and block size for a batch and step mode.
const void* kernel_for(int B, bool chained, int* threads) {
  *threads = B == 1 ? Cfg1::THREADS : CfgB::THREADS;
  if (chained) {
    *threads = B == 1 ? Cfg1C::THREADS : CfgBC::THREADS;
    return B == 1 ? reinterpret_cast<const void*>(persist_kernel<Cfg1C>)
                  : reinterpret_cast<const void*>(persist_kernel<CfgBC>);
  }
  return B == 1 ? reinterpret_cast<const void*>(persist_kernel<Cfg1>)
                : reinterpret_cast<const void*>(persist_kernel<CfgB>);
}

}  // namespace

nt_status persist_prepare(nt_decode_plan* p) {
  int kmax = p->has_head ? p->head_K : 16;
  for (const MatDesc& m : p->mats) kmax = std::max<int>(kmax, (int)padded_k(m.K));
  p->act_stride = (int)padded_k(kmax);
  if (!pick_config(p->B, p->act_stride, &p->nslots, &p->chunk_b, &p->smem_bytes, p->mode == NT_STEP_CHAINED))
    return set_error(NT_ERR_INVALID_ARG, "persistent launcher: K too large for the shared-memory budget");
  NT_TRY(configure_kernel(p->device));
  int per_sm = 0, threads = 0;
  const void* kern = kernel_for(p->B, p->mode == NT_STEP_CHAINED, &threads);
  NT_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, p->smem_bytes));
  if (per_sm < 1) return set_error(NT_ERR_CUDA, "persistent kernel cannot be resident on an SM");
  const int grid = p->sm_count;
  p->grid = grid;

  std::vector<std::vector<WorkItem>> per_cta(grid);
  std::vector<std::vector<std::vector<WorkItem>>> seg_cta;  // segmented plans
  p->seg_barriers.clear();
  p->seg_off_bytes.clear();
  const int n_proj = (int)p->mats.size();
  auto ternary = [&](int mi) {
    return Unitset{kItemTernary, mi, padded_rows(p->mats[mi].N) / 4, padded_k(p->mats[mi].K)};
  };
  const Unitset head{kItemHead, 0, p->head_V, p->head_K};
  const bool chained = p->mode == NT_STEP_CHAINED;
  int barriers = (p->n_qjobs > 0 ? 1 : 0) + (p->embed_T && (p->n_qjobs > 0 || chained) ? 1 : 0);
  p->head_fixed = 0;
  if (p->mode == NT_STEP_INDEPENDENT) {
    // Each CTA gets 1/grid of the ternary bytes. The output table follows as rows handed out
    // at run time (one pass: every CTA ends with the same dynamic item, so CTAs that finish
    // their ternary share early take more rows and all finish together); with several passes
    // each CTA gets 1/grid of the table per pass.
    const bool dyn = p->has_head && p->B <= p->chunk_b;
    if (dyn) p->head_fixed = head_fixed_rows(kernel_cw(p->B, false), p->nslots, p->head_K, p->head_V, grid);
    for (int b0 = 0; b0 < p->B; b0 += p->chunk_b) {
      std::vector<Unitset> all;
      for (int i = 0; i < n_proj; ++i) all.push_back(ternary(i));
      partition_stage(all, grid, b0, false, per_cta);
      if (dyn) {
        for (int c = 0; c < grid; ++c) per_cta[c].push_back(WorkItem{kItemHeadDyn, 0, 0, b0, 0, p->head_V});
      } else if (p->has_head) {
        partition_stage({head}, grid, b0, false, per_cta);
      }
    }
  } else if (chained && p->attn) {
    // one launch per segment; the attention side runs between segments
    const int L = p->n_layers;
    auto stage_into = [&](std::vector<std::vector<WorkItem>>& pc, bool& first, int& nbar,
                          const std::vector<Unitset>& sets) {
      for (int b0 = 0; b0 < p->B; b0 += p->chunk_b) partition_stage_chained(sets, grid, b0, !first && b0 == 0, pc);
      nbar += first ? 0 : 1;
      first = false;
    };
    for (int sg = 0; sg <= L; ++sg) {
      std::vector<std::vector<WorkItem>> pc(grid);
      bool first = true;
      int nbar = sg == 0 ? barriers : 0;  // the first segment also gathers / quantizes the inputs
      if (sg > 0) {
        const int b = (sg - 1) * kProjPerLayer;
        stage_into(pc, first, nbar, {ternary(b + 3)});
        stage_into(pc, first, nbar, {ternary(b + 4), ternary(b + 5)});
        stage_into(pc, first, nbar, {ternary(b + 6)});
      }
      if (sg < L) {
        const int b = sg * kProjPerLayer;
        stage_into(pc, first, nbar, {ternary(b), ternary(b + 1), ternary(b + 2)});
      } else if (p->has_head) {
        stage_into(pc, first, nbar, {head});
      }
      seg_cta.push_back(std::move(pc));
      p->seg_barriers.push_back(nbar);
      barriers = std::max(barriers, nbar);
    }
  } else {
    bool first = true;
    auto stage = [&](const std::vector<Unitset>& sets) {
      for (int b0 = 0; b0 < p->B; b0 += p->chunk_b) {
        if (chained) partition_stage_chained(sets, grid, b0, !first && b0 == 0, per_cta);
        else partition_stage(sets, grid, b0, !first && b0 == 0, per_cta, true);
      }
      barriers += first ? 0 : 1;
      first = false;
    };
    for (int l = 0; l < p->n_layers; ++l) {
      const int b = l * kProjPerLayer;
      const int groups[4][2] = {{b, 3}, {b + 3, 1}, {b + 4, 2}, {b + 6, 1}};
      for (const auto& g : groups) {
        std::vector<Unitset> sets;
        for (int i = 0; i < g[1]; ++i) sets.push_back(ternary(g[0] + i));
        stage(sets);
      }
    }
    if (p->has_head) stage({head});
  }
  p->n_barriers = barriers;

  // every segment's per-CTA items, then each segment's (grid + 1) offsets into the items
  std::vector<std::vector<std::vector<WorkItem>>> segs;
  if (p->seg_barriers.empty()) segs.push_back(std::move(per_cta));
  else segs = std::move(seg_cta);
  std::vector<WorkItem> items;
  std::vector<int> off;
  for (const auto& pc : segs) {
    for (int c = 0; c < grid; ++c) {
      off.push_back((int)items.size());
      items.insert(items.end(), pc[c].begin(), pc[c].end());
    }
    off.push_back((int)items.size());
  }
  const size_t item_bytes = sizeof(WorkItem) * std::max<size_t>(items.size(), 1);
  NT_CUDA_TRY(cudaMalloc(&p->d_sched, item_bytes + sizeof(int) * off.size()));
  if (!items.empty()) NT_CUDA_TRY(cudaMemcpy(p->d_sched, items.data(), sizeof(WorkItem) * items.size(), cudaMemcpyHostToDevice));
  NT_CUDA_TRY(cudaMemcpy(reinterpret_cast<uint8_t*>(p->d_sched) + item_bytes, off.data(), sizeof(int) * off.size(),
                         cudaMemcpyHostToDevice));
  p->sched_item_bytes = item_bytes;
  for (size_t s = 0; s < p->seg_barriers.size(); ++s)
    p->seg_off_bytes.push_back(item_bytes + sizeof(int) * (grid + 1) * s);
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
  P.head_next = &p->d_ctrl->head_next;
  P.head_fixed = p->head_fixed;
  P.head_V = p->head_V;
  P.head_K = p->head_K;
  P.has_head = p->has_head ? 1 : 0;
  P.B = p->B;
  P.chunk_b = p->chunk_b;
  P.nslots = p->nslots;
  P.act_k = p->act_stride;
  P.barrier_extra = p->test_fault == 1 ? 1u : 0u;
  P.timeout_ns = p->timeout_ns;
  P.trace = p->trace;
  P.embed_T = p->embed_T;
  P.embed_s = p->embed_s;
  P.embed_V = p->embed_V;
  P.embed_K = p->embed_K;
  P.tokens = p->tokens;
  P.embed_x = p->embed_x;
  P.verify_draft = p->verify_draft;
  P.verify_emit = p->verify_emit;
  P.verify_n = p->verify_n;
  P.head_src = p->head_src;
  int threads = 0;
  const void* kern = kernel_for(p->B, p->mode == NT_STEP_CHAINED, &threads);
  // a single launch per step resets the barrier counter itself (its parameters are the same
  // on every call); segmented steps count barriers across their launches on the host
  P.reset_barriers = p->seg_barriers.empty() ? 1 : 0;
  auto launch = [&](int n_barriers) -> nt_status {
    P.n_barriers = n_barriers;
    P.barrier_base = P.reset_barriers ? 0u : p->barrier_count * (uint32_t)p->grid;
    void* args[] = {&P};
    const cudaError_t e = cudaLaunchCooperativeKernel(kern, dim3(p->grid), dim3(threads), args, p->smem_bytes, st);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return set_error(NT_ERR_CUDA, std::string("persistent launch: ") + cudaGetErrorString(e));
    }
    if (!P.reset_barriers) p->barrier_count += (uint32_t)n_barriers;
    return NT_OK;
  };
  if (p->seg_barriers.empty()) {
    NT_TRY(launch(p->n_barriers));
  } else {
    // one launch per segment, the layer's rotation, cache append and attention in between;
    // input gathering and quantization belong to the first segment, the output projection
    // (and the verify acceptance) to the last
    const int nseg = (int)p->seg_barriers.size();
    const uint8_t* base = reinterpret_cast<const uint8_t*>(p->d_sched);
    P.trace = nullptr;
    for (int sg = 0; sg < nseg; ++sg) {
      const bool last = sg == nseg - 1;
      P.item_off = reinterpret_cast<const int*>(base + p->seg_off_bytes[sg]);
      P.n_qjobs = sg == 0 ? p->n_qjobs : 0;
      P.embed_T = sg == 0 ? p->embed_T : nullptr;
      P.has_head = last && p->has_head ? 1 : 0;
      P.verify_emit = last ? p->verify_emit : nullptr;
      NT_TRY(launch(p->seg_barriers[sg]));
      if (!last) {
        const int l = sg;
        const MatDesc* m = p->mats.data() + l * kProjPerLayer;
        NT_TRY(launch_rope_append(m[0].y, m[1].y, m[2].y, p->B, p->Hq, p->Hkv, 0, p->rope_base, p->d_qrot,
                                  p->k_cache[l], p->v_cache[l], p->t_stride, st, p->d_pos, true));
        NT_TRY(launch_attention(p->d_qrot, p->k_cache[l], p->v_cache[l], p->B, p->Hq, p->Hkv, p->t_stride,
                                p->t_stride, p->d_attn_out, p->d_attn_ws, st, p->d_pos + 1, true));
      }
    }
  }
  ++p->launches;
  return NT_OK;
}

bool persist_head_fits(int K, int B) {
  int ns, cb;
  size_t smem;
  return B >= 1 && B <= kStepMaxBatch && pick_config(B, (int)padded_k(K), &ns, &cb, &smem);
}

nt_status persist_launch_head(const int8_t* T, const float* s_T, int V, int K, const int8_t* q,
                              const float* s_x, int B, float* logits, int32_t* argmax, HeadWs* ws,
                              cudaStream_t st, bool pdl) {
  int dev = 0;
  NT_CUDA_TRY(cudaGetDevice(&dev));
  PersistParams P{};
  P.act_k = (int)padded_k(K);
  size_t smem = 0;
  if (!pick_config(B, P.act_k, &P.nslots, &P.chunk_b, &smem))
    return set_error(NT_ERR_INVALID_ARG, "output projection: K too large for the streaming kernel");
  NT_TRY(configure_kernel(dev));
  // The workspace's 16-byte status header serves as the control word (error, counter): zero
  // before the first call, and every call leaves the counter zero; an error code stays until
  // the caller clears the workspace.
  P.ctrl = reinterpret_cast<StepCtrl*>(ws);
  P.head_ws = ws;
  P.head_T = T;
  P.head_s = s_T;
  P.head_q = q;
  P.head_sx = s_x;
  P.head_logits = logits;
  P.head_argmax = argmax;
  P.head_V = V;
  P.head_K = K;
  P.has_head = 1;
  P.B = B;
  const int grid = (int)std::min<int64_t>(device_sm_count(), V);
  // one pass: rows handed out at run time (the counter is the header's third word, which the
  // standalone call has no other use for)
  P.head_dyn = B <= P.chunk_b ? 1 : 0;
  P.head_next = reinterpret_cast<unsigned int*>(ws) + 2;
  P.head_fixed = head_fixed_rows(B == 1 ? Cfg1::CW : CfgB::CW, P.nslots, K, V, grid);
  P.timeout_ns = test_fault_timeout_ns(250000000ull);
  P.no_copies = test_fault() == kFaultHeadStream;
  if (B == 1) NT_CUDA_TRY(launch_kernel(persist_kernel<Cfg1>, dim3(grid), dim3(Cfg1::THREADS), smem, st, pdl, P));
  else NT_CUDA_TRY(launch_kernel(persist_kernel<CfgB>, dim3(grid), dim3(CfgB::THREADS), smem, st, pdl, P));
  return check_launch("persist_kernel (output projection)");
}

}  // namespace nt
