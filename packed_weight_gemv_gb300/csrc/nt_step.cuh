// nt_step.cuh -- the decode plan's host state and the persistent launcher's schedule.
#pragma once

#include <vector>

#include "nt_kernels.cuh"

namespace nt {

constexpr int kProjPerLayer = 7;   // q, k, v, o, gate, up, down
constexpr int kStepMaxBatch = 16;

struct PlanStage {
  int first_mat, n_mats;
  int64_t prefix_off;   // into the plan's prefix array
  int64_t total_tiles;
  int64_t mma_ctas;     // batched plans on the tensor-core path: CTAs of the stage's launch
  int64_t mma_tab_off;  //   and the offset of its CTA -> matrix table in the plan's table
};

// Device control word of a plan: error word of the bounded waits and the grid-barrier
// arrival counter of the persistent kernel.
struct StepCtrl {
  unsigned int error;      // 0 = fine; otherwise the code of the wait that ran out
  unsigned int error_cta;
  unsigned int arrive;     // grid-barrier arrivals (wraps; compared modulo 2^32)
  unsigned int head_done;  // CTAs finished with the output projection's arg-max
  unsigned int head_next;  // output-table rows handed out so far (dynamic rows; the last CTA resets it)
  unsigned int exit_done;  // CTAs past their last grid barrier (single-launch plans without an output table)
  unsigned int pad_[2];
};

// One contiguous run of work for one CTA of the persistent kernel. kItemHeadDyn: the output
// table's rows handed out at run time (a few fixed rows per CTA first, then CW rows per grab from
// a global counter), so that CTAs on SMs that stream faster take more rows.
enum : int { kItemTernary = 0, kItemHead = 1, kItemHeadDyn = 2 };
enum : int { kFlagStage = 1 };  // a grid-wide barrier precedes this item (ordered mode)
struct WorkItem {
  int kind;      // kItemTernary (begin/end count tiles of mats[mat]) or kItemHead (rows)
  int mat;
  int flags;
  int b0;        // first activation vector of this pass
  int64_t begin, end;
};

}  // namespace nt

struct nt_decode_plan {
  int device = 0, sm_count = 0;
  int n_layers = 0, B = 1, mode = 0, launcher = 0;
  uint64_t timeout_ns = 0;
  int test_fault = 0;
  std::vector<nt::MatDesc> mats;
  std::vector<nt::PlanStage> stages;
  nt::MatDesc* d_mats = nullptr;
  int64_t* d_prefix = nullptr;
  // stream / graph launchers of batched plans: the tensor-core path's matrices (step order,
  // each stage's CTAs numbered from 0) and its int32 workspace (reused by every stage)
  nt::MmaMat* d_mma = nullptr;
  void* d_mma_ws = nullptr;
  uint16_t* d_mma_tab = nullptr;
  // independent batched plans (one stage, every matrix >= 128 rows): the tcgen05 path instead
  nt::Tc8Plan tc8;
  nt::QuantJob* d_qjobs = nullptr;
  int n_qjobs = 0;
  bool has_head = false;
  const int8_t* head_T = nullptr;
  const float* head_s = nullptr;
  int head_V = 0, head_K = 0;
  const int8_t* head_q = nullptr;
  const float* head_sx = nullptr;
  float* head_logits = nullptr;
  int32_t* head_argmax = nullptr;
  nt::HeadWs* d_head_ws = nullptr;
  // input-table gather at the start of the step
  const int8_t* embed_T = nullptr;
  const float* embed_s = nullptr;
  int embed_V = 0, embed_K = 0;
  const int32_t* tokens = nullptr;
  float* embed_x = nullptr;
  // verify-pass acceptance after the output projection
  const int32_t* verify_draft = nullptr;
  int32_t* verify_emit = nullptr;
  int32_t* verify_n = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  nt::StepCtrl* d_ctrl = nullptr;
  // persistent launcher
  nt::WorkItem* d_sched = nullptr;  // items, then (grid + 1) int offsets
  size_t sched_item_bytes = 0;
  int grid = 0, n_barriers = 0;
  size_t smem_bytes = 0;
  int act_stride = 0;               // bytes of one activation vector in shared memory
  int nslots = 0, chunk_b = 0;      // ring slots per consumer warp; vectors per pass
  int head_fixed = 0;               // output-table rows per CTA before the dynamic ones (independent mode)
  uint64_t launches = 0;
  uint32_t barrier_count = 0;       // grid barriers passed by all launches so far (mod 2^32)
  // chained plans with the attention side: one persistent launch per segment (the stages
  // between two attention sides: [A_0], [B_l C_l D_l A_l+1] ..., [B_L-1 C_L-1 D_L-1 head]),
  // each with its own grid barriers and per-CTA item offsets in d_sched
  std::vector<int> seg_barriers;
  std::vector<size_t> seg_off_bytes;
  unsigned long long* trace = nullptr;  // optional step timeline (nt_decode_plan_set_trace)
  // chained steps (NT_STEP_CHAINED)
  int head_dim = 128;
  nt::ChainSrc head_src{};          // the output projection's input (persistent launcher)
  float* d_resid = nullptr;         // [B][d] residual stream, owned by the plan
  float* d_chain_tmp = nullptr;     // [B][max K] stage inputs of the stream / graph launchers
  nt::ChainJob* d_cjobs = nullptr;  // one per stage, then one for the output projection
  int n_cjobs = 0;
  std::vector<nt::ChainJob> cjobs;  // host copy of d_cjobs (nt_decode_plan_set_capture edits it)
  // chained steps with the attention side
  bool attn = false;
  int Hq = 0, Hkv = 0, t_stride = 0;
  float rope_base = 10000.0f;
  std::vector<uint16_t*> k_cache, v_cache;  // per layer
  int* d_pos = nullptr;             // {position of the first vector, cache length after the append}
  float* d_qrot = nullptr;          // [B][Hq * 128] rotated queries
  float* d_attn_out = nullptr;      // [B][Hq * 128] attention output
  void* d_attn_ws = nullptr;        // attention workspace (counters zero)
  size_t attn_ws_bytes = 0;
};

namespace nt {
nt_status persist_prepare(nt_decode_plan* p);
nt_status persist_launch(nt_decode_plan* p, cudaStream_t st);
// Standalone output projection on the streaming kernel (no plan): B <= 16 and K small
// enough for its shared-memory activation buffers.
bool persist_head_fits(int K, int B);
// With pdl the launch is a programmatic dependent one: the weight stream starts while the
// previous kernel in the stream finishes.
nt_status persist_launch_head(const int8_t* T, const float* s_T, int V, int K, const int8_t* q,
                              const float* s_x, int B, float* logits, int32_t* argmax, HeadWs* ws,
                              cudaStream_t st, bool pdl);
}  // namespace nt
