// nt_kernels.cuh -- descriptors and launch helpers of the library's kernels.
#pragma once

#include "nt_internal.cuh"

namespace nt {

// One activation vector set to quantize: B vectors of length K.
struct QuantJob {
  const float* x;  // [B][K]
  int8_t* q;       // [B][K]
  float* s;        // [B]
  int K, B;
};

// Where a chained stage's input comes from (vector b, element k of K):
//   kChainDirect   in0[b][k]
//   kChainHeads    in0[b][((k / hd) / grp) * hd + k % hd]: attention over one cached position,
//                  query head i takes value head i / grp (in0 has K / grp columns)
//   kChainProduct  fl(in0[b][k] * in1[b][k])
//   kChainSum      fl(in0[b][k] + in1[b][k])
//   kChainSiluProduct fl(silu(in0[b][k]) * in1[b][k]), silu(x) = x / (1 + exp(-x)) in fp32
// With gamma set, the quantized vector is the RMS-normalised fl(fl(v * r) * gamma[k]),
// r = fl32(1 / sqrt(mean(v^2) + eps)): the squares summed in fp32 within each warp, the warps'
// sums added and r formed in double by one thread. With cap set, the kernel that quantizes the
// stage also stores the fp32 values it quantized there ([B][K]; nt_decode_plan_set_capture).
enum : int { kChainNone = 0, kChainDirect = 1, kChainHeads = 2, kChainProduct = 3, kChainSum = 4,
             kChainSiluProduct = 5 };
struct ChainSrc {
  const float* in0;
  const float* in1;
  int kind, K, grp, hd;
  const float* gamma;
  float eps;
  int pad_;
  float* cap;
};

// One ternary projection in the tiled layout, B activation vectors.
struct MatDesc {
  const uint8_t* w;  // tiles (nt_repack_ternary output)
  const float* s_w;  // [N]
  const int8_t* q;   // [B][K]
  const float* s_x;  // [B]
  float* y;          // [B][N]
  int32_t* acc;      // [B][N] or null
  int N, K, B;
  int rec_first;     // chained steps: first of the rec_count matrices whose q / s_x record
  int rec_count;     //   this matrix's input (the stage's matrices)
  int pad_;
  ChainSrc src;      // chained steps (persistent launcher): the stage input; kind 0 = none
  const float* res_in;  // chained steps: res_out[b][n] = fl(res_in[b][n] + y[b][n]), or null
  float* res_out;
};

// One stage input of a chained step on the stream / graph launchers: the source, a buffer
// for the fp32 values (the residual stream itself for kChainSum), and the matrices whose
// q / s_x receive the codes.
struct ChainJob {
  ChainSrc src;
  float* vbuf;       // [B][K]
  int n_rec;
  int pad_;
  int8_t* q[3];
  float* s[3];
};

// Scratch of the output-projection kernel's cross-CTA arg-max (caller-owned workspace).
constexpr int kHeadMaxCtas = 1024;
struct HeadPartial {
  float val;
  int idx;
};
// The first 16 bytes of every workspace are its status header (nt_workspace_status): the
// error code and CTA of a bounded wait that ran out, then, for the output projection, the
// counter of CTAs done with the arg-max at the offset the decode plan's StepCtrl keeps it.
struct WsHeader {
  unsigned int error;      // 0 = fine; otherwise the code of the wait that ran out
  unsigned int error_cta;
  unsigned int pad_;
  unsigned int done;       // output projection: CTAs finished; the last one resets it to 0
};
struct HeadWs {
  unsigned int error, error_cta, pad_;
  unsigned int done;
  HeadPartial part[1];     // [kHeadMaxCtas][B]
};
// Bytes in front of the data of the GEMM workspaces (the status header, padded so the data
// keeps the alignment its tensor maps need).
constexpr size_t kWsHeaderBytes = 256;
inline size_t head_ws_bytes(int B) { return 16 + sizeof(HeadPartial) * (size_t)kHeadMaxCtas * B; }

// Launchers (asynchronous on `st`; they return launch-configuration errors only).
nt_status launch_quantize(const float* x, int B, int K, int8_t* q, float* s, cudaStream_t st);
nt_status launch_quantize_jobs(const QuantJob* d_jobs, int n_jobs, int max_B, cudaStream_t st, bool pdl = false);
nt_status launch_repack(const uint32_t* w, int N, int K, uint8_t* out, uint32_t* n_invalid,
                        cudaStream_t st);
nt_status launch_validate(const uint32_t* w, int N, int K, unsigned long long* n_invalid, cudaStream_t st);
nt_status launch_gemv_plain(const uint32_t* w, const float* s_w, int N, int K, const int8_t* q,
                            const float* s_x, int B, float* y, int32_t* acc, cudaStream_t st);
nt_status launch_gemv_tiled(const MatDesc& m, cudaStream_t st);
// Several tiled projections in one launch: d_mats[n] in device memory, d_tile_prefix[n+1]
// their cumulative tile counts.
// Batched projections on the tensor cores (nt_gemv_mma.cu): 2..16 vectors, f16 MMA.
constexpr int kMmaMinBatch = 2, kMmaMaxBatch = 16;
struct MmaMat {
  const uint8_t* w;  // tiles (nt_repack_ternary output)
  const float* s_w;  // [N]
  const int8_t* q;   // [B][K]
  const float* s_x;  // [B]
  float* y;          // [B][N]
  int32_t* acc;      // [B][N] or null
  int32_t* acc_ws;   // [B][N] int32 workspace, zero between calls
  unsigned int* cnt; // [ugroups] part counters of each unit group, zero between calls
  int N, K, B;
  int units32, kchunks, ugroups, cpp, nparts;  // set by mma_geometry (cpp: chunks per part)
  int64_t cta_begin;              // first CTA of this matrix in its launch
};
void mma_geometry(MmaMat& m, int parts);
int64_t mma_ctas(const MmaMat& m);
size_t mma_ws_bytes(int64_t rows, int64_t groups, int B);
nt_status launch_gemv_mma(const MmaMat* d_mats, int n_mats, const uint16_t* d_cta_mat, int64_t total_ctas, int max_B,
                          cudaStream_t st, bool pdl = false);
// One tiled matrix per call on the same path (nt_ternary_gemm with a workspace of
// mma_single_ws_bytes, zero before its first use and left zero).
size_t mma_single_ws_bytes(int N, int K, int B);
nt_status launch_gemv_mma_single(const uint8_t* w, const float* s_w, int N, int K, const int8_t* q, const float* s_x,
                                 int B, float* y, int32_t* acc, void* ws, cudaStream_t st);
// One tiled matrix per call on tcgen05 (nt_gemv_tc8.cu): decoded weights in tensor memory,
// e4m3 digits of the activations; 2..16 vectors and at least 128 rows; workspace of
// tc8_ws_bytes (zero before its first use and left zero except for the digit rows).
bool tc8_supported(int N, int K, int B);
size_t tc8_ws_bytes(int N, int K, int B);
nt_status launch_gemv_tc8(const uint8_t* w, const float* s_w, int N, int K, const int8_t* q, const float* s_x, int B,
                          float* y, int32_t* acc, void* ws, cudaStream_t st);
// All matrices of one decode-plan stage on the same tcgen05 path (2..16 vectors, every
// matrix >= 128 rows): a digit-row launch, then one launch over every matrix's row tiles.
struct Tc8Plan {
  void* d_mats = nullptr;    // per matrix: tensor maps and parameters (device)
  uint16_t* d_tab = nullptr; // CTA -> matrix
  void* d_jobs = nullptr;    // per matrix: its digit-row job
  void* d_buf = nullptr;     // digit rows, then each matrix's partial sums and tile counters
  int n = 0, nn = 16, digit_grid = 1;
  int64_t ctas = 0;
  size_t buf_bytes = 0;      // d_buf (zeroed again by a plan reset)
};
bool tc8_plan_supported(const MatDesc* mats, int n, int B);
// err: the plan's status word (error code, then the CTA); a wait that runs out (after
// timeout_ns) records code 16; fault != 0 makes every CTA's producer issue no copies (tests)
nt_status tc8_plan_create(const MatDesc* mats, int n, int B, unsigned int* err, uint64_t timeout_ns, int fault,
                          Tc8Plan* t);
nt_status tc8_plan_launch(const Tc8Plan& t, cudaStream_t st, bool pdl);
void tc8_plan_destroy(Tc8Plan* t);
// Output projection on the tensor cores (nt_gemv_mma.cu): 2..16 vectors, one pass over T.
nt_status launch_head_mma(const int8_t* T, const float* s_T, int V, int K, const int8_t* q, const float* s_x,
                          int B, float* logits, int32_t* argmax, HeadWs* ws, cudaStream_t st);
nt_status launch_gemv_tiled_group(const MatDesc* d_mats, const int64_t* d_tile_prefix, int n,
                                  int64_t total_tiles, int max_B, cudaStream_t st, bool pdl = false);
nt_status launch_head(const int8_t* T, const float* s_T, int V, int K, const int8_t* q,
                      const float* s_x, int B, float* logits, int32_t* argmax, HeadWs* ws,
                      cudaStream_t st, bool pdl = false);

// Quantizes one chained stage input per vector (one CTA per vector).
nt_status launch_chain_quant(const ChainJob* d_job, int B, cudaStream_t st, bool pdl = false);

nt_status launch_embed(const int8_t* T, const float* s, int V, int K, const int32_t* tokens, int B, float* x,
                       uint32_t* n_bad, cudaStream_t st, bool pdl = false);
nt_status launch_verify(const int32_t* draft, const int32_t* argmax, int B, int32_t* emit, int32_t* n_emit,
                        cudaStream_t st, bool pdl = false);

// Attention side of a layer (nt_attention.cu): head dimension 128.
// The workspace's counters (after the partial results) must be zero before the first call;
// every call leaves them zero.
size_t attention_ws_bytes(int B, int Hq, int Hkv, int T);
// T_dev / pos_dev (optional): the cache length / first new position read from device memory
// when the kernel runs (a plan's position); T then only sizes the grid.
nt_status launch_attention(const float* q, const uint16_t* kc, const uint16_t* vc, int B, int Hq, int Hkv, int T,
                           int ts, float* out, void* ws, cudaStream_t st, const int* T_dev = nullptr,
                           bool pdl = false);
nt_status launch_rope_append(const float* q, const float* k, const float* v, int B, int Hq, int Hkv, int pos0,
                             float base, float* q_out, uint16_t* kc, uint16_t* vc, int ts, cudaStream_t st,
                             const int* pos_dev = nullptr, bool pdl = false);
nt_status launch_rmsnorm(const float* x, const float* gamma, int B, int D, float eps, float* y, cudaStream_t st);

// Tensor-core ternary GEMM (tcgen05, bf16 operands, exact fp32 accumulation) for
// prefill-shaped batches of at least kTcMinBatch vectors.
constexpr int kTcMinBatch = 64;
bool tc_gemm_supported(int M, int K);
size_t tc_gemm_workspace_bytes(int M, int N, int K);
nt_status launch_gemm_tc(const uint8_t* w, const float* s_w, int N, int K, const int8_t* q, const float* s_x,
                         int M, float* y, int32_t* acc, void* ws, cudaStream_t st);
// Up to 8 matrices sharing the activations: one activation conversion, one tile set.
size_t tc_gemm_multi_workspace_bytes(int M, int n, const int* N, int K);
nt_status launch_gemm_tc_multi(int n, const uint8_t* const* w, const float* const* s_w, const int* N, int K,
                               const int8_t* q, const float* s_x, int M, float* const* y, int32_t* const* acc,
                               void* ws, cudaStream_t st);

#ifdef __CUDACC__
// Four consecutive elements k..k+3 (k % 4 == 0) of vector b of a chained stage input. The
// sources were written earlier in the same step by other CTAs, so they are read through L2.
__device__ __forceinline__ float4 chain_load4(const ChainSrc& c, int b, int k) {
  if (c.kind == kChainHeads) {
    const int kv = c.K / c.grp;
    const int i = ((k / c.hd) / c.grp) * c.hd + k % c.hd;
    return __ldcg(reinterpret_cast<const float4*>(c.in0 + (int64_t)b * kv + i));
  }
  const float4 a = __ldcg(reinterpret_cast<const float4*>(c.in0 + (int64_t)b * c.K + k));
  if (c.kind == kChainDirect) return a;
  const float4 d = __ldcg(reinterpret_cast<const float4*>(c.in1 + (int64_t)b * c.K + k));
  if (c.kind == kChainProduct)
    return make_float4(__fmul_rn(a.x, d.x), __fmul_rn(a.y, d.y), __fmul_rn(a.z, d.z), __fmul_rn(a.w, d.w));
  if (c.kind == kChainSiluProduct) {
    auto silu = [](float x) { return __fdiv_rn(x, __fadd_rn(1.0f, expf(-x))); };
    return make_float4(__fmul_rn(silu(a.x), d.x), __fmul_rn(silu(a.y), d.y), __fmul_rn(silu(a.z), d.z),
                       __fmul_rn(silu(a.w), d.w));
  }
  return make_float4(__fadd_rn(a.x, d.x), __fadd_rn(a.y, d.y), __fadd_rn(a.z, d.z), __fadd_rn(a.w, d.w));
}

// The int8 code of x for scale s of a vector whose absmax m is nonzero (nz), as in the
// quantizer (m = 0 gives code 0 everywhere).
__device__ __forceinline__ uint32_t quant_byte(float x, float s, bool nz) {
  int v = 0;
  if (nz) {
    v = __float2int_rn(__fdiv_rn(x, s));
    v = v > 127 ? 127 : (v < -127 ? -127 : v);
  }
  return (uint32_t)(v & 0xFF);
}
__device__ __forceinline__ uint32_t quant4(float4 v, float s, bool nz) {
  return quant_byte(v.x, s, nz) | (quant_byte(v.y, s, nz) << 8) | (quant_byte(v.z, s, nz) << 16) |
         (quant_byte(v.w, s, nz) << 24);
}
#endif

}  // namespace nt
