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

// One ternary projection in the tiled layout, B activation vectors.
struct MatDesc {
  const uint8_t* w;  // tiles (nt_repack_ternary output)
  const float* s_w;  // [N]
  const int8_t* q;   // [B][K]
  const float* s_x;  // [B]
  float* y;          // [B][N]
  int32_t* acc;      // [B][N] or null
  int N, K, B;
  int pad_;
};

// Scratch of the output-projection kernel's cross-CTA arg-max (caller-owned workspace).
constexpr int kHeadMaxCtas = 1024;
struct HeadPartial {
  float val;
  int idx;
};
struct HeadWs {
  unsigned int done;       // CTAs finished; the last one resets it to 0
  unsigned int pad_[3];
  HeadPartial part[1];     // [kHeadMaxCtas][B]
};
inline size_t head_ws_bytes(int B) { return 16 + sizeof(HeadPartial) * (size_t)kHeadMaxCtas * B; }

// Launchers (asynchronous on `st`; they return launch-configuration errors only).
nt_status launch_quantize(const float* x, int B, int K, int8_t* q, float* s, cudaStream_t st);
nt_status launch_quantize_jobs(const QuantJob* d_jobs, int n_jobs, int max_B, cudaStream_t st);
nt_status launch_repack(const uint32_t* w, int N, int K, uint8_t* out, uint32_t* n_invalid,
                        cudaStream_t st);
nt_status launch_gemv_plain(const uint32_t* w, const float* s_w, int N, int K, const int8_t* q,
                            const float* s_x, int B, float* y, int32_t* acc, cudaStream_t st);
nt_status launch_gemv_tiled(const MatDesc& m, cudaStream_t st);
// Several tiled projections in one launch: d_mats[n] in device memory, d_tile_prefix[n+1]
// their cumulative tile counts.
nt_status launch_gemv_tiled_group(const MatDesc* d_mats, const int64_t* d_tile_prefix, int n,
                                  int64_t total_tiles, int max_B, cudaStream_t st);
nt_status launch_head(const int8_t* T, const float* s_T, int V, int K, const int8_t* q,
                      const float* s_x, int B, float* logits, int32_t* argmax, HeadWs* ws,
                      cudaStream_t st);

nt_status launch_embed(const int8_t* T, const float* s, int V, int K, const int32_t* tokens, int B, float* x,
                       uint32_t* n_bad, cudaStream_t st);
nt_status launch_verify(const int32_t* draft, const int32_t* argmax, int B, int32_t* emit, int32_t* n_emit,
                        cudaStream_t st);

// Tensor-core ternary GEMM (tcgen05, bf16 operands, exact fp32 accumulation) for
// prefill-shaped batches of at least kTcMinBatch vectors.
constexpr int kTcMinBatch = 64;
bool tc_gemm_supported(int M, int K);
size_t tc_gemm_workspace_bytes(int M, int N, int K);
nt_status launch_gemm_tc(const uint8_t* w, const float* s_w, int N, int K, const int8_t* q, const float* s_x,
                         int M, float* y, int32_t* acc, void* ws, cudaStream_t st);

}  // namespace nt
