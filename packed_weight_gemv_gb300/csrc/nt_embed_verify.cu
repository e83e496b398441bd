// nt_embed_verify.cu -- the two steps either side of the projections in a decode step:
//   input-table row gather ("The Neutrino Engine", § "The file is not the traffic": of the
//     input table only the rows of the current tokens are read; each row is dequantized by
//     its scale into the fp32 hidden vector the first layer quantizes), and
//   verify-pass acceptance (§ "The 0.6B model does not get to decide": the large model scores
//     every drafted position in one batched pass, the longest prefix where the draft agrees
//     with it is kept, and at the first disagreement the large model's own token is emitted).
#include "nt_kernels.cuh"

namespace nt {
namespace {

// One CTA per token: x[b][k] = fl((float)T[tok][k] * s[tok]); an out-of-range token gives a
// zero row and is counted.
__global__ void __launch_bounds__(256) embed_kernel(const int8_t* __restrict__ T, const float* __restrict__ s,
                                                   int V, int K, const int32_t* __restrict__ tokens,
                                                   float* __restrict__ x, uint32_t* __restrict__ n_bad) {
  dependent_launch_wait();
  const int b = blockIdx.x;
  const int t = tokens[b];
  const bool ok = t >= 0 && t < V;
  if (!ok && threadIdx.x == 0 && n_bad) atomicAdd(n_bad, 1u);
  const float sc = ok ? s[t] : 0.0f;
  float4* out = reinterpret_cast<float4*>(x + (int64_t)b * K);
  for (int g = threadIdx.x; g < K / 16; g += blockDim.x) {
    uint4 v = make_uint4(0, 0, 0, 0);
    if (ok) v = __ldg(reinterpret_cast<const uint4*>(T + (int64_t)t * K) + g);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int8_t* c = reinterpret_cast<const int8_t*>(&w[i]);
      out[4 * g + i] = make_float4(__fmul_rn((float)c[0], sc), __fmul_rn((float)c[1], sc),
                                   __fmul_rn((float)c[2], sc), __fmul_rn((float)c[3], sc));
    }
  }
}

__global__ void verify_kernel(const int32_t* __restrict__ draft, const int32_t* __restrict__ argmax, int B,
                              int32_t* __restrict__ emit, int32_t* __restrict__ n_emit) {
  dependent_launch_wait();
  if (threadIdx.x == 0 && blockIdx.x == 0) *n_emit = verify_accept_device(draft, argmax, B, emit);
}

}  // namespace

nt_status launch_embed(const int8_t* T, const float* s, int V, int K, const int32_t* tokens, int B, float* x,
                       uint32_t* n_bad, cudaStream_t st, bool pdl) {
  NT_CUDA_TRY(launch_kernel(embed_kernel, dim3(B), dim3(256), 0, st, pdl, T, s, V, K, tokens, x, n_bad));
  return check_launch("embed_kernel");
}

nt_status launch_verify(const int32_t* draft, const int32_t* argmax, int B, int32_t* emit, int32_t* n_emit,
                        cudaStream_t st, bool pdl) {
  NT_CUDA_TRY(launch_kernel(verify_kernel, dim3(1), dim3(32), 0, st, pdl, draft, argmax, B, emit, n_emit));
  return check_launch("verify_kernel");
}

}  // namespace nt

using namespace nt;

extern "C" {

nt_status nt_embed_rows(const int8_t* T, const float* s_T, int V, int K, const int32_t* tokens, int B,
                        float* x, uint32_t* n_bad_opt, void* stream) {
  clear_error();
  if (!T || !s_T || !tokens || !x) return set_error(NT_ERR_INVALID_ARG, "NULL tensor pointer");
  if (V < 1 || K < 16 || K % 16 != 0 || B < 1 || B > 65535)
    return set_error(NT_ERR_INVALID_ARG, "need V >= 1, 1 <= B <= 65535 and K a positive multiple of 16");
  if (!aligned(T, 16) || !aligned(x, 16)) return set_error(NT_ERR_ALIGNMENT, "T and x must be 16-byte aligned");
  if (!aligned(s_T, 4) || !aligned(tokens, 4) || (n_bad_opt && !aligned(n_bad_opt, 4)))
    return set_error(NT_ERR_ALIGNMENT, "s_T, tokens and the counter must be 4-byte aligned");
  NT_TRY(check_device());
  return launch_embed(T, s_T, V, K, tokens, B, x, n_bad_opt, reinterpret_cast<cudaStream_t>(stream));
}

nt_status nt_verify_accept(const int32_t* draft, const int32_t* argmax, int B, int32_t* emit, int32_t* n_emit,
                           void* stream) {
  clear_error();
  if (!argmax || !emit || !n_emit || (B > 1 && !draft)) return set_error(NT_ERR_INVALID_ARG, "NULL pointer");
  if (B < 1) return set_error(NT_ERR_INVALID_ARG, "need B >= 1");
  if (!aligned(argmax, 4) || !aligned(emit, 4) || !aligned(n_emit, 4) || (draft && !aligned(draft, 4)))
    return set_error(NT_ERR_ALIGNMENT, "int32 arrays must be 4-byte aligned");
  NT_TRY(check_device());
  return launch_verify(draft, argmax, B, emit, n_emit, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
