// nt_noalloc.cu -- the output projection with fused arg-max for callers that cannot allocate
// device memory: the cross-CTA scratch lives in a fixed array in the library's own device
// globals instead of a caller-provided workspace.
//
// Some callers have no way to obtain device memory for a workspace: a plugin whose host
// process owns every device allocation through its own allocator, a serving loop that must
// not call cudaMalloc (it can synchronize the device and stall unrelated streams), or code
// running under a fixed memory budget where a late allocation may fail. This entry point
// needs only the inputs and outputs the caller already has.
#include <string>

#include "nt_kernels.cuh"

namespace nt {
namespace {

// Largest batch the fixed scratch serves; the scratch holds the arg-max counter and one
// partial (best logit, row) per CTA and batch row for up to kHeadMaxCtas CTAs.
constexpr int kNoAllocMaxBatch = 16;
constexpr size_t kNoAllocScratchBytes = 16 + sizeof(HeadPartial) * (size_t)kHeadMaxCtas * kNoAllocMaxBatch;

// One copy per device that loads the library, held until the process exits (~128 KiB).
static __device__ __align__(256) unsigned char g_head_scratch[kNoAllocScratchBytes];

// Device address of the current device's scratch. In host code g_head_scratch names a
// host-side stand-in, not device memory, so only the address from cudaGetSymbolAddress may be
// handed to a kernel. It is looked up on every call (a cheap lookup once the module is loaded),
// so a device reset that reloads the module and moves the array is harmless.
nt_status scratch_for_current_device(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_head_scratch);
  if (e != cudaSuccess || !p)
    return set_error(NT_ERR_CUDA, std::string("cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(e));
  *out = p;
  return NT_OK;
}

}  // namespace
}  // namespace nt

using namespace nt;

extern "C" nt_status nt_int8_logits_argmax_noalloc(const int8_t* T, const float* s_T, int V, int K,
                                                   const int8_t* q, const float* s_x, int B,
                                                   float* logits_opt, int32_t* argmax, void* stream) {
  clear_error();
  if (!T || !s_T || !q || !s_x || !argmax) return set_error(NT_ERR_INVALID_ARG, "NULL tensor pointer");
  if (V < 1 || K < 16 || K % 16 != 0 || B < 1)
    return set_error(NT_ERR_INVALID_ARG, "need V >= 1, B >= 1 and K a positive multiple of 16");
  if (B > kNoAllocMaxBatch)
    return set_error(NT_ERR_INVALID_ARG, "nt_int8_logits_argmax_noalloc serves batch <= 16 (its fixed "
                                         "scratch size); use nt_int8_logits_argmax for larger batches");
  if (!aligned(T, 16) || !aligned(q, 16)) return set_error(NT_ERR_ALIGNMENT, "T and q must be 16-byte aligned");
  if (!aligned(s_T, 4) || !aligned(s_x, 4) || !aligned(argmax, 4) || (logits_opt && !aligned(logits_opt, 4)))
    return set_error(NT_ERR_ALIGNMENT, "fp32/int32 arrays must be 4-byte aligned");
  NT_TRY(check_device());
  void* scratch = nullptr;
  NT_TRY(scratch_for_current_device(&scratch));
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // The scratch keeps whatever the previous call left; the CTA counter must start at zero.
  NT_CUDA_TRY(cudaMemsetAsync(scratch, 0, 16, st));
  return launch_head(T, s_T, V, K, q, s_x, B, logits_opt, argmax, static_cast<HeadWs*>(scratch), st);
}
