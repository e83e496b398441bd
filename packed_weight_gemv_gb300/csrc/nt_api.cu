// nt_api.cu -- the C ABI entry points of nt.h: argument validation, the device check, error
// strings and the per-call launches. The decode plan lives in nt_step.cu.
#include <atomic>
#include <cstdio>
#include <mutex>
#include <string>

#include "nt_kernels.cuh"

namespace nt {

namespace {
thread_local std::string g_last_error;

constexpr int kMaxDevices = 64;
std::atomic<int> g_dev_state[kMaxDevices];  // 0 unknown, 1 GB300, 2 other
std::atomic<int> g_dev_sms[kMaxDevices];
std::atomic<int> g_fault{0};
std::atomic<uint64_t> g_fault_timeout_ns{0};
}  // namespace

int test_fault() { return g_fault.load(std::memory_order_relaxed); }

uint64_t test_fault_timeout_ns(uint64_t dflt) {
  const uint64_t t = g_fault_timeout_ns.load(std::memory_order_relaxed);
  return (g_fault.load(std::memory_order_relaxed) != kFaultNone && t > 0) ? t : dflt;
}

nt_status set_error(nt_status s, const std::string& detail) {
  g_last_error = detail;
  return s;
}

nt_status clear_error() {
  g_last_error.clear();
  return NT_OK;
}

nt_status check_launch(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return set_error(NT_ERR_CUDA, std::string(what) + " launch: " + cudaGetErrorString(e));
  return NT_OK;
}

nt_status check_device(int* sm_count) {
  int dev = 0;
  NT_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return set_error(NT_ERR_UNSUPPORTED, "device index out of range");
  int state = g_dev_state[dev].load(std::memory_order_acquire);
  if (state == 0) {
    int major = 0, minor = 0, sms = 0;
    NT_CUDA_TRY(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
    NT_CUDA_TRY(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
    NT_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    g_dev_sms[dev].store(sms, std::memory_order_relaxed);
    state = (major == 10 && minor == 3) ? 1 : 2;
    g_dev_state[dev].store(state, std::memory_order_release);
  }
  if (state != 1) {
    char buf[96];
    snprintf(buf, sizeof buf, "device %d is not compute capability 10.3 (GB300)", dev);
    return set_error(NT_ERR_UNSUPPORTED, buf);
  }
  if (sm_count) *sm_count = g_dev_sms[dev].load(std::memory_order_relaxed);
  return NT_OK;
}

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  const int s = g_dev_sms[dev].load(std::memory_order_relaxed);
  return s > 0 ? s : 1;
}

}  // namespace nt

using namespace nt;

namespace {
cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

nt_status validate_ternary(const void* w, int layout, const float* s_w, int N, int K,
                           const int8_t* q, const float* s_x, int B, const float* y) {
  if (!w || !s_w || !q || !s_x || !y) return set_error(NT_ERR_INVALID_ARG, "NULL tensor pointer");
  if (N < 1 || K < 16 || K % 16 != 0 || B < 1)
    return set_error(NT_ERR_INVALID_ARG, "need N >= 1, B >= 1 and K a positive multiple of 16");
  if (layout != NT_LAYOUT_PLAIN && layout != NT_LAYOUT_TILED)
    return set_error(NT_ERR_INVALID_ARG, "layout must be NT_LAYOUT_PLAIN or NT_LAYOUT_TILED");
  if (!aligned(w, layout == NT_LAYOUT_TILED ? 16 : 4))
    return set_error(NT_ERR_ALIGNMENT, "weights must be 16-byte (tiled) or 4-byte (plain) aligned");
  if (!aligned(q, 16)) return set_error(NT_ERR_ALIGNMENT, "activations q must be 16-byte aligned");
  if (!aligned(s_w, 4) || !aligned(s_x, 4) || !aligned(y, 4))
    return set_error(NT_ERR_ALIGNMENT, "fp32 arrays must be 4-byte aligned");
  return NT_OK;
}
}  // namespace

extern "C" {

int nt_abi_version(void) { return NT_ABI_VERSION; }

const char* nt_status_string(nt_status s) {
  switch (s) {
    case NT_OK: return "ok";
    case NT_ERR_INVALID_ARG: return "invalid argument";
    case NT_ERR_ALIGNMENT: return "misaligned pointer";
    case NT_ERR_UNSUPPORTED: return "unsupported device (needs a GB300, compute capability 10.3)";
    case NT_ERR_CUDA: return "CUDA error";
    case NT_ERR_TIMEOUT: return "device-side wait timed out";
    case NT_ERR_WORKSPACE: return "workspace missing or too small";
    case NT_ERR_INVALID_CODE: return "invalid ternary field code (binary 10)";
  }
  return "unknown status";
}

const char* nt_last_error_string(void) { return g_last_error.c_str(); }

nt_status nt_set_test_fault(int fault, double timeout_ms) {
  clear_error();
  if (fault < kFaultNone || fault > kFaultPrefill) return set_error(NT_ERR_INVALID_ARG, "fault must be 0..3");
  g_fault_timeout_ns.store(timeout_ms > 0 ? (uint64_t)(timeout_ms * 1e6) : 0, std::memory_order_relaxed);
  g_fault.store(fault, std::memory_order_relaxed);
  return NT_OK;
}

nt_status nt_workspace_status(const void* ws, nt_status* device_status) {
  clear_error();
  if (!ws || !device_status) return set_error(NT_ERR_INVALID_ARG, "NULL argument");
  WsHeader h;
  NT_CUDA_TRY(cudaMemcpy(&h, ws, sizeof h, cudaMemcpyDeviceToHost));
  *device_status = h.error ? NT_ERR_TIMEOUT : NT_OK;
  if (h.error) {
    char buf[160];
    snprintf(buf, sizeof buf, "workspace: a bounded wait ran out (code %u, CTA %u)", h.error, h.error_cta);
    set_error(NT_ERR_TIMEOUT, buf);
  }
  return NT_OK;
}

nt_status nt_device_check(int* sm_count_opt) {
  clear_error();
  return check_device(sm_count_opt);
}

nt_status nt_quantize_act(const float* x, int B, int K, int8_t* q, float* s_x, void* stream) {
  clear_error();
  if (!x || !q || !s_x) return set_error(NT_ERR_INVALID_ARG, "NULL tensor pointer");
  if (B < 1 || K < 1) return set_error(NT_ERR_INVALID_ARG, "need B >= 1 and K >= 1");
  if (B > 65535 * 64) return set_error(NT_ERR_INVALID_ARG, "B too large");
  if (!aligned(x, 4) || !aligned(s_x, 4)) return set_error(NT_ERR_ALIGNMENT, "fp32 arrays must be 4-byte aligned");
  NT_TRY(check_device());
  return launch_quantize(x, B, K, q, s_x, as_stream(stream));
}

nt_status nt_repack_size(int N, int K, size_t* bytes) {
  clear_error();
  if (!bytes) return set_error(NT_ERR_INVALID_ARG, "NULL size pointer");
  if (N < 1 || K < 16 || K % 16 != 0)
    return set_error(NT_ERR_INVALID_ARG, "need N >= 1 and K a positive multiple of 16");
  *bytes = (size_t)(padded_rows(N) * tile_bytes(K) / 4);
  return NT_OK;
}

nt_status nt_repack_ternary(const uint32_t* w_plain, int N, int K, void* w_tiled,
                            uint32_t* n_invalid_opt, void* stream) {
  clear_error();
  if (!w_plain || !w_tiled) return set_error(NT_ERR_INVALID_ARG, "NULL tensor pointer");
  if (N < 1 || K < 16 || K % 16 != 0)
    return set_error(NT_ERR_INVALID_ARG, "need N >= 1 and K a positive multiple of 16");
  if (!aligned(w_plain, 4) || !aligned(w_tiled, 16))
    return set_error(NT_ERR_ALIGNMENT, "w_plain must be 4-byte and w_tiled 16-byte aligned");
  if (n_invalid_opt && !aligned(n_invalid_opt, 4)) return set_error(NT_ERR_ALIGNMENT, "counter must be 4-byte aligned");
  NT_TRY(check_device());
  return launch_repack(w_plain, N, K, static_cast<uint8_t*>(w_tiled), n_invalid_opt, as_stream(stream));
}

nt_status nt_validate_ternary(const uint32_t* w_plain, int N, int K, uint64_t* n_invalid_opt, void* stream) {
  clear_error();
  if (!w_plain) return set_error(NT_ERR_INVALID_ARG, "NULL tensor pointer");
  if (N < 1 || K < 16 || K % 16 != 0)
    return set_error(NT_ERR_INVALID_ARG, "need N >= 1 and K a positive multiple of 16");
  if (!aligned(w_plain, 4)) return set_error(NT_ERR_ALIGNMENT, "w_plain must be 4-byte aligned");
  NT_TRY(check_device());
  const cudaStream_t st = as_stream(stream);
  unsigned long long* d_count = nullptr;
  NT_CUDA_TRY(cudaMalloc(&d_count, sizeof *d_count));
  unsigned long long count = 0;
  cudaError_t e = cudaMemsetAsync(d_count, 0, sizeof *d_count, st);
  nt_status s = e == cudaSuccess ? launch_validate(w_plain, N, K, d_count, st)
                                 : set_error(NT_ERR_CUDA, std::string("cudaMemsetAsync: ") + cudaGetErrorString(e));
  if (s == NT_OK && (e = cudaMemcpyAsync(&count, d_count, sizeof count, cudaMemcpyDeviceToHost, st)) == cudaSuccess)
    e = cudaStreamSynchronize(st);
  if (s == NT_OK && e != cudaSuccess) s = set_error(NT_ERR_CUDA, std::string("validate: ") + cudaGetErrorString(e));
  cudaFree(d_count);
  if (s != NT_OK) return s;
  if (n_invalid_opt) *n_invalid_opt = count;
  if (count) {
    char buf[96];
    snprintf(buf, sizeof buf, "%llu invalid 10 field(s)", count);
    return set_error(NT_ERR_INVALID_CODE, buf);
  }
  return NT_OK;
}

nt_status nt_ternary_gemm_workspace_size(int N, int K, int B, int layout, size_t* bytes) {
  clear_error();
  if (!bytes) return set_error(NT_ERR_INVALID_ARG, "NULL size pointer");
  if (N < 1 || K < 16 || K % 16 != 0 || B < 1)
    return set_error(NT_ERR_INVALID_ARG, "need N >= 1, B >= 1 and K a positive multiple of 16");
  if (layout != NT_LAYOUT_PLAIN && layout != NT_LAYOUT_TILED)
    return set_error(NT_ERR_INVALID_ARG, "layout must be NT_LAYOUT_PLAIN or NT_LAYOUT_TILED");
  *bytes = 0;
  if (layout == NT_LAYOUT_TILED && tc_gemm_supported(B, K)) *bytes = tc_gemm_workspace_bytes(B, N, K);
  else if (layout == NT_LAYOUT_TILED && B >= kMmaMinBatch && B <= kMmaMaxBatch)
    *bytes = tc8_supported(N, K, B) ? tc8_ws_bytes(N, K, B) : mma_single_ws_bytes(N, K, B);
  return NT_OK;
}

nt_status nt_ternary_gemm(const void* w, int layout, const float* s_w, int N, int K,
                          const int8_t* q, const float* s_x, int B, float* y, int32_t* acc_opt,
                          void* ws, size_t ws_bytes, void* stream) {
  clear_error();
  NT_TRY(validate_ternary(w, layout, s_w, N, K, q, s_x, B, y));
  if (acc_opt && !aligned(acc_opt, 4)) return set_error(NT_ERR_ALIGNMENT, "acc must be 4-byte aligned");
  const bool tc = layout == NT_LAYOUT_TILED && tc_gemm_supported(B, K);
  if (tc && (!ws || !aligned(ws, 16) || ws_bytes < tc_gemm_workspace_bytes(B, N, K)))
    return set_error(NT_ERR_WORKSPACE, "tensor-core path: workspace NULL, misaligned or smaller than "
                                       "nt_ternary_gemm_workspace_size");
  NT_TRY(check_device());
  if (layout == NT_LAYOUT_PLAIN)
    return launch_gemv_plain(static_cast<const uint32_t*>(w), s_w, N, K, q, s_x, B, y, acc_opt,
                             as_stream(stream));
  if (tc)  // prefill-shaped batch: tensor cores
    return launch_gemm_tc(static_cast<const uint8_t*>(w), s_w, N, K, q, s_x, B, y, acc_opt, ws, as_stream(stream));
  if (tc8_supported(N, K, B) && ws && aligned(ws, 16) && ws_bytes >= tc8_ws_bytes(N, K, B))
    return launch_gemv_tc8(static_cast<const uint8_t*>(w), s_w, N, K, q, s_x, B, y, acc_opt, ws,
                           as_stream(stream));  // a few vectors with a workspace: tcgen05
  if (B >= kMmaMinBatch && B <= kMmaMaxBatch && ws && aligned(ws, 16) && ws_bytes >= mma_single_ws_bytes(N, K, B))
    return launch_gemv_mma_single(static_cast<const uint8_t*>(w), s_w, N, K, q, s_x, B, y, acc_opt, ws,
                                  as_stream(stream));  // a few vectors with a workspace: tensor cores
  MatDesc m{};
  m.w = static_cast<const uint8_t*>(w);
  m.s_w = s_w;
  m.q = q;
  m.s_x = s_x;
  m.y = y;
  m.acc = acc_opt;
  m.N = N;
  m.K = K;
  m.B = B;
  return launch_gemv_tiled(m, as_stream(stream));
}

nt_status nt_ternary_gemm_multi_workspace_size(int n, const int* N, int K, int B, size_t* bytes) {
  clear_error();
  if (!bytes || !N) return set_error(NT_ERR_INVALID_ARG, "NULL pointer");
  if (n < 1 || n > 8 || K < 16 || K % 16 != 0 || B < 1)
    return set_error(NT_ERR_INVALID_ARG, "need 1 <= n <= 8, B >= 1 and K a positive multiple of 16");
  for (int i = 0; i < n; ++i)
    if (N[i] < 1) return set_error(NT_ERR_INVALID_ARG, "every N must be >= 1");
  *bytes = tc_gemm_supported(B, K) ? tc_gemm_multi_workspace_bytes(B, n, N, K) : 0;
  return NT_OK;
}

nt_status nt_ternary_gemm_multi(int n, const void* const* w, const float* const* s_w, const int* N, int K,
                                const int8_t* q, const float* s_x, int B, float* const* y,
                                int32_t* const* acc_opt, void* ws, size_t ws_bytes, void* stream) {
  clear_error();
  if (!w || !s_w || !N || !y) return set_error(NT_ERR_INVALID_ARG, "NULL host array");
  if (n < 1 || n > 8) return set_error(NT_ERR_INVALID_ARG, "need 1 <= n <= 8");
  for (int i = 0; i < n; ++i) {
    NT_TRY(validate_ternary(w[i], NT_LAYOUT_TILED, s_w[i], N[i], K, q, s_x, B, y[i]));
    if (acc_opt && acc_opt[i] && !aligned(acc_opt[i], 4)) return set_error(NT_ERR_ALIGNMENT, "acc must be 4-byte aligned");
  }
  const bool tc = tc_gemm_supported(B, K);
  if (tc && (!ws || !aligned(ws, 16) || ws_bytes < tc_gemm_multi_workspace_bytes(B, n, N, K)))
    return set_error(NT_ERR_WORKSPACE, "tensor-core path: workspace NULL, misaligned or smaller than "
                                       "nt_ternary_gemm_multi_workspace_size");
  NT_TRY(check_device());
  if (tc)
    return launch_gemm_tc_multi(n, reinterpret_cast<const uint8_t* const*>(w), s_w, N, K, q, s_x, B, y, acc_opt, ws,
                                as_stream(stream));
  for (int i = 0; i < n; ++i) {  // small batches: the streaming kernel per matrix
    MatDesc m{};
    m.w = static_cast<const uint8_t*>(w[i]);
    m.s_w = s_w[i];
    m.q = q;
    m.s_x = s_x;
    m.y = y[i];
    m.acc = acc_opt ? acc_opt[i] : nullptr;
    m.N = N[i];
    m.K = K;
    m.B = B;
    NT_TRY(launch_gemv_tiled(m, as_stream(stream)));
  }
  return NT_OK;
}

nt_status nt_ternary_gemv(const void* w, int layout, const float* s_w, int N, int K,
                          const int8_t* q, const float* s_x, float* y, int32_t* acc_opt,
                          void* stream) {
  return nt_ternary_gemm(w, layout, s_w, N, K, q, s_x, 1, y, acc_opt, nullptr, 0, stream);
}

nt_status nt_int8_logits_workspace_size(int V, int K, int B, size_t* bytes) {
  clear_error();
  if (!bytes) return set_error(NT_ERR_INVALID_ARG, "NULL size pointer");
  if (V < 1 || K < 16 || K % 16 != 0 || B < 1)
    return set_error(NT_ERR_INVALID_ARG, "need V >= 1, B >= 1 and K a positive multiple of 16");
  *bytes = head_ws_bytes(B);
  return NT_OK;
}

nt_status nt_int8_logits_argmax(const int8_t* T, const float* s_T, int V, int K, const int8_t* q,
                                const float* s_x, int B, float* logits_opt, int32_t* argmax,
                                void* ws, size_t ws_bytes, void* stream) {
  clear_error();
  if (!T || !s_T || !q || !s_x || !argmax) return set_error(NT_ERR_INVALID_ARG, "NULL tensor pointer");
  if (V < 1 || K < 16 || K % 16 != 0 || B < 1)
    return set_error(NT_ERR_INVALID_ARG, "need V >= 1, B >= 1 and K a positive multiple of 16");
  if (!aligned(T, 16) || !aligned(q, 16)) return set_error(NT_ERR_ALIGNMENT, "T and q must be 16-byte aligned");
  if (!aligned(s_T, 4) || !aligned(s_x, 4) || !aligned(argmax, 4) || (logits_opt && !aligned(logits_opt, 4)))
    return set_error(NT_ERR_ALIGNMENT, "fp32/int32 arrays must be 4-byte aligned");
  if (!ws || ws_bytes < head_ws_bytes(B) || !aligned(ws, 16))
    return set_error(NT_ERR_WORKSPACE, "workspace NULL, misaligned or smaller than nt_int8_logits_workspace_size");
  NT_TRY(check_device());
  return launch_head(T, s_T, V, K, q, s_x, B, logits_opt, argmax, static_cast<HeadWs*>(ws),
                     as_stream(stream), /*pdl=*/true);
}

}  // extern "C"
