/*
 * nt.h -- C ABI of the packed ternary-weight decode library (libnt).
 *
 * What the library computes comes from "The Neutrino Engine" (Fermion Research):
 *
 *   - § "A 104 microsecond floor inside a 694 microsecond step": at batch one each weight
 *     feeds a single multiply-accumulate per token and nearly all of them are touched, so
 *     the weight bytes divided by the memory bandwidth give a floor on the time per token.
 *     Weights are consumed in their packed form: no floating-point copy of them exists,
 *     nothing is converted per token and each tensor is read at most once per token. The
 *     final projection covers every vocabulary row.
 *   - § "The file is not the traffic": per token, all ternary projection matrices (q, k, v,
 *     o, gate, up and down of every layer) are streamed, each row carrying a scale; the
 *     vocabulary tables hold int8 values in 151,936 rows of 4,096 columns, and every row of
 *     the output table is scored.
 *   - § "One changed token fails the release" and § "The 0.6B model does not get to decide":
 *     the emitted token is the greedy (arg-max) choice.
 *   - § "The same weights take four execution paths": the values are rearranged for each
 *     device once, when the model is loaded (here: nt_repack_ternary).
 *
 * The pages publish no kernel and no format, so the bit layout, the activation quantizer,
 * the epilogue rounding order and the tie rule below are this library's stated readings.
 *
 * Conventions (every call):
 *   - Returns nt_status; NT_OK is 0. No C++ exception crosses this boundary.
 *     nt_last_error_string() gives a detail string for the calling host thread.
 *   - Every tensor argument is a DEVICE pointer (CUDA global memory) owned by the caller,
 *     unless the argument says "host". The library never frees or retains caller memory
 *     beyond the call, except a decode plan, which keeps the pointers its descriptor named.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL = the legacy
 *     default stream) and never synchronize the device. Argument errors are detected on the
 *     host before any launch; launch errors return NT_ERR_CUDA; faults inside a kernel
 *     surface at the caller's next synchronization.
 *   - Inputs are never modified. Outputs are written in full.
 *   - Hot calls allocate nothing. Where scratch is needed the caller passes a workspace of
 *     the size the matching *_workspace_size call reports.
 *   - Sizes are int; every product that addresses memory is computed in 64-bit.
 *
 * Data formats:
 *   - Plain ternary layout (NT_LAYOUT_PLAIN), the exchange format: row-major uint32
 *     W[N][K/16]; trit k of row n is the 2-bit field at bits [2(k%16), 2(k%16)+1] of word
 *     W[n][k/16] (least-significant field first). Field codes: 00 -> 0, 01 -> +1,
 *     11 -> -1; 10 is invalid (decoded as 0 by every kernel, counted by
 *     nt_repack_ternary). K must be a multiple of 16.
 *   - Tiled ternary layout (NT_LAYOUT_TILED), made by nt_repack_ternary: rows are padded
 *     to Np = roundup(N, 4) and columns to Kp = roundup(K, 512) with zero trits. Tile t
 *     holds rows 4t..4t+3 as Kp/16 consecutive 16-byte groups; group j holds, for each of
 *     the 4 rows r (in order), one 32-bit word with trits 16j..16j+15 of row 4t+r. Inside
 *     a word, nibble i (i = 0..3) codes the pair (trit 16j+i, trit 16j+4+i) and nibble 4+i
 *     codes (trit 16j+8+i, trit 16j+12+i) with the pair codes
 *        (0,0)=0 (+1,0)=1 (-1,0)=2 (0,+1)=3 (+1,+1)=4 (-1,+1)=5 (+1,-1)=6 (-1,-1)=7
 *        (0,-1)=14
 *     -- the code the byte-permute decode in the kernels reads directly. Same 2 bits per
 *     trit as the plain layout; only padding adds bytes.
 *   - Activations: int8 q[B][K] row-major with one fp32 scale s_x[b] per vector.
 *   - Output table (lm-head): int8 T[V][K] row-major with fp32 row scales s_T[V].
 *
 * Arithmetic (the reading every kernel and the oracle follow):
 *   quantize:  m = max_k |x_k|; if m == 0 then s = 0 and q = 0; else s = m / 127 (fp32
 *              division, round to nearest even) and q_k = clamp(rint(x_k / s), -127, 127)
 *              with an fp32 division and round-half-to-even.
 *   project:   acc[n] = sum_k t[n][k] * q[k] (exact int32);
 *              y[n] = fl(fl(float(acc[n]) * s_w[n]) * s_x) -- int-to-float round to nearest,
 *              then two fp32 products, each rounded to nearest, no fused multiply-add.
 *   lm-head:   logit[v] = fl(fl(float(acc[v]) * s_T[v]) * s_x) the same way; argmax is the
 *              lowest v whose logit is maximal (+0 and -0 compare equal).
 */
#ifndef NT_H_
#define NT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define NT_ABI_VERSION 1

typedef enum nt_status {
  NT_OK = 0,
  NT_ERR_INVALID_ARG = 1, /* a size, enum or pointer argument is out of range or NULL */
  NT_ERR_ALIGNMENT = 2,   /* a pointer is not aligned as the call requires */
  NT_ERR_UNSUPPORTED = 3, /* the current device is not compute capability 10.3 (GB300) */
  NT_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed (detail string has it) */
  NT_ERR_TIMEOUT = 5,     /* a bounded device-side wait ran out (decode plan or workspace status) */
  NT_ERR_WORKSPACE = 6,   /* the workspace is NULL or smaller than the size call reported */
  NT_ERR_INVALID_CODE = 7 /* a plain ternary matrix holds the invalid field code 10 */
} nt_status;

enum nt_layout { NT_LAYOUT_PLAIN = 0, NT_LAYOUT_TILED = 1 };

/* Version of this header's ABI; equals NT_ABI_VERSION of the library that was built. */
int nt_abi_version(void);

/* Static English text for a status code. Never NULL. */
const char* nt_status_string(nt_status s);

/* Detail of the last error returned to the calling host thread ("" if none). The pointer
 * stays valid until the next nt_* call on the same thread. */
const char* nt_last_error_string(void);

/* Status of a workspace after the calls that used it ("A 104 microsecond floor ...": the
 * kernels that stream the weights wait on copies in flight, and every such wait here has a time
 * limit). Every workspace the library takes (nt_ternary_gemm, nt_ternary_gemm_multi,
 * nt_int8_logits_argmax) begins with a 16-byte status header. When a bounded device-side wait
 * of a call runs out (the streaming output projection: 250 ms; the tensor-core GEMMs: 2 s), the
 * kernel records an error code and its CTA there instead of hanging; that call's outputs are
 * invalid (the output projection writes -1 as every vector's arg-max). The code stays until the
 * caller zero-fills the whole workspace again, and until then the results of every call that
 * uses the workspace are invalid (the streaming output projection does no work and writes -1).
 *   ws             the workspace (device pointer, as passed to the calls); it must have been
 *                  zero-filled before its first use for its header to mean anything
 *   device_status  host: NT_OK, or NT_ERR_TIMEOUT (the detail string names the code and CTA)
 * Synchronous (reads 16 bytes); call it after synchronizing with the calls that used ws. */
nt_status nt_workspace_status(const void* ws, nt_status* device_status);

/* Test hook of the per-call timeout paths, for tests only: with `fault` set, the next launches
 * of one kernel issue no weight copies, so their consumers' bounded waits run out after
 * timeout_ms (<= 0 keeps the normal limits) and the call's workspace reports NT_ERR_TIMEOUT.
 *   fault 1: the streaming output projection (nt_int8_logits_argmax and its allocation-free
 *            variant at B = 1); 2: the tcgen05 path of nt_ternary_gemm (2..16 vectors with a
 *            workspace, N >= 128); 3: the prefill GEMM (64 or more vectors); 0: none.
 * Process-wide; set it only while no other thread launches library calls. No GPU fault is
 * involved: every wait gives up cleanly and the context stays usable. */
nt_status nt_set_test_fault(int fault, double timeout_ms);

/* Checks that the current CUDA device is a GB300 (compute capability 10.3) and reports its
 * SM count (host int*, may be NULL). Every other call performs the same check once per
 * device and returns NT_ERR_UNSUPPORTED on any other device. */
nt_status nt_device_check(int* sm_count_opt);

/* ---------------------------------------------------------------------------------------
 * Activation quantization (int8, one absmax scale per vector).
 * The pages state the int8 tables but not how activations reach int8; this call is the
 * plain symmetric absmax reading given at the top of this header.
 *   x    [B][K] fp32, 4-byte aligned         q   [B][K] int8
 *   s_x  [B] fp32 (output)                   B >= 1, K >= 1
 * Non-finite inputs give unspecified (but memory-safe) results.
 */
nt_status nt_quantize_act(const float* x, int B, int K, int8_t* q, float* s_x, void* stream);

/* ---------------------------------------------------------------------------------------
 * Load-time arrangement ("The same weights take four execution paths": values are
 * rearranged per device once, at load). Converts a plain ternary matrix into the
 * tiled layout. Run once per matrix; not part of a decode step.
 *   w_plain     [N][K/16] uint32, 4-byte aligned; K % 16 == 0, N >= 1
 *   w_tiled     nt_repack_size(N, K) bytes, 16-byte aligned (output)
 *   n_invalid_opt  device uint32 counter or NULL; when given, the call ADDS the number of
 *                  invalid 10 fields it met (each decoded as 0).
 */
nt_status nt_repack_size(int N, int K, size_t* bytes);

/* Load-time check of a plain ternary matrix for the one field code the format leaves
 * invalid (binary 10; the pages publish no format, so the 2-bit code is this library's
 * reading). The kernels decode such a field as 0 and never check it on the hot path; a loader
 * calls this once per matrix.
 *   w_plain        [N][K/16] uint32 (device, 4-byte aligned); K % 16 == 0, N >= 1
 *   n_invalid_opt  host uint64 or NULL: the number of invalid fields
 * Returns NT_OK when every field is 00, 01 or 11, NT_ERR_INVALID_CODE otherwise. Synchronous:
 * allocates an 8-byte device counter, runs one counting kernel on `stream`, waits for it and
 * frees the counter (not a hot call). */
nt_status nt_validate_ternary(const uint32_t* w_plain, int N, int K, uint64_t* n_invalid_opt,
                              void* stream);
nt_status nt_repack_ternary(const uint32_t* w_plain, int N, int K, void* w_tiled,
                            uint32_t* n_invalid_opt, void* stream);

/* ---------------------------------------------------------------------------------------
 * Ternary projection, batch 1 ("A 104 microsecond floor ...": each weight feeds one
 * multiply-accumulate per token; "The file is not the traffic": ternary projection
 * matrices with a scale per row).
 *   w        layout NT_LAYOUT_PLAIN ([N][K/16] uint32, 4-byte aligned) or
 *            NT_LAYOUT_TILED (nt_repack_ternary output, 16-byte aligned)
 *   s_w      [N] fp32 row scales            q  [K] int8      s_x  [1] fp32
 *   y        [N] fp32 (output)              acc_opt [N] int32 (output) or NULL
 *   K % 16 == 0, N >= 1.
 * The int32 sums are exact while they fit: |acc| <= 127 K, so for any K up to 16,909,320.
 * Past that, an input whose sum leaves the int32 range gets no exact result.
 */
nt_status nt_ternary_gemv(const void* w, int layout, const float* s_w, int N, int K,
                          const int8_t* q, const float* s_x, float* y, int32_t* acc_opt,
                          void* stream);

/* Ternary projection of B activation vectors that share the weights (the batched verify
 * pass in "The 0.6B model does not get to decide" scores several positions in one pass;
 * prefill pushes whole prompts through the same weights).
 *   q [B][K] int8, s_x [B], y [B][N] fp32 (output), acc_opt [B][N] int32 or NULL.
 * Results equal B independent nt_ternary_gemv calls, bit for bit. Any B >= 1 is accepted.
 * With NT_LAYOUT_TILED, B >= 64 and K <= 131072 the call runs on the tensor cores and needs
 * a workspace of nt_ternary_gemm_workspace_size bytes (16-byte aligned device memory; its
 * contents are scratch: an f16 copy of this call's activations, overwritten by the next call
 * that uses it -- the weights are read in their packed form and decoded inside the kernel;
 * calls sharing it must not overlap). A missing or short
 * workspace returns NT_ERR_WORKSPACE.
 * With NT_LAYOUT_TILED and 2 <= B <= 16 the workspace is optional: given one of at least
 * nt_ternary_gemm_workspace_size bytes (16-byte aligned, zero-filled before its first use;
 * calls sharing it must not overlap) the call runs on the tensor cores: from N >= 128 on
 * tcgen05 with the decoded trits in tensor memory (e4m3) and the activations split exactly
 * into two e4m3 digits kept in the workspace, below that f16 mma.sync; int32 partial sums of
 * K parts meet in the workspace, which every call leaves zero apart from the digit rows.
 * With ws NULL or short it runs the dp4a kernel. Otherwise the size is 0 and ws may be NULL.
 */
/* Every workspace of this call starts with the 16-byte status header nt_workspace_status
 * reads (the tensor-core kernels' waits are bounded at 2 s); after NT_ERR_TIMEOUT the whole
 * workspace must be zero-filled again before its next use. */
nt_status nt_ternary_gemm_workspace_size(int N, int K, int B, int layout, size_t* bytes);
nt_status nt_ternary_gemm(const void* w, int layout, const float* s_w, int N, int K,
                          const int8_t* q, const float* s_x, int B, float* y,
                          int32_t* acc_opt, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------
 * int8 output projection with fused greedy arg-max ("A 104 microsecond floor ...": the
 * last projection turns the final hidden vector into a score for every vocabulary entry;
 * "The file is not the traffic": int8 tables, 151,936 x 4,096, every output row scored;
 * greedy decode per "One changed token fails the release").
 *   T [V][K] int8 (16-byte aligned, K % 16 == 0)   s_T [V] fp32
 *   q [B][K] int8 (16-byte aligned)                s_x [B] fp32
 *   logits_opt [B][V] fp32 (output) or NULL        argmax [B] int32 (output)
 *   ws: nt_int8_logits_workspace_size(V, K, B) bytes of device memory that is zero-filled
 *       before its first use; every call returns it to that state (unless a wait ran out:
 *       see nt_workspace_status). Calls that share one workspace must not overlap on the
 *       device.
 * The int32 sums are exact while they fit: |acc| <= 127 * 127 K, so for any K up to 133,144
 * (the 8B-shaped table has K = 4,096). Past that, a sum that leaves the int32 range gets no
 * exact result.
 * B = 1 streams T through the persistent dp4a kernel; 2 <= B <= 16 reads T once on the
 * tensor cores (f16 MMA of exactly converted int8 with exact int32 sums); larger B takes
 * several passes of 16. Logits and arg-max are the same in every case.
 * At B = 1 the call is a programmatic dependent launch: it starts streaming T while the
 * previous kernel on the stream finishes, and reads q, s_x and s_T and writes its outputs
 * only after that kernel has completed. T is treated as a constant: do not write it with the
 * kernel launched immediately before this call on the same stream. A bounded wait of the
 * streaming kernel that runs out (250 ms) makes argmax -1 for every vector and leaves
 * NT_ERR_TIMEOUT in the workspace's status header (nt_workspace_status).
 */
nt_status nt_int8_logits_workspace_size(int V, int K, int B, size_t* bytes);
nt_status nt_int8_logits_argmax(const int8_t* T, const float* s_T, int V, int K,
                                const int8_t* q, const float* s_x, int B, float* logits_opt,
                                int32_t* argmax, void* ws, size_t ws_bytes, void* stream);

/* The same output projection and arg-max for callers that cannot allocate device memory.
 * The pages have no counterpart to this call; it is a convenience of this library. Some
 * callers cannot obtain a workspace: a plugin whose host process owns every device
 * allocation, a serving loop that must not call cudaMalloc (it can synchronize the device),
 * or code under a fixed memory budget. This call takes only the inputs and outputs of
 * nt_int8_logits_argmax (same meaning, layout and alignment) and allocates nothing: its
 * scratch is a fixed ~128 KiB array in the library's device globals, present on every device
 * that loads the library until the process exits.
 *   B must be <= 16 (the scratch's size); larger B returns NT_ERR_INVALID_ARG.
 *   Every call looks up the current device's scratch address (the first call on a device
 *   may load the library's device code); make that first call before any stream capture.
 *   Every call on a device shares the one scratch array, so calls that overlap on that
 *   device (e.g. from two streams) race and give wrong results; serialize them. Each call
 *   clears the part of the scratch that must start at zero (an asynchronous 16-byte memset
 *   on `stream` before the kernel), so a wait that ran out in one call does not carry over:
 *   the only sign of it is -1 as that call's arg-max (B = 1, the streaming kernel).
 */
nt_status nt_int8_logits_argmax_noalloc(const int8_t* T, const float* s_T, int V, int K,
                                        const int8_t* q, const float* s_x, int B,
                                        float* logits_opt, int32_t* argmax, void* stream);

/* Several tiled projections of the same activations (q, k and v read one input, and so do
 * gate and up): y_i = nt_ternary_gemm(w_i, NT_LAYOUT_TILED, s_w_i, N_i, K, q, s_x, B) for
 * i < n, in one call. With B >= 64 the tensor-core path converts the activations once for all
 * n matrices and runs one tile set over their rows (more tiles per launch, fewer launches);
 * smaller B runs the streaming kernel per matrix. w, s_w, N, y: host arrays of n (1..8)
 * entries (device pointers, as nt_ternary_gemm); acc_opt: NULL or a host array of n device
 * pointers, each may be NULL. ws: device workspace of
 * nt_ternary_gemm_multi_workspace_size(n, N, K, B) bytes (0 below 64 vectors). */
nt_status nt_ternary_gemm_multi_workspace_size(int n, const int* N, int K, int B, size_t* bytes);
nt_status nt_ternary_gemm_multi(int n, const void* const* w, const float* const* s_w, const int* N,
                                int K, const int8_t* q, const float* s_x, int B, float* const* y,
                                int32_t* const* acc_opt, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------
 * Input-table row gather ("The file is not the traffic": of the input table only the rows of
 * the current tokens are read). x[b][k] = fl((float)T[tokens[b]][k] * s_T[tokens[b]]): the
 * int8 value converted exactly, one rounded product -- the fp32 hidden vector the first layer
 * quantizes (the pages do not say how the row becomes the hidden vector; this is the plain
 * reading of an int8 table with row scales).
 *   T [V][K] int8 (16-byte aligned, K % 16 == 0)   s_T [V] fp32   tokens [B] int32
 *   x [B][K] fp32 (output, 16-byte aligned)
 *   n_bad_opt: device uint32 counter or NULL; the call ADDS the number of tokens outside
 *   [0, V), whose rows are written as zeros.
 */
nt_status nt_embed_rows(const int8_t* T, const float* s_T, int V, int K, const int32_t* tokens,
                        int B, float* x, uint32_t* n_bad_opt, void* stream);

/* ---------------------------------------------------------------------------------------
 * Verify-pass acceptance ("The 0.6B model does not get to decide": the large model scores
 * every drafted position in one batched pass; the longest prefix on which the draft agrees
 * with it is kept, and at the first disagreement the large model's own token is emitted).
 * Positions 0..B-1 of the verify pass hold the last emitted token and the drafts
 * draft[0..B-2]; argmax[i] is the pass's greedy token after position i (for example the
 * argmax output of nt_int8_logits_argmax with B vectors). With j leading drafts accepted
 * (draft[i] == argmax[i] for all i < j), emit[0..j] = draft[0..j-1], argmax[j] and
 * *n_emit = j + 1. All pointers device; draft may be NULL when B == 1. One tiny kernel.
 */
nt_status nt_verify_accept(const int32_t* draft, const int32_t* argmax, int B, int32_t* emit,
                           int32_t* n_emit, void* stream);

/* ---------------------------------------------------------------------------------------
 * Attention side of a layer ("At 26K tokens, the cache becomes larger than the model": 36
 * layers x 8 key-value heads x 128 dimensions at 16 bits = 147,456 bytes per cached position;
 * grouped-query attention, so the 32 query heads read the 8 key-value heads). The pages give
 * no formulas for the layer's other operations; the plain readings are stated per call.
 * Head dimension D must be 128 (NT_ERR_UNSUPPORTED otherwise).
 *
 * nt_attention_decode: B new positions attend over a cache of T rows whose last B rows are
 * those positions (they were appended first, e.g. by nt_rope_append): position b sees rows
 * 0 .. T - B + b. out[b][h] = sum_t softmax_t(q[b][h] . k[g][t] / sqrt(D)) v[g][t] with
 * g = h / (Hq / Hkv). Both products on the tensor cores with bf16 operands and fp32 sums: q
 * enters as three bf16 terms and the softmax weights as two, so the result is within a few
 * 1e-6 of the exact value relative to max |v| (one launch: units of cache positions per
 * key-value head, merged by the last unit to finish).
 *   q [B][Hq][D] fp32; k_cache, v_cache [Hkv][t_stride][D] bf16 bit patterns (16-byte
 *   aligned); out [B][Hq][D] fp32; Hq / Hkv in {1, 2, 4, 8}; 1 <= B <= 64; B <= T <= t_stride.
 *   ws: device workspace of nt_attention_workspace_size(B, Hq, Hkv, T) bytes (16-byte
 *   aligned), all zero before its first use (every call leaves its counters zero again);
 *   calls sharing a workspace must not overlap.
 */
nt_status nt_attention_workspace_size(int B, int Hq, int Hkv, int T, size_t* bytes);
nt_status nt_attention_decode(const float* q, const uint16_t* k_cache, const uint16_t* v_cache,
                              int B, int Hq, int Hkv, int D, int T, int t_stride, float* out,
                              void* ws, size_t ws_bytes, void* stream);

/* Rotary embedding of B new positions pos0 .. pos0 + B - 1 and their append to the cache.
 * Rotate-half pairing (dimension i with i + D/2) by the angle pos * base^(-2i/D), the angles
 * formed and reduced modulo 2 pi in double precision, their sine and cosine and the rotations
 * in fp32. q_out[b][h] = rotated q[b][h] (fp32);
 * k_cache[g][pos0 + b] = bf16(rotated k_new[b][g]); v_cache[g][pos0 + b] = bf16(v_new[b][g])
 * (round to nearest even). q [B][Hq][D], k_new / v_new [B][Hkv][D] fp32; base > 1 (10000 is
 * the textbook value); pos0 + B <= t_stride. q_out may alias q. */
nt_status nt_rope_append(const float* q, const float* k_new, const float* v_new, int B, int Hq,
                         int Hkv, int D, int pos0, float base, float* q_out, uint16_t* k_cache,
                         uint16_t* v_cache, int t_stride, void* stream);

/* RMS normalisation of B vectors of length D: y = fl(fl(x * r) * gamma) with
 * r = fl32(1 / sqrt(mean(x^2) + eps)) formed in double. x, y [B][D]; gamma [D]; y may alias x. */
nt_status nt_rmsnorm(const float* x, const float* gamma, int B, int D, float eps, float* y,
                     void* stream);

/* ---------------------------------------------------------------------------------------
 * Decode step: every projection of every layer, then optionally the output projection, in
 * one submission ("A 104 microsecond floor ...": on the instrumented A100 step, roughly
 * 590 of 694 microseconds were spent across about 120 kernel boundaries rather than in
 * DRAM transfers; fusing the step into one kernel moved that cost into its grid-wide
 * synchronisation instead of removing it).
 */
enum nt_step_mode {
  NT_STEP_INDEPENDENT = 0, /* every projection has its own supplied input; no ordering */
  NT_STEP_ORDERED = 1,     /* per layer {q,k,v} -> {o} -> {gate,up} -> {down}, layer by
                              layer, each stage complete before the next one starts */
  NT_STEP_CHAINED = 2      /* the ORDERED stages, each quantizing what the previous stages
                              produced ("A 104 microsecond floor ...": each layer applies its
                              matrices to the current activations and the engine reads no
                              tensor twice per token). With hidden h (fp32 [B][d], d = the q
                              projection's K) and every + and * one fp32 rounding:
                                {q,k,v} <- Q(h);
                                {o}     <- Q(u), u = attention over one cached position: query
                                           head i (head_dim columns) takes the value head
                                           i / G, G = o.K / v.N (grouped-query attention);
                                {gate,up} <- Q(a), a = h + y_o;
                                {down}  <- Q(y_gate * y_up);
                                next h = a + y_down; the output projection scores Q(h_last).
                              h of the first layer is proj[0].x (or the gathered rows when it
                              points at embed_x); every other x and head_x is ignored. Every
                              projection's q / s_x (and head_q / head_sx) receive the codes and
                              scale of its input. Needs matching shapes (d = k.K = v.K = o.N =
                              gate.K = up.K = down.N = head_K, o.K = q.N, gate.N = up.N =
                              down.K, v.N = k.N a multiple of head_dim dividing o.K). The plan
                              owns the residual stream (B x d fp32). Normalisations, rotary
                              embedding and the gate's activation function are not applied. */
};
enum nt_launcher {
  NT_LAUNCH_PERSISTENT = 0, /* one cooperative kernel streams the whole step */
  NT_LAUNCH_GRAPH = 1,      /* a CUDA graph of one launch per stage, replayed per step */
  NT_LAUNCH_STREAM = 2      /* the same launches issued one by one (the launch-gap case) */
};

/* One projection. All pointers device; the weights in NT_LAYOUT_TILED. The fp32 inputs x
 * (and head_x) of an NT_STEP_INDEPENDENT or NT_STEP_ORDERED plan may also point into pinned
 * host memory that the device can address (page-locked, mapped; on this platform every pinned
 * allocation is): the step's first phase then reads them over the host link each step, with
 * no separate copy. */
typedef struct nt_proj {
  int N, K;
  const void* w;     /* nt_repack_ternary output for an N x K matrix */
  const float* s_w;  /* [N] */
  const float* x;    /* [B][K] fp32 input to quantize inside the step, or NULL */
  int8_t* q;         /* [B][K] int8: written by the step when x != NULL, else read */
  float* s_x;        /* [B]: written when x != NULL, else read */
  float* y;          /* [B][N] fp32 output */
} nt_proj;

typedef struct nt_decode_desc {
  int n_layers;          /* >= 1 */
  int batch;             /* B, 1..16 */
  const nt_proj* proj;   /* host array of n_layers * 7 entries, per layer in the order
                            q, k, v, o, gate, up, down; copied at plan creation */
  /* Output projection; head_T == NULL leaves it out. */
  const int8_t* head_T;  /* [V][K] int8 */
  const float* head_s;   /* [V] */
  int head_V, head_K;
  const float* head_x;   /* [B][K] fp32 hidden to quantize in the step, or NULL */
  int8_t* head_q;        /* [B][K] int8 (written when head_x != NULL, else read) */
  float* head_sx;        /* [B] */
  float* head_logits;    /* [B][V] fp32 or NULL */
  int32_t* head_argmax;  /* [B] int32 */
  int mode;              /* enum nt_step_mode */
  int launcher;          /* enum nt_launcher */
  double timeout_ms;     /* bound on every device-side wait of the persistent kernel and of
                            the tcgen05 batched kernel; <= 0 selects 250 ms */
  int test_fault;        /* 0 in normal use. 1 makes the first grid barrier of the
                            persistent kernel wait for one arrival more than the grid makes,
                            so that wait runs out after timeout_ms and the step reports
                            NT_ERR_TIMEOUT: the hook the tests of the timeout path use. 2
                            does the same for the tcgen05 batched kernel (independent plans,
                            2..16 vectors, graph / stream launchers): its producers issue no
                            copies, so the consumers' waits run out. */
  /* Input-table gather at the start of the step (nt_embed_rows); embed_T == NULL leaves it
     out. Projection inputs (x) may point into embed_x: the gather finishes before any
     input is quantized. Tokens outside [0, embed_V) give zero rows. */
  const int8_t* embed_T;   /* [embed_V][embed_K] int8 */
  const float* embed_s;    /* [embed_V] */
  int embed_V, embed_K;
  const int32_t* tokens;   /* [batch] */
  float* embed_x;          /* [batch][embed_K] fp32 output */
  /* Verify-pass acceptance after the output projection (nt_verify_accept on head_argmax);
     needs the head; verify_emit == NULL leaves it out. */
  const int32_t* verify_draft;  /* [batch - 1] drafted tokens (NULL when batch == 1) */
  int32_t* verify_emit;         /* [batch] emitted tokens */
  int32_t* verify_n;            /* [1] number of emitted tokens */
  int head_dim;                 /* NT_STEP_CHAINED: dimensions per attention head, a multiple of
                                   4 (0 selects 128, "At 26K tokens ...": 128 per head) */
  /* NT_STEP_CHAINED with the layer's attention side (attn_k_cache != NULL; head_dim must be
     128). The persistent launcher runs one cooperative launch per segment of stages between
     two attention sides ({q,k,v} of layer 0; then {o},{gate,up},{down} of layer l with
     {q,k,v} of layer l + 1; the last segment ends with the output projection), the rotation,
     cache append and attention launches in between: 3 launches per layer.
     Per layer, with the step's B vectors at positions pos .. pos + B - 1:
       {q,k,v} <- Q(rmsnorm(h) * norm_attn[l]);
       q, k rotated (nt_rope_append); k, v appended to the layer's cache at rows pos ..;
       u = attention of the B positions over rows 0 .. pos + B - 1 (nt_attention_decode);
       {o} <- Q(u); a = h + y_o; {gate,up} <- Q(rmsnorm(a) * norm_ffn[l]);
       {down} <- Q(silu(y_gate) * y_up); next h = a + y_down;
     the output projection scores Q(rmsnorm(h_last) * norm_final). A NULL weight array or
     vector leaves that normalisation out. */
  uint16_t* const* attn_k_cache; /* host array [n_layers] of device [Hkv][attn_t_stride][128] bf16 */
  uint16_t* const* attn_v_cache; /* Hkv = k.N / 128; Hq = q.N / 128; Hq / Hkv in {1, 2, 4, 8} */
  int attn_t_stride;             /* rows per head in each cache */
  int attn_pos;                  /* position of the first vector (rows 0 .. attn_pos - 1 are filled);
                                    nt_decode_plan_set_position changes it between steps */
  float rope_base;               /* <= 0 selects 10000 */
  float norm_eps;                /* <= 0 selects 1e-6 */
  const float* const* norm_attn; /* host array [n_layers] of device [d] weights, or NULL */
  const float* const* norm_ffn;  /* host array [n_layers] of device [d] weights, or NULL */
  const float* norm_final;       /* device [d] weights, or NULL */
} nt_decode_desc;

typedef struct nt_decode_plan nt_decode_plan;

/* Validates the descriptor, allocates the plan's own small device state (schedule, barrier
 * counters, workspace) and, for NT_LAUNCH_GRAPH, builds the graph. Not a hot call. */
nt_status nt_decode_plan_create(const nt_decode_desc* d, nt_decode_plan** plan);

/* Runs one decode step on `stream`. Allocates nothing. Steps of one plan must not overlap
 * on the device (issue them on one stream). NT_LAUNCH_PERSISTENT needs every CTA of its
 * grid resident at once and returns NT_ERR_CUDA if the device cannot provide that.
 * A persistent step that is one launch (every plan but a chained one with attention) takes
 * the same launch parameters on every call -- its grid-barrier counter is reset on the device
 * by the CTA that finishes last -- so it can be recorded into a CUDA graph by stream capture
 * and replayed; inputs written in place between replays are read by the next replay. A
 * trace or capture buffer set after recording is not seen by the recorded launch. A chained
 * step with attention (several launches that count grid barriers on the host) returns
 * NT_ERR_UNSUPPORTED when called while its stream is being recorded. */
nt_status nt_decode_step(nt_decode_plan* plan, void* stream);

/* After the caller has synchronized with the last step: NT_OK, or NT_ERR_TIMEOUT when a
 * bounded wait inside the persistent kernel or the tcgen05 batched kernel (independent plans
 * with 2..16 vectors on the graph / stream launchers) ran out (the step's outputs are then
 * invalid and the plan must be reset before reuse). Reads the device status word
 * (synchronous). */
nt_status nt_decode_step_status(nt_decode_plan* plan, nt_status* device_status);

/* Chained plans with attention: the position of the next step's first vector, set in stream
 * order on `stream` (one tiny kernel; graph launchers read it at run time). pos + batch must
 * not exceed attn_t_stride. */
nt_status nt_decode_plan_set_position(nt_decode_plan* plan, int pos, void* stream);

/* Clears the plan's device-side error word and barrier counters (synchronous). */
nt_status nt_decode_plan_reset(nt_decode_plan* plan);

/* Step timeline of the persistent launcher, the instrumentation "A 104 microsecond floor
 * ..." describes for one decoder step (Fig. 1: DRAM time against launch/dependency latency).
 * nt_decode_plan_trace_layout reports the grid size G and the number of grid barriers S per
 * step (host ints). A trace buffer is G * (S + 1) * 4 device uint64 values; record (c, b) =
 * trace[(c * (S + 1) + b) * 4 + i] holds %globaltimer nanoseconds of CTA c:
 *   b = 0:      i = 0 kernel start, i = 1 consumers done with the whole step;
 *   b = 1..S:   i = 0 consumers done with the work before barrier b, i = 1 barrier b passed,
 *               i = 2 the next stage's activations in shared memory.
 * nt_decode_plan_set_trace installs (or, with NULL, removes) the buffer; every later step
 * of the plan overwrites it. Other launchers and stream/graph plans record nothing. */
nt_status nt_decode_plan_trace_layout(const nt_decode_plan* plan, int* grid, int* barriers);
nt_status nt_decode_plan_set_trace(nt_decode_plan* plan, unsigned long long* trace);

/* Stage inputs of a chained plan, as the step quantized them: the fp32 vector each stage
 * turned into int8 codes after every operation before it (residual additions, RMS
 * normalisation, attention, the SiLU-gated product), for checking each stage on its own
 * inputs ("A 104 microsecond floor ...": each layer applies its matrices to the current
 * activations). nt_decode_plan_capture_size reports the buffer's length in floats (host
 * size_t): per stage in step order -- per layer {q,k,v}, {o}, {gate,up}, {down}, then the
 * output projection if the plan has one -- B x K values, K the stage's reduction length,
 * vector-major. nt_decode_plan_set_capture installs a 16-byte aligned device buffer of that
 * length (or, with NULL, removes it; synchronous); every later step of the plan overwrites
 * it. Only NT_STEP_CHAINED plans (NT_ERR_INVALID_ARG otherwise). */
nt_status nt_decode_plan_capture_size(const nt_decode_plan* plan, size_t* floats);
nt_status nt_decode_plan_set_capture(nt_decode_plan* plan, float* buf);

/* Releases the plan and everything it allocated. NULL is ignored. */
void nt_decode_plan_destroy(nt_decode_plan* plan);

#ifdef __cplusplus
}
#endif

#endif /* NT_H_ */
