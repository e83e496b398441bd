// nt_step.cu -- the decode plan: every projection of every layer, then the output projection,
// submitted as one step ("The Neutrino Engine", § "A 104 microsecond floor inside a 694
// microsecond step": on the instrumented step most of the time went to about 120 kernel
// boundaries, and one fused kernel's software barriers brought the waits back).
//
// Launchers:
//   NT_LAUNCH_STREAM     one launch per stage issued on the caller's stream every step;
//   NT_LAUNCH_GRAPH      the same launches captured once into a CUDA graph, replayed per step;
//   NT_LAUNCH_PERSISTENT one cooperative kernel streams the whole step (nt_persist.cu).
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <string>
#include <vector>

#include "nt_kernels.cuh"
#include "nt_step.cuh"

using namespace nt;

namespace {

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Shapes of a chained step: every stage input has the length its matrices reduce over.
nt_status validate_chain(const nt_decode_desc* d) {
  const int hd = d->head_dim > 0 ? d->head_dim : 128;
  if (hd % 4 != 0) return set_error(NT_ERR_INVALID_ARG, "chained: head_dim must be a multiple of 4");
  if (!d->proj[0].x) return set_error(NT_ERR_INVALID_ARG, "chained: proj[0].x (the first hidden state) is NULL");
  const int dm = d->proj[0].K;
  for (int l = 0; l < d->n_layers; ++l) {
    const nt_proj* p = d->proj + l * kProjPerLayer;
    const nt_proj &q = p[0], &k = p[1], &v = p[2], &o = p[3], &g = p[4], &u = p[5], &dn = p[6];
    const std::string at = "chained: layer " + std::to_string(l) + ": ";
    if (q.K != dm || k.K != dm || v.K != dm || o.N != dm || g.K != dm || u.K != dm || dn.N != dm)
      return set_error(NT_ERR_INVALID_ARG, at + "q/k/v/gate/up K and o/down N must all equal proj[0].K");
    if (o.K != q.N || k.N != v.N || g.N != u.N || dn.K != g.N)
      return set_error(NT_ERR_INVALID_ARG, at + "need o.K == q.N, k.N == v.N, gate.N == up.N == down.K");
    if (v.N % hd != 0 || o.K % v.N != 0)
      return set_error(NT_ERR_INVALID_ARG, at + "v.N must be a multiple of head_dim and divide o.K");
    for (int i = 0; i < kProjPerLayer; ++i)
      if (!aligned(p[i].y, 16)) return set_error(NT_ERR_ALIGNMENT, at + "outputs must be 16-byte aligned");
  }
  if (!aligned(d->proj[0].x, 16)) return set_error(NT_ERR_ALIGNMENT, "chained: proj[0].x must be 16-byte aligned");
  if (d->head_T && d->head_K != dm) return set_error(NT_ERR_INVALID_ARG, "chained: head_K must equal proj[0].K");
  if (d->attn_k_cache) {  // the attention side
    if (hd != 128) return set_error(NT_ERR_UNSUPPORTED, "chained steps with attention need head_dim 128");
    const int Hq = d->proj[0].N / 128, Hkv = d->proj[1].N / 128;
    if (d->proj[0].N % 128 || d->proj[1].N % 128 || Hkv < 1 || Hq % Hkv != 0)
      return set_error(NT_ERR_INVALID_ARG, "attention: q.N and k.N must be multiples of 128 with Hq a multiple of Hkv");
    const int G = Hq / Hkv;
    if (G != 1 && G != 2 && G != 4 && G != 8) return set_error(NT_ERR_UNSUPPORTED, "attention: Hq / Hkv must be 1, 2, 4 or 8");
    if (!d->attn_v_cache) return set_error(NT_ERR_INVALID_ARG, "attention: attn_v_cache is NULL");
    if (d->attn_pos < 0 || (int64_t)d->attn_pos + d->batch > d->attn_t_stride)
      return set_error(NT_ERR_INVALID_ARG, "attention: need 0 <= attn_pos and attn_pos + batch <= attn_t_stride");
    for (int l = 0; l < d->n_layers; ++l) {
      if (d->proj[l * kProjPerLayer].N != Hq * 128 || d->proj[l * kProjPerLayer + 1].N != Hkv * 128)
        return set_error(NT_ERR_INVALID_ARG, "attention: every layer needs the same head counts");
      if (!d->attn_k_cache[l] || !d->attn_v_cache[l]) return set_error(NT_ERR_INVALID_ARG, "attention: NULL cache");
      if (!aligned(d->attn_k_cache[l], 16) || !aligned(d->attn_v_cache[l], 16))
        return set_error(NT_ERR_ALIGNMENT, "attention: caches must be 16-byte aligned");
      if ((d->norm_attn && (!d->norm_attn[l] || !aligned(d->norm_attn[l], 16))) ||
          (d->norm_ffn && (!d->norm_ffn[l] || !aligned(d->norm_ffn[l], 16))))
        return set_error(NT_ERR_INVALID_ARG, "attention: normalisation weights NULL or not 16-byte aligned");
    }
    if (d->norm_final && !aligned(d->norm_final, 16))
      return set_error(NT_ERR_ALIGNMENT, "attention: norm_final must be 16-byte aligned");
  }
  return NT_OK;
}

__global__ void set_position_kernel(int* pos, int p, int B) {
  pos[0] = p;
  pos[1] = p + B;
}

nt_status validate_desc(const nt_decode_desc* d) {
  if (!d) return set_error(NT_ERR_INVALID_ARG, "NULL descriptor");
  if (d->n_layers < 1 || !d->proj) return set_error(NT_ERR_INVALID_ARG, "need n_layers >= 1 and a projection array");
  if (d->batch < 1 || d->batch > kStepMaxBatch) return set_error(NT_ERR_INVALID_ARG, "batch must be in [1, 16]");
  if (d->mode != NT_STEP_INDEPENDENT && d->mode != NT_STEP_ORDERED && d->mode != NT_STEP_CHAINED)
    return set_error(NT_ERR_INVALID_ARG, "mode must be NT_STEP_INDEPENDENT, NT_STEP_ORDERED or NT_STEP_CHAINED");
  if (d->launcher != NT_LAUNCH_PERSISTENT && d->launcher != NT_LAUNCH_GRAPH && d->launcher != NT_LAUNCH_STREAM)
    return set_error(NT_ERR_INVALID_ARG, "unknown launcher");
  for (int i = 0; i < d->n_layers * kProjPerLayer; ++i) {
    const nt_proj& p = d->proj[i];
    if (p.N < 1 || p.K < 16 || p.K % 16 != 0)
      return set_error(NT_ERR_INVALID_ARG, "projection " + std::to_string(i) + ": need N >= 1 and K a positive multiple of 16");
    if (!p.w || !p.s_w || !p.q || !p.s_x || !p.y)
      return set_error(NT_ERR_INVALID_ARG, "projection " + std::to_string(i) + ": NULL pointer");
    if (!aligned(p.w, 16) || !aligned(p.q, 16) || !aligned(p.s_w, 4) || !aligned(p.s_x, 4) ||
        !aligned(p.y, 4) || (p.x && !aligned(p.x, 4)))
      return set_error(NT_ERR_ALIGNMENT, "projection " + std::to_string(i) + ": misaligned pointer");
  }
  if (d->head_T) {
    if (d->head_V < 1 || d->head_K < 16 || d->head_K % 16 != 0)
      return set_error(NT_ERR_INVALID_ARG, "head: need V >= 1 and K a positive multiple of 16");
    if (!d->head_s || !d->head_q || !d->head_sx || !d->head_argmax)
      return set_error(NT_ERR_INVALID_ARG, "head: NULL pointer");
    if (!aligned(d->head_T, 16) || !aligned(d->head_q, 16) || (d->head_x && !aligned(d->head_x, 4)))
      return set_error(NT_ERR_ALIGNMENT, "head: misaligned pointer");
  }
  if (d->embed_T) {
    if (d->embed_V < 1 || d->embed_K < 16 || d->embed_K % 16 != 0)
      return set_error(NT_ERR_INVALID_ARG, "embed: need V >= 1 and K a positive multiple of 16");
    if (!d->embed_s || !d->tokens || !d->embed_x) return set_error(NT_ERR_INVALID_ARG, "embed: NULL pointer");
    if (!aligned(d->embed_T, 16) || !aligned(d->embed_x, 16) || !aligned(d->tokens, 4) || !aligned(d->embed_s, 4))
      return set_error(NT_ERR_ALIGNMENT, "embed: misaligned pointer");
  }
  if (d->verify_emit) {
    if (!d->head_T) return set_error(NT_ERR_INVALID_ARG, "verify: needs the output projection (head_T)");
    if (!d->verify_n || (d->batch > 1 && !d->verify_draft))
      return set_error(NT_ERR_INVALID_ARG, "verify: NULL pointer");
  }
  if (d->mode == NT_STEP_CHAINED) return validate_chain(d);
  return NT_OK;
}

// Issues the per-stage launches of one step on `st` (stream and graph launchers). Every launch
// but the output projection's is a programmatic dependent launch: the kernel is scheduled while
// its predecessor finishes and waits for it before its first memory access.
nt_status issue_launches(nt_decode_plan* p, cudaStream_t st) {
  constexpr bool pdl = true;
  if (p->embed_T)
    NT_TRY(launch_embed(p->embed_T, p->embed_s, p->embed_V, p->embed_K, p->tokens, p->B, p->embed_x, nullptr, st,
                        pdl));
  if (p->n_qjobs) NT_TRY(launch_quantize_jobs(p->d_qjobs, p->n_qjobs, p->B, st, pdl));
  const bool chained = p->mode == NT_STEP_CHAINED;
  for (size_t i = 0; i < p->stages.size(); ++i) {
    const PlanStage& s = p->stages[i];
    if (p->attn && i % 4 == 1) {  // after q, k, v: rotate, append, attend
      const int l = (int)(i / 4);
      const MatDesc* m = p->mats.data() + l * kProjPerLayer;
      NT_TRY(launch_rope_append(m[0].y, m[1].y, m[2].y, p->B, p->Hq, p->Hkv, 0, p->rope_base, p->d_qrot,
                                p->k_cache[l], p->v_cache[l], p->t_stride, st, p->d_pos, pdl));
      NT_TRY(launch_attention(p->d_qrot, p->k_cache[l], p->v_cache[l], p->B, p->Hq, p->Hkv, p->t_stride, p->t_stride,
                              p->d_attn_out, p->d_attn_ws, st, p->d_pos + 1, pdl));
    }
    if (chained) NT_TRY(launch_chain_quant(p->d_cjobs + i, p->B, st, pdl));
    if (p->tc8.n)
      NT_TRY(tc8_plan_launch(p->tc8, st, pdl));
    else if (p->d_mma)
      NT_TRY(launch_gemv_mma(p->d_mma + s.first_mat, s.n_mats, p->d_mma_tab + s.mma_tab_off, s.mma_ctas, p->B, st,
                             pdl));
    else
      NT_TRY(launch_gemv_tiled_group(p->d_mats + s.first_mat, p->d_prefix + s.prefix_off, s.n_mats,
                                     s.total_tiles, p->B, st, pdl));
  }
  if (p->has_head && chained) NT_TRY(launch_chain_quant(p->d_cjobs + p->stages.size(), p->B, st, pdl));
  if (p->has_head)
    NT_TRY(launch_head(p->head_T, p->head_s, p->head_V, p->head_K, p->head_q, p->head_sx, p->B,
                       p->head_logits, p->head_argmax, p->d_head_ws, st));
  if (p->verify_emit)
    NT_TRY(launch_verify(p->verify_draft, p->head_argmax, p->B, p->verify_emit, p->verify_n, st, pdl));
  return NT_OK;
}

// Quantization jobs of the persistent launcher: CTA c runs entries c, c + grid, c + 2 grid, ...
// before the step's first grid barrier, so that phase ends with its most loaded CTA. Each
// vector becomes a job of its own, the jobs go largest first to the least loaded CTA, and
// empty jobs (B = 0) fill the rounds a CTA has no work in; no CTA then holds more than one
// 12,288-wide vector, or two 4,096-wide ones, of the 8B-shaped batch-1 step.
std::vector<QuantJob> place_quant_jobs(const std::vector<QuantJob>& jobs, int grid) {
  std::vector<QuantJob> one;
  for (const QuantJob& j : jobs)
    for (int b = 0; b < j.B; ++b) one.push_back(QuantJob{j.x + (int64_t)b * j.K, j.q + (int64_t)b * j.K, j.s + b, j.K, 1});
  std::stable_sort(one.begin(), one.end(), [](const QuantJob& a, const QuantJob& b) { return a.K > b.K; });
  std::vector<std::vector<QuantJob>> per(grid);
  std::vector<int64_t> load(grid, 0);
  for (const QuantJob& j : one) {
    const int c = (int)(std::min_element(load.begin(), load.end()) - load.begin());
    per[c].push_back(j);
    load[c] += j.K + 1024;  // + the two consumer barriers and the scale, as elements
  }
  size_t rounds = 0;
  for (const auto& v : per) rounds = std::max(rounds, v.size());
  std::vector<QuantJob> out(rounds * grid, QuantJob{nullptr, nullptr, nullptr, 0, 0});
  for (int c = 0; c < grid; ++c)
    for (size_t r = 0; r < per[c].size(); ++r) out[r * grid + c] = per[c][r];
  return out;
}

void free_plan(nt_decode_plan* p) {
  if (!p) return;
  if (p->exec) cudaGraphExecDestroy(p->exec);
  if (p->graph) cudaGraphDestroy(p->graph);
  cudaFree(p->d_mats);
  cudaFree(p->d_prefix);
  cudaFree(p->d_mma);
  cudaFree(p->d_mma_ws);
  cudaFree(p->d_mma_tab);
  tc8_plan_destroy(&p->tc8);
  cudaFree(p->d_qjobs);
  cudaFree(p->d_head_ws);
  cudaFree(p->d_ctrl);
  cudaFree(p->d_sched);
  cudaFree(p->d_resid);
  cudaFree(p->d_chain_tmp);
  cudaFree(p->d_cjobs);
  cudaFree(p->d_pos);
  cudaFree(p->d_qrot);
  cudaFree(p->d_attn_out);
  cudaFree(p->d_attn_ws);
  delete p;
}

}  // namespace

extern "C" {

nt_status nt_decode_plan_create(const nt_decode_desc* d, nt_decode_plan** out) {
  clear_error();
  if (!out) return set_error(NT_ERR_INVALID_ARG, "NULL plan pointer");
  *out = nullptr;
  NT_TRY(validate_desc(d));
  int sms = 0;
  NT_TRY(check_device(&sms));
  nt_decode_plan* p = new nt_decode_plan();
  p->sm_count = sms;
  cudaGetDevice(&p->device);
  p->n_layers = d->n_layers;
  p->B = d->batch;
  p->mode = d->mode;
  p->launcher = d->launcher;
  p->timeout_ns = (uint64_t)((d->timeout_ms > 0 ? d->timeout_ms : 250.0) * 1e6);
  p->test_fault = d->test_fault;

  // Matrices in step order, and the stages that group them.
  const int n_proj = d->n_layers * kProjPerLayer;
  std::vector<MatDesc> mats(n_proj);
  std::vector<QuantJob> jobs;
  for (int i = 0; i < n_proj; ++i) {
    const nt_proj& pr = d->proj[i];
    MatDesc& m = mats[i];
    m.w = static_cast<const uint8_t*>(pr.w);
    m.s_w = pr.s_w;
    m.q = pr.q;
    m.s_x = pr.s_x;
    m.y = pr.y;
    m.acc = nullptr;
    m.N = pr.N;
    m.K = pr.K;
    m.B = d->batch;
    if (pr.x && d->mode != NT_STEP_CHAINED) jobs.push_back(QuantJob{pr.x, pr.q, pr.s_x, pr.K, d->batch});
  }
  p->mats = mats;
  std::vector<int64_t> prefix;
  auto add_stage = [&](int first, int n) {
    PlanStage s{first, n, (int64_t)prefix.size(), 0};
    int64_t acc = 0;
    for (int i = 0; i < n; ++i) {
      prefix.push_back(acc);
      acc += padded_rows(mats[first + i].N) / 4;
    }
    prefix.push_back(acc);
    s.total_tiles = acc;
    p->stages.push_back(s);
  };
  if (d->mode == NT_STEP_INDEPENDENT) {
    add_stage(0, n_proj);
  } else {
    for (int l = 0; l < d->n_layers; ++l) {
      const int b = l * kProjPerLayer;
      add_stage(b + 0, 3);  // q, k, v
      add_stage(b + 3, 1);  // o
      add_stage(b + 4, 2);  // gate, up
      add_stage(b + 6, 1);  // down
    }
  }

  p->has_head = d->head_T != nullptr;
  if (p->has_head) {
    p->head_T = d->head_T;
    p->head_s = d->head_s;
    p->head_V = d->head_V;
    p->head_K = d->head_K;
    p->head_q = d->head_q;
    p->head_sx = d->head_sx;
    p->head_logits = d->head_logits;
    p->head_argmax = d->head_argmax;
    if (d->head_x && d->mode != NT_STEP_CHAINED)
      jobs.push_back(QuantJob{d->head_x, d->head_q, d->head_sx, d->head_K, d->batch});
  }
  p->n_qjobs = (int)jobs.size();
  p->embed_T = d->embed_T;
  p->embed_s = d->embed_s;
  p->embed_V = d->embed_V;
  p->embed_K = d->embed_K;
  p->tokens = d->tokens;
  p->embed_x = d->embed_x;
  p->verify_draft = d->verify_draft;
  p->verify_emit = d->verify_emit;
  p->verify_n = d->verify_n;

  auto fail = [&](nt_status s) { free_plan(p); return s; };
  auto cuda_fail = [&](cudaError_t e, const char* what) {
    set_error(NT_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
    free_plan(p);
    return NT_ERR_CUDA;
  };
  cudaError_t e;
  std::vector<ChainJob> cjobs;
  if (d->mode == NT_STEP_CHAINED) {
    // The residual stream and the stage inputs (see nt_step_mode): the persistent kernel
    // reads each stage's input from the matrices' ChainSrc and adds o / down outputs into the
    // residual stream in their epilogue; the stream / graph launchers run one ChainJob per
    // stage, which also writes the residual stream.
    const int dm = d->proj[0].K, B = d->batch;
    p->head_dim = d->head_dim > 0 ? d->head_dim : 128;
    int kmax = dm;
    for (const MatDesc& m : mats) kmax = std::max(kmax, m.K);
    if ((e = cudaMalloc(&p->d_resid, sizeof(float) * (size_t)B * dm)) != cudaSuccess) return cuda_fail(e, "cudaMalloc");
    if ((e = cudaMalloc(&p->d_chain_tmp, sizeof(float) * (size_t)B * kmax)) != cudaSuccess)
      return cuda_fail(e, "cudaMalloc");
    float* R = p->d_resid;
    const float* x0 = d->proj[0].x;
    const int hd = p->head_dim;
    auto job = [&](ChainSrc src, float* vbuf, int first, int n) {
      ChainJob j{};
      j.src = src;
      j.vbuf = vbuf;
      j.n_rec = n;
      for (int r = 0; r < n; ++r) {
        j.q[r] = const_cast<int8_t*>(mats[first + r].q);
        j.s[r] = const_cast<float*>(mats[first + r].s_x);
      }
      cjobs.push_back(j);
    };
    p->attn = d->attn_k_cache != nullptr;
    if (p->attn) {
      p->Hq = d->proj[0].N / 128;
      p->Hkv = d->proj[1].N / 128;
      p->t_stride = d->attn_t_stride;
      p->rope_base = d->rope_base > 0 ? d->rope_base : 10000.0f;
      p->k_cache.assign(d->attn_k_cache, d->attn_k_cache + d->n_layers);
      p->v_cache.assign(d->attn_v_cache, d->attn_v_cache + d->n_layers);
      p->attn_ws_bytes = attention_ws_bytes(B, p->Hq, p->Hkv, p->t_stride);
      const size_t qb = sizeof(float) * (size_t)B * p->Hq * 128;
      if ((e = cudaMalloc(&p->d_pos, 2 * sizeof(int))) != cudaSuccess) return cuda_fail(e, "cudaMalloc");
      if ((e = cudaMalloc(&p->d_qrot, qb)) != cudaSuccess) return cuda_fail(e, "cudaMalloc");
      if ((e = cudaMalloc(&p->d_attn_out, qb)) != cudaSuccess) return cuda_fail(e, "cudaMalloc");
      if ((e = cudaMalloc(&p->d_attn_ws, p->attn_ws_bytes)) != cudaSuccess) return cuda_fail(e, "cudaMalloc");
      if ((e = cudaMemset(p->d_attn_ws, 0, p->attn_ws_bytes)) != cudaSuccess) return cuda_fail(e, "cudaMemset");
      const int pos[2] = {d->attn_pos, d->attn_pos + B};
      if ((e = cudaMemcpy(p->d_pos, pos, sizeof pos, cudaMemcpyHostToDevice)) != cudaSuccess)
        return cuda_fail(e, "cudaMemcpy");
    }
    const float eps = d->norm_eps > 0 ? d->norm_eps : 1e-6f;
    auto normed = [&](ChainSrc src, const float* gamma) {
      src.gamma = gamma;
      src.eps = eps;
      return src;
    };
    for (int l = 0; l < d->n_layers; ++l) {
      const int b = l * kProjPerLayer;
      MatDesc* m = mats.data() + b;
      const float* h = l == 0 ? x0 : R;
      const int G = m[3].K / m[2].N;
      for (int i = 0; i < 3; ++i) m[i].src = ChainSrc{h, nullptr, kChainDirect, dm, 1, hd};
      m[3].src = ChainSrc{m[2].y, nullptr, kChainHeads, m[3].K, G, hd};
      m[3].res_in = h;
      m[3].res_out = R;
      for (int i = 4; i < 6; ++i) m[i].src = ChainSrc{R, nullptr, kChainDirect, dm, 1, hd};
      m[6].src = ChainSrc{m[4].y, m[5].y, kChainProduct, m[6].K, 1, hd};
      m[6].res_in = R;
      m[6].res_out = R;
      const int recf[4] = {b, b + 3, b + 4, b + 6}, recn[4] = {3, 1, 2, 1};
      for (int g = 0; g < 4; ++g)
        for (int i = 0; i < recn[g]; ++i) {
          mats[recf[g] + i].rec_first = recf[g];
          mats[recf[g] + i].rec_count = recn[g];
        }
      // stream / graph launchers: the residual additions happen in the stage-input jobs
      if (p->attn) {
        const float* ga = d->norm_attn ? d->norm_attn[l] : nullptr;
        const float* gf = d->norm_ffn ? d->norm_ffn[l] : nullptr;
        // persistent launcher: normalised inputs, the attention output for o, the SiLU gate
        for (int i = 0; i < 3; ++i) m[i].src = normed(ChainSrc{h, nullptr, kChainDirect, dm, 1, hd}, ga);
        m[3].src = ChainSrc{p->d_attn_out, nullptr, kChainDirect, m[3].K, 1, hd};
        for (int i = 4; i < 6; ++i) m[i].src = normed(ChainSrc{R, nullptr, kChainDirect, dm, 1, hd}, gf);
        m[6].src = ChainSrc{m[4].y, m[5].y, kChainSiluProduct, m[6].K, 1, hd};
        if (l == 0) job(normed(ChainSrc{x0, nullptr, kChainDirect, dm, 1, hd}, ga), R, b, 3);
        else job(normed(ChainSrc{R, mats[b - 1].y, kChainSum, dm, 1, hd}, ga), R, b, 3);
        job(ChainSrc{p->d_attn_out, nullptr, kChainDirect, m[3].K, 1, hd}, p->d_chain_tmp, b + 3, 1);
        job(normed(ChainSrc{R, m[3].y, kChainSum, dm, 1, hd}, gf), R, b + 4, 2);
        job(ChainSrc{m[4].y, m[5].y, kChainSiluProduct, m[6].K, 1, hd}, p->d_chain_tmp, b + 6, 1);
        continue;
      }
      if (l == 0) job(ChainSrc{x0, nullptr, kChainDirect, dm, 1, hd}, p->d_chain_tmp, b, 3);
      else job(ChainSrc{R, mats[b - 1].y, kChainSum, dm, 1, hd}, R, b, 3);
      job(m[3].src, p->d_chain_tmp, b + 3, 1);
      job(ChainSrc{h, m[3].y, kChainSum, dm, 1, hd}, R, b + 4, 2);
      job(m[6].src, p->d_chain_tmp, b + 6, 1);
    }
    p->head_src = ChainSrc{R, nullptr, kChainDirect, dm, 1, hd};
    if (p->attn) p->head_src = normed(p->head_src, d->norm_final);
    if (p->has_head) {
      ChainJob j{};
      j.src = ChainSrc{R, mats[n_proj - 1].y, kChainSum, dm, 1, hd};
      if (p->attn) j.src = normed(j.src, d->norm_final);
      j.vbuf = R;
      j.n_rec = 1;
      j.q[0] = const_cast<int8_t*>(p->head_q);
      j.s[0] = const_cast<float*>(p->head_sx);
      cjobs.push_back(j);
    }
    p->mats = mats;
    p->n_cjobs = (int)cjobs.size();
    p->cjobs = cjobs;
    if ((e = cudaMalloc(&p->d_cjobs, sizeof(ChainJob) * cjobs.size())) != cudaSuccess) return cuda_fail(e, "cudaMalloc");
    if ((e = cudaMemcpy(p->d_cjobs, cjobs.data(), sizeof(ChainJob) * cjobs.size(), cudaMemcpyHostToDevice)) != cudaSuccess)
      return cuda_fail(e, "cudaMemcpy");
  }
  if ((e = cudaMalloc(&p->d_mats, sizeof(MatDesc) * mats.size())) != cudaSuccess) return cuda_fail(e, "cudaMalloc");
  if ((e = cudaMemcpy(p->d_mats, mats.data(), sizeof(MatDesc) * mats.size(), cudaMemcpyHostToDevice)) != cudaSuccess)
    return cuda_fail(e, "cudaMemcpy");
  if ((e = cudaMalloc(&p->d_prefix, sizeof(int64_t) * prefix.size())) != cudaSuccess) return cuda_fail(e, "cudaMalloc");
  if ((e = cudaMemcpy(p->d_prefix, prefix.data(), sizeof(int64_t) * prefix.size(), cudaMemcpyHostToDevice)) != cudaSuccess)
    return cuda_fail(e, "cudaMemcpy");
  if ((e = cudaMalloc(&p->d_ctrl, sizeof(StepCtrl))) != cudaSuccess) return cuda_fail(e, "cudaMalloc");
  if ((e = cudaMemset(p->d_ctrl, 0, sizeof(StepCtrl))) != cudaSuccess) return cuda_fail(e, "cudaMemset");
  if (p->launcher != NT_LAUNCH_PERSISTENT && p->B >= kMmaMinBatch && p->B <= kMmaMaxBatch &&
      p->mode == NT_STEP_INDEPENDENT && p->stages.size() == 1 &&
      tc8_plan_supported(mats.data(), (int)mats.size(), p->B)) {
    // one stage of matrices of >= 128 rows: tcgen05 with the decoded trits in tensor memory
    const nt_status s = tc8_plan_create(mats.data(), (int)mats.size(), p->B, &p->d_ctrl->error, p->timeout_ns,
                                        p->test_fault == 2, &p->tc8);
    if (s != NT_OK) return fail(s);
  } else if (p->launcher != NT_LAUNCH_PERSISTENT && p->B >= kMmaMinBatch && p->B <= kMmaMaxBatch) {
    // batched plans on the stream / graph launchers: the tensor-core path. Every stage's
    // matrices take disjoint parts of one workspace ([B][N] int32 sums of each matrix, then
    // the unit groups' counters); stages run one after another and leave it zero.
    std::vector<MmaMat> mm(mats.size());
    std::vector<int64_t> acc_off(mats.size()), cnt_off(mats.size());
    std::vector<uint16_t> tab;  // every stage's CTA -> matrix (index within the stage)
    size_t ws_bytes = 0;
    for (PlanStage& st : p->stages) {
      if (st.n_mats > 65535) return fail(set_error(NT_ERR_INVALID_ARG, "too many projections in one stage"));
      st.mma_tab_off = (int64_t)tab.size();
      // K parts: every matrix of the stage is cut into parts as long as the shortest K (so
      // the CTAs do equal work), then all parts are halved while the stage has fewer than 8
      // waves of CTAs; the parts meet in the workspace, unsplit matrices write y straight
      // from the sums
      std::vector<int> chunks_of;
      int64_t min_chunks = INT64_MAX;
      for (int i = st.first_mat; i < st.first_mat + st.n_mats; ++i) {
        MmaMat g{};
        g.N = mats[i].N;
        g.K = mats[i].K;
        mma_geometry(g, 1);
        chunks_of.push_back(g.kchunks);
        min_chunks = std::min<int64_t>(min_chunks, g.kchunks);
      }
      auto stage_ctas = [&](int64_t mult) {
        int64_t n = 0;
        for (int i = st.first_mat; i < st.first_mat + st.n_mats; ++i) {
          MmaMat g{};
          g.N = mats[i].N;
          g.K = mats[i].K;
          const int64_t c = chunks_of[i - st.first_mat];
          mma_geometry(g, (int)(mult * ((c + min_chunks - 1) / min_chunks)));
          n += mma_ctas(g);
        }
        return n;
      };
      int64_t mult = 1;
      while (mult < min_chunks && stage_ctas(mult) < 8LL * device_sm_count()) mult *= 2;
      int64_t ctas = 0, rows = 0, units = 0;
      for (int i = st.first_mat; i < st.first_mat + st.n_mats; ++i) {
        const MatDesc& d = mats[i];
        MmaMat& x = mm[i];
        x = MmaMat{};
        x.w = d.w;
        x.s_w = d.s_w;
        x.q = d.q;
        x.s_x = d.s_x;
        x.y = d.y;
        x.acc = d.acc;
        x.N = d.N;
        x.K = d.K;
        x.B = d.B;
        const int64_t c = chunks_of[i - st.first_mat];
        mma_geometry(x, (int)(mult * ((c + min_chunks - 1) / min_chunks)));
        x.cta_begin = ctas;
        ctas += mma_ctas(x);
        tab.insert(tab.end(), (size_t)mma_ctas(x), (uint16_t)(i - st.first_mat));
        acc_off[i] = rows * d.B;
        rows += d.N;
        cnt_off[i] = units;
        units += x.ugroups;
      }
      for (int i = st.first_mat; i < st.first_mat + st.n_mats; ++i) cnt_off[i] += rows * p->B;  // in 4-byte words
      st.mma_ctas = ctas;
      ws_bytes = std::max(ws_bytes, mma_ws_bytes(rows, units, p->B));
    }
    if ((e = cudaMalloc(&p->d_mma_ws, ws_bytes)) != cudaSuccess) return cuda_fail(e, "cudaMalloc");
    if ((e = cudaMemset(p->d_mma_ws, 0, ws_bytes)) != cudaSuccess) return cuda_fail(e, "cudaMemset");
    for (size_t i = 0; i < mm.size(); ++i) {
      mm[i].acc_ws = static_cast<int32_t*>(p->d_mma_ws) + acc_off[i];
      mm[i].cnt = static_cast<unsigned int*>(p->d_mma_ws) + cnt_off[i];
    }
    if ((e = cudaMalloc(&p->d_mma_tab, sizeof(uint16_t) * tab.size())) != cudaSuccess) return cuda_fail(e, "cudaMalloc");
    if ((e = cudaMemcpy(p->d_mma_tab, tab.data(), sizeof(uint16_t) * tab.size(), cudaMemcpyHostToDevice)) != cudaSuccess)
      return cuda_fail(e, "cudaMemcpy");
    if ((e = cudaMalloc(&p->d_mma, sizeof(MmaMat) * mm.size())) != cudaSuccess) return cuda_fail(e, "cudaMalloc");
    if ((e = cudaMemcpy(p->d_mma, mm.data(), sizeof(MmaMat) * mm.size(), cudaMemcpyHostToDevice)) != cudaSuccess)
      return cuda_fail(e, "cudaMemcpy");
  }
  if (!jobs.empty() && p->launcher == NT_LAUNCH_PERSISTENT) {
    jobs = place_quant_jobs(jobs, p->sm_count);
    p->n_qjobs = (int)jobs.size();
  }
  if (!jobs.empty()) {
    if ((e = cudaMalloc(&p->d_qjobs, sizeof(QuantJob) * jobs.size())) != cudaSuccess) return cuda_fail(e, "cudaMalloc");
    if ((e = cudaMemcpy(p->d_qjobs, jobs.data(), sizeof(QuantJob) * jobs.size(), cudaMemcpyHostToDevice)) != cudaSuccess)
      return cuda_fail(e, "cudaMemcpy");
  }
  if (p->has_head) {
    const size_t ws = head_ws_bytes(p->B);
    if ((e = cudaMalloc(&p->d_head_ws, ws)) != cudaSuccess) return cuda_fail(e, "cudaMalloc");
    if ((e = cudaMemset(p->d_head_ws, 0, ws)) != cudaSuccess) return cuda_fail(e, "cudaMemset");
  }

  if (p->launcher == NT_LAUNCH_PERSISTENT) {
    const nt_status s = persist_prepare(p);
    if (s != NT_OK) return fail(s);
  } else if (p->launcher == NT_LAUNCH_GRAPH) {
    cudaStream_t cs;
    if ((e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking)) != cudaSuccess) return cuda_fail(e, "cudaStreamCreate");
    e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) { cudaStreamDestroy(cs); return cuda_fail(e, "cudaStreamBeginCapture"); }
    const nt_status s = issue_launches(p, cs);
    cudaGraph_t g = nullptr;
    e = cudaStreamEndCapture(cs, &g);
    cudaStreamDestroy(cs);
    p->graph = g;
    if (s != NT_OK) return fail(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamEndCapture");
    if ((e = cudaGraphInstantiate(&p->exec, p->graph, 0)) != cudaSuccess) return cuda_fail(e, "cudaGraphInstantiate");
  }
  if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  *out = p;
  return NT_OK;
}

nt_status nt_decode_step(nt_decode_plan* p, void* stream) {
  clear_error();
  if (!p) return set_error(NT_ERR_INVALID_ARG, "NULL plan");
  const cudaStream_t st = as_stream(stream);
  switch (p->launcher) {
    case NT_LAUNCH_GRAPH:
      NT_CUDA_TRY(cudaGraphLaunch(p->exec, st));
      return NT_OK;
    case NT_LAUNCH_STREAM:
      return issue_launches(p, st);
    default:
      if (!p->seg_barriers.empty()) {
        // a segmented step counts its grid barriers on the host across its launches, so a
        // recorded copy of it would replay stale counts: refuse to be recorded
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        NT_CUDA_TRY(cudaStreamIsCapturing(st, &cs));
        if (cs != cudaStreamCaptureStatusNone)
          return set_error(NT_ERR_UNSUPPORTED, "a chained step with attention cannot be recorded into a CUDA graph");
      }
      return persist_launch(p, st);
  }
}

nt_status nt_decode_plan_set_position(nt_decode_plan* p, int pos, void* stream) {
  clear_error();
  if (!p) return set_error(NT_ERR_INVALID_ARG, "NULL plan");
  if (!p->attn) return set_error(NT_ERR_INVALID_ARG, "the plan has no attention side");
  if (pos < 0 || (int64_t)pos + p->B > p->t_stride) return set_error(NT_ERR_INVALID_ARG, "need 0 <= pos and pos + batch <= attn_t_stride");
  set_position_kernel<<<1, 1, 0, as_stream(stream)>>>(p->d_pos, pos, p->B);
  return check_launch("set_position_kernel");
}

nt_status nt_decode_step_status(nt_decode_plan* p, nt_status* device_status) {
  clear_error();
  if (!p || !device_status) return set_error(NT_ERR_INVALID_ARG, "NULL argument");
  StepCtrl c;
  NT_CUDA_TRY(cudaMemcpy(&c, p->d_ctrl, sizeof c, cudaMemcpyDeviceToHost));
  *device_status = c.error ? NT_ERR_TIMEOUT : NT_OK;
  if (c.error) {
    char buf[160];
    snprintf(buf, sizeof buf, "decode step: a bounded wait ran out (code %u, CTA %u)", c.error, c.error_cta);
    set_error(NT_ERR_TIMEOUT, buf);
  }
  return NT_OK;
}

nt_status nt_decode_plan_reset(nt_decode_plan* p) {
  clear_error();
  if (!p) return set_error(NT_ERR_INVALID_ARG, "NULL plan");
  NT_CUDA_TRY(cudaDeviceSynchronize());
  NT_CUDA_TRY(cudaMemset(p->d_ctrl, 0, sizeof(StepCtrl)));
  if (p->d_head_ws) NT_CUDA_TRY(cudaMemset(p->d_head_ws, 0, head_ws_bytes(p->B)));
  if (p->tc8.d_buf) NT_CUDA_TRY(cudaMemset(p->tc8.d_buf, 0, p->tc8.buf_bytes));  // partial sums a timeout left
  p->launches = 0;
  p->barrier_count = 0;
  NT_CUDA_TRY(cudaDeviceSynchronize());
  return NT_OK;
}

nt_status nt_decode_plan_trace_layout(const nt_decode_plan* p, int* grid, int* barriers) {
  clear_error();
  if (!p || !grid || !barriers) return set_error(NT_ERR_INVALID_ARG, "NULL argument");
  *grid = p->launcher == NT_LAUNCH_PERSISTENT ? p->grid : 0;
  *barriers = p->launcher == NT_LAUNCH_PERSISTENT ? p->n_barriers : 0;
  return NT_OK;
}

nt_status nt_decode_plan_set_trace(nt_decode_plan* p, unsigned long long* trace) {
  clear_error();
  if (!p) return set_error(NT_ERR_INVALID_ARG, "NULL plan");
  if (trace && !aligned(trace, 8)) return set_error(NT_ERR_ALIGNMENT, "trace must be 8-byte aligned");
  p->trace = trace;
  return NT_OK;
}

nt_status nt_decode_plan_capture_size(const nt_decode_plan* p, size_t* floats) {
  clear_error();
  if (!p || !floats) return set_error(NT_ERR_INVALID_ARG, "NULL argument");
  if (p->mode != NT_STEP_CHAINED) return set_error(NT_ERR_INVALID_ARG, "capture needs a chained plan");
  size_t n = 0;
  for (const PlanStage& s : p->stages) n += (size_t)p->B * p->mats[s.first_mat].K;
  if (p->has_head) n += (size_t)p->B * p->head_K;
  *floats = n;
  return NT_OK;
}

nt_status nt_decode_plan_set_capture(nt_decode_plan* p, float* buf) {
  clear_error();
  if (!p) return set_error(NT_ERR_INVALID_ARG, "NULL plan");
  if (p->mode != NT_STEP_CHAINED) return set_error(NT_ERR_INVALID_ARG, "capture needs a chained plan");
  if (buf && !aligned(buf, 16)) return set_error(NT_ERR_ALIGNMENT, "capture buffer must be 16-byte aligned");
  // every stage's slice starts at B times the K of the stages before it (K % 16 == 0, so each
  // slice stays 16-byte aligned)
  size_t off = 0;
  for (size_t i = 0; i < p->stages.size(); ++i) {
    const PlanStage& s = p->stages[i];
    float* cap = buf ? buf + off : nullptr;
    for (int m = s.first_mat; m < s.first_mat + s.n_mats; ++m) p->mats[m].src.cap = cap;
    p->cjobs[i].src.cap = cap;
    off += (size_t)p->B * p->mats[s.first_mat].K;
  }
  p->head_src.cap = buf && p->has_head ? buf + off : nullptr;
  if (p->has_head) p->cjobs[p->stages.size()].src.cap = p->head_src.cap;
  NT_CUDA_TRY(cudaDeviceSynchronize());  // no step of this plan may be reading the descriptors
  NT_CUDA_TRY(cudaMemcpy(p->d_mats, p->mats.data(), sizeof(MatDesc) * p->mats.size(), cudaMemcpyHostToDevice));
  NT_CUDA_TRY(cudaMemcpy(p->d_cjobs, p->cjobs.data(), sizeof(ChainJob) * p->cjobs.size(), cudaMemcpyHostToDevice));
  return NT_OK;
}

void nt_decode_plan_destroy(nt_decode_plan* p) {
  if (!p) return;
  cudaDeviceSynchronize();
  free_plan(p);
}

}  // extern "C"
