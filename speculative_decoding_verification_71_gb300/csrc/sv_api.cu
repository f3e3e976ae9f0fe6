// C ABI of the verification library (declared in include/specverify.h).
//
// Host side only: argument checks, the context and its workspace, the
// launch configuration.  Every step of the verification itself runs in the
// kernels of sv_kernels.cu.

#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>

#include "../../include/specverify.h"
#include "sv_internal.h"

struct sv_ctx {
  int max_B = 0, max_k = 0, V = 0;
  sv_dtype dtype = SV_BF16;
  int elt = 2;
  int device = 0;
  int stages = 3;
  int ctas_per_sm = 0;
  int cluster = 0;             // 0: chosen per call
  int early_exit = 0;          // 1: rows after a decided rejection are not read
  int diagnostics = 0;         // 1: calls write the per-row diagnostics spec_verify_debug reads
  int max_clusters[4] = {0};   // clusters of 1, 2, 4, 8 CTAs that fit at once
  int num_sms = 0;
  int smem_bytes = 0;
  long long wait_limit_ns = sv::kDrainLimitNs;
  void* ws_mem = nullptr;
  sv::Workspace ws{};
  void* pw_mem = nullptr;      // workspace of the pieces kernel (null: not available)
  sv::PiecesWs pw{};
  int kernel = SV_KERNEL_AUTO;
  unsigned long long* timeline = nullptr;   // caller's buffer of per-CTA timestamps (or null)
  int timeline_cap = 0;
  int pieces_ctas = 0;         // grid of the pieces kernel (one CTA per SM)
  int np = 0, nr = 0;
  long long calls = 0;
  int last_B = 0, last_k = 0, last_greedy = 0, last_diag = 0;
  float last_inv_T = 1.f;
  char cuda_msg[256] = {0};
};

namespace {

thread_local char g_create_msg[256] = {0};

sv_status cuda_fail(sv_ctx* ctx, cudaError_t e, const char* where) {
  char* dst = ctx ? ctx->cuda_msg : g_create_msg;
  std::snprintf(dst, 256, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
  return SV_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Configure the staging ring (slots of 64 KB per CTA) and how many CTAs
// share an SM (0: as many as fit); fails if the shape cannot be launched.
sv_status configure(sv_ctx* ctx, int stages, int ctas_per_sm) {
  const int smem = sv::verify_smem_bytes(stages);
  cudaDeviceProp prop;
  cudaError_t e = cudaGetDeviceProperties(&prop, ctx->device);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaGetDeviceProperties");
  if (smem > static_cast<int>(prop.sharedMemPerBlockOptin)) return SV_ERR_UNSUPPORTED;
  e = sv::prepare_verify_kernel(smem);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaFuncSetAttribute");
  int fit = 0;
  e = sv::query_ctas_per_sm(smem, &fit);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
  if (fit <= 0) return SV_ERR_UNSUPPORTED;
  if (ctas_per_sm > fit) return SV_ERR_UNSUPPORTED;
  const int per_sm = ctas_per_sm > 0 ? ctas_per_sm : fit;
  int clusters[4] = {0, 0, 0, 0};
  for (int i = 0; i < 4; ++i) {
    const int c = 1 << i;
    e = sv::query_max_clusters(c, smem, &clusters[i]);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();   // a size the device cannot place is simply not offered
      clusters[i] = 0;
    }
    const int cap = prop.multiProcessorCount * per_sm / c;
    if (clusters[i] > cap) clusters[i] = cap;
  }
  if (clusters[0] <= 0) return SV_ERR_UNSUPPORTED;
  if (ctx->cluster > 0 && clusters[__builtin_ctz(static_cast<unsigned>(ctx->cluster))] <= 0)
    return SV_ERR_UNSUPPORTED;
  ctx->stages = stages;
  ctx->ctas_per_sm = per_sm;
  ctx->num_sms = prop.multiProcessorCount;
  ctx->smem_bytes = smem;
  for (int i = 0; i < 4; ++i) ctx->max_clusters[i] = clusters[i];
  return SV_OK;
}

// Automatic choice: three 64 KB slots per CTA, one CTA per SM.
sv_status configure_auto(sv_ctx* ctx) {
  if (configure(ctx, 3, 0) == SV_OK) return SV_OK;
  return configure(ctx, 2, 0);
}

// Whether a call (rows 16-byte aligned) runs row streaming: the default
// where it qualifies, the faster schedule on every measured workload.
// Batches above kPiecesMaxB sequences run as consecutive row-streaming calls
// of at most kPiecesMaxB sequences each.
bool use_pieces(const sv_ctx* ctx) {
  if (ctx->kernel == SV_KERNEL_CLUSTER || !ctx->pw_mem || ctx->pieces_ctas <= 0) return false;
  return !ctx->early_exit && ctx->cluster == 0;
}

// The row-streaming schedule's workspace for (max_B, max_k) and rows of V
// logits: one allocation, 256-byte aligned sub-arrays.  Also the launch shape.
sv_status create_pieces(sv_ctx* ctx) {
  sv::pieces_shape(ctx->V, ctx->elt, ctx->np, ctx->nr);
  cudaDeviceProp prop;
  cudaError_t e = cudaGetDeviceProperties(&prop, ctx->device);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaGetDeviceProperties");
  if (sv::pieces_smem_bytes() > static_cast<int>(prop.sharedMemPerBlockOptin)) return SV_OK;
  if (ctx->np > sv::kMaxChunks) return SV_OK;   // rows of at most 1 MiB, as for the cluster kernel
  e = sv::prepare_pieces_kernel();
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaFuncSetAttribute(pieces)");
  // sized for one call of at most kPiecesMaxB sequences (larger batches run in chunks of that size)
  const size_t B = static_cast<size_t>(ctx->max_B < sv::kPiecesMaxB ? ctx->max_B : sv::kPiecesMaxB);
  const size_t k = static_cast<size_t>(ctx->max_k);
  const size_t rows = B * (2 * k + 1);
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off += (bytes + 255) / 256 * 256; return o; };
  const size_t o_rec = take(rows * ctx->np * 16), o_bseg = take(B * ctx->np * 16 * 8);
  const size_t o_job = take(B * 16), o_jobn = take(B * 16), o_njobs = take(4);
  const size_t o_bonus = take(B * 16), o_epoch = take(4);
  const size_t o_rmass = take(B * ctx->nr * 16 * 4), o_pmass = take(B * ctx->nr * 16 * 4);
  e = cudaMalloc(&ctx->pw_mem, off);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaMalloc(pieces workspace)");
  e = cudaMemset(ctx->pw_mem, 0, off);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaMemset(pieces workspace)");
  char* base = static_cast<char*>(ctx->pw_mem);
  sv::PiecesWs& w = ctx->pw;
  w.rec = reinterpret_cast<float4*>(base + o_rec);
  w.bseg = reinterpret_cast<float2*>(base + o_bseg);
  w.job = reinterpret_cast<int4*>(base + o_job);
  w.jobn = reinterpret_cast<float4*>(base + o_jobn);
  w.njobs = reinterpret_cast<int*>(base + o_njobs);
  w.bonus = reinterpret_cast<float4*>(base + o_bonus);
  w.epoch = reinterpret_cast<int*>(base + o_epoch);
  w.rmass = reinterpret_cast<float*>(base + o_rmass);
  w.pmass = reinterpret_cast<float*>(base + o_pmass);
  ctx->pieces_ctas = prop.multiProcessorCount;   // one CTA per SM (the shared memory allows no more)
  return SV_OK;
}

// Cluster size and grid of a call with batch B.
void launch_shape(const sv_ctx* ctx, int B, int* cluster, int* ctas) {
  int cs = ctx->cluster;
  if (cs == 0)
    cs = sv::auto_cluster(B, static_cast<long long>(ctx->V) * ctx->elt, ctx->num_sms, ctx->max_clusters);
  const int fit = ctx->max_clusters[__builtin_ctz(static_cast<unsigned>(cs))];
  const int clusters = B < fit ? B : fit;
  *cluster = cs;
  *ctas = clusters * cs;
}

}  // namespace

extern "C" {

const char* sv_status_string(sv_status s) {
  switch (s) {
    case SV_OK: return "SV_OK";
    case SV_ERR_INVALID_ARG: return "SV_ERR_INVALID_ARG";
    case SV_ERR_BAD_DRAFT_LEN: return "SV_ERR_BAD_DRAFT_LEN";
    case SV_ERR_BAD_TOKEN: return "SV_ERR_BAD_TOKEN";
    case SV_ERR_NONFINITE: return "SV_ERR_NONFINITE";
    case SV_ERR_TIMEOUT: return "SV_ERR_TIMEOUT";
    case SV_ERR_CUDA: return "SV_ERR_CUDA";
    case SV_ERR_UNSUPPORTED: return "SV_ERR_UNSUPPORTED";
  }
  return "SV_ERR_UNKNOWN";
}

const char* sv_last_cuda_error(const sv_ctx* ctx) { return ctx ? ctx->cuda_msg : g_create_msg; }

sv_status sv_create(sv_ctx** out, int max_B, int max_k, int V, sv_dtype dtype) {
  if (!out) return SV_ERR_INVALID_ARG;
  *out = nullptr;
  if (max_B <= 0 || max_k < 0 || V <= 0) return SV_ERR_INVALID_ARG;
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  // per-call index arithmetic is 32-bit in cluster ids and 64-bit in bytes
  if (static_cast<long long>(max_B) * (max_k + 1) > (1LL << 26)) return SV_ERR_INVALID_ARG;
  if (max_k > 31) return SV_ERR_INVALID_ARG;              // one warp lane per position
  const long long row_bytes = static_cast<long long>(V) * (dtype == SV_F32 ? 4 : 2);
  if (row_bytes > static_cast<long long>(sv::kMaxChunks) * sv::kChunkBytes) return SV_ERR_INVALID_ARG;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "cudaGetDevice");
  cudaDeviceProp prop;
  e = cudaGetDeviceProperties(&prop, dev);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "cudaGetDeviceProperties");
  if (!(prop.major == 10 && prop.minor == 3)) {
    std::snprintf(g_create_msg, sizeof g_create_msg,
                  "built for sm_103a; device is sm_%d%d", prop.major, prop.minor);
    return SV_ERR_UNSUPPORTED;
  }

  sv_ctx* ctx = new (std::nothrow) sv_ctx();
  if (!ctx) return SV_ERR_CUDA;
  ctx->max_B = max_B;
  ctx->max_k = max_k;
  ctx->V = V;
  ctx->dtype = dtype;
  ctx->elt = dtype == SV_F32 ? 4 : 2;
  ctx->device = dev;

  // one allocation, 256-byte aligned sub-arrays
  const size_t nB = static_cast<size_t>(max_B);
  const size_t nT = nB * (max_k + 1);
  const size_t nD = nB * (max_k > 0 ? max_k : 1);
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off += (bytes + 255) / 256 * 256; return o; };
  const size_t o_seqs = take(nB * 8), o_nseqs = take(4), o_ticket = take(4);
  const size_t o_mt = take(nT * 4), o_Lt = take(nT * 4);
  const size_t o_md = take(nD * 4), o_Ld = take(nD * 4), o_al = take(nD * 4), o_mass = take(nT * 4);
  const size_t o_stats = take(sv::kStatCount * 8), o_word = take(4);
  e = cudaMalloc(&ctx->ws_mem, off);
  if (e != cudaSuccess) {
    sv_status s = cuda_fail(nullptr, e, "cudaMalloc(workspace)");
    delete ctx;
    return s;
  }
  char* base = static_cast<char*>(ctx->ws_mem);
  sv::Workspace& ws = ctx->ws;
  ws.seqs = reinterpret_cast<int2*>(base + o_seqs);
  ws.n_seqs = reinterpret_cast<int*>(base + o_nseqs);
  ws.ticket = reinterpret_cast<int*>(base + o_ticket);
  ws.m_t = reinterpret_cast<float*>(base + o_mt);
  ws.L_t = reinterpret_cast<float*>(base + o_Lt);
  ws.m_d = reinterpret_cast<float*>(base + o_md);
  ws.L_d = reinterpret_cast<float*>(base + o_Ld);
  ws.alpha = reinterpret_cast<float*>(base + o_al);
  ws.mass = reinterpret_cast<float*>(base + o_mass);
  ws.stats = reinterpret_cast<unsigned long long*>(base + o_stats);
  ws.err_word = reinterpret_cast<unsigned int*>(base + o_word);

  e = cudaMemset(ctx->ws_mem, 0, off);
  if (e == cudaSuccess) e = sv::launch_init_workspace(ws, nullptr);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    sv_status s = cuda_fail(nullptr, e, "workspace init");
    cudaFree(ctx->ws_mem);
    delete ctx;
    return s;
  }
  sv_status s = configure_auto(ctx);
  if (s != SV_OK) {
    std::snprintf(g_create_msg, sizeof g_create_msg, "no launchable shape for V=%d", V);
    cudaFree(ctx->ws_mem);
    delete ctx;
    return s;
  }
  s = create_pieces(ctx);
  if (s != SV_OK) {
    std::snprintf(g_create_msg, sizeof g_create_msg, "%s", ctx->cuda_msg);
    cudaFree(ctx->ws_mem);
    if (ctx->pw_mem) cudaFree(ctx->pw_mem);
    delete ctx;
    return s;
  }
  *out = ctx;
  return SV_OK;
}

sv_status sv_destroy(sv_ctx* ctx) {
  if (!ctx) return SV_OK;
  cudaError_t e = cudaFree(ctx->ws_mem);
  if (ctx->pw_mem) {
    const cudaError_t e2 = cudaFree(ctx->pw_mem);
    if (e == cudaSuccess) e = e2;
  }
  delete ctx;
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

sv_status spec_verify(sv_ctx* ctx, int B, int k, const void* target_logits, const void* draft_logits,
                      const int32_t* draft_tokens, const int32_t* draft_len, const float* uniforms,
                      float temperature, int32_t* out_tokens, int32_t* out_len, sv_stream_t stream) {
  if (!ctx) return SV_ERR_INVALID_ARG;
  if (B < 1 || B > ctx->max_B || k < 0 || k > ctx->max_k) return SV_ERR_INVALID_ARG;
  if (!(temperature >= 0.f) || !std::isfinite(temperature)) return SV_ERR_INVALID_ARG;
  const bool greedy = temperature == 0.f;
  const double c2 = greedy ? 0.0 : 1.4426950408889634 / static_cast<double>(temperature);
  if (!greedy && !(c2 < 1e30)) return SV_ERR_INVALID_ARG;
  if (!target_logits || !draft_len || !out_tokens || !out_len) return SV_ERR_INVALID_ARG;
  if (k > 0 && !draft_tokens) return SV_ERR_INVALID_ARG;
  if (k > 0 && !greedy && !draft_logits) return SV_ERR_INVALID_ARG;
  if (!greedy && !uniforms) return SV_ERR_INVALID_ARG;

  sv::VerifyParams p{};
  p.target = target_logits;
  p.draft = draft_logits;
  p.tokens = draft_tokens;
  p.draft_len = draft_len;
  p.uniforms = uniforms;
  p.out_tokens = out_tokens;
  p.out_len = out_len;
  p.B = B;
  p.k = k;
  p.V = ctx->V;
  p.elt = ctx->elt;
  p.greedy = greedy ? 1 : 0;
  p.c2 = static_cast<float>(c2);
  p.stages = ctx->stages;
  p.bulk = ((static_cast<long long>(ctx->V) * ctx->elt) % 16 == 0) && aligned16(target_logits) &&
           (draft_logits == nullptr || aligned16(draft_logits));
  p.wait_limit_ns = ctx->wait_limit_ns;
  p.ws = ctx->ws;
  p.early_exit = ctx->early_exit;
  p.diag = ctx->diagnostics;
  // persistent grid: every cluster that fits at once, but never more than sequences
  int ctas = 0;
  launch_shape(ctx, B, &p.cluster, &ctas);
  p.ctas = ctas;
  if (p.bulk && use_pieces(ctx)) {
    p.pieces = 1;
    p.np = ctx->np; p.nr = ctx->nr;
    p.ctas = ctx->pieces_ctas;
    p.pw = ctx->pw;
  }
  // the timeline covers the cluster kernel's grid (and the work-list kernel)
  if (!p.pieces && ctx->timeline && (ctas + 1) * sv::kTimelineSlots <= ctx->timeline_cap) p.timeline = ctx->timeline;
  cudaError_t e = cudaSuccess;
  if (!p.pieces || B <= sv::kPiecesMaxB) {
    e = sv::launch_verify(p, ctas, ctx->smem_bytes, reinterpret_cast<cudaStream_t>(stream));
  } else {
    // row streaming, kPiecesMaxB sequences at a time: every per-sequence
    // array (inputs, outputs, diagnostics) offset to the chunk's first
    // sequence; the chunks are consecutive calls on the stream
    const size_t rb = static_cast<size_t>(ctx->V) * ctx->elt;
    const size_t k1 = static_cast<size_t>(k) + 1, kk = static_cast<size_t>(k);
    for (int b0 = 0; b0 < B && e == cudaSuccess; b0 += sv::kPiecesMaxB) {
      const size_t o = static_cast<size_t>(b0);
      sv::VerifyParams q = p;
      q.B = std::min(sv::kPiecesMaxB, B - b0);
      q.target = static_cast<const char*>(p.target) + o * k1 * rb;
      q.draft = p.draft ? static_cast<const char*>(p.draft) + o * kk * rb : nullptr;
      q.tokens = p.tokens ? p.tokens + o * kk : nullptr;
      q.draft_len = p.draft_len + o;
      q.uniforms = p.uniforms ? p.uniforms + o * k1 : nullptr;
      q.out_tokens = p.out_tokens + o * k1;
      q.out_len = p.out_len + o;
      q.ws.m_t = p.ws.m_t + o * k1;
      q.ws.L_t = p.ws.L_t + o * k1;
      q.ws.mass = p.ws.mass + o * k1;
      q.ws.m_d = p.ws.m_d + o * kk;
      q.ws.L_d = p.ws.L_d + o * kk;
      q.ws.alpha = p.ws.alpha + o * kk;
      e = sv::launch_verify(q, ctas, ctx->smem_bytes, reinterpret_cast<cudaStream_t>(stream));
    }
  }
  if (e != cudaSuccess) return cuda_fail(ctx, e, "launch verify");
  ctx->calls += 1;
  ctx->last_B = B;
  ctx->last_k = k;
  ctx->last_greedy = greedy ? 1 : 0;
  ctx->last_diag = ctx->diagnostics;
  ctx->last_inv_T = greedy ? 0.f : 1.f / temperature;
  return SV_OK;
}

sv_status spec_verify_compact(sv_ctx* ctx, int B, int k, const int32_t* out_tokens, const int32_t* out_len,
                              int32_t* packed, int32_t* offsets, sv_stream_t stream) {
  if (!ctx || B < 1 || B > ctx->max_B || k < 0 || k > ctx->max_k) return SV_ERR_INVALID_ARG;
  if (!out_tokens || !out_len || !packed || !offsets) return SV_ERR_INVALID_ARG;
  cudaError_t e = sv::launch_compact(B, k, out_tokens, out_len, packed, offsets,
                                     reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SV_OK : cuda_fail(ctx, e, "launch compact");
}

sv_status spec_verify_debug(sv_ctx* ctx, int B, int k, double* lse_t, double* lse_d, double* accept_prob,
                            double* mass, sv_stream_t stream) {
  if (!ctx || ctx->calls == 0 || !ctx->last_diag) return SV_ERR_INVALID_ARG;
  if (B != ctx->last_B || k != ctx->last_k) return SV_ERR_INVALID_ARG;
  cudaError_t e = sv::launch_debug(ctx->ws, B, k, ctx->last_greedy, ctx->last_inv_T, lse_t, lse_d,
                                   accept_prob, mass, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SV_OK : cuda_fail(ctx, e, "launch debug");
}

sv_status spec_verify_stats(sv_ctx* ctx, sv_stream_t stream, sv_stats* out) {
  if (!ctx || !out) return SV_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned long long st[sv::kStatCount];
  unsigned int word = 0;
  cudaError_t e = cudaMemcpyAsync(st, ctx->ws.stats, sizeof st, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&word, ctx->ws.err_word, sizeof word, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "spec_verify_stats");
  std::memset(out, 0, sizeof *out);
  out->calls = ctx->calls;
  out->sequences = static_cast<long long>(st[sv::kStatSequences]);
  out->drafts_proposed = static_cast<long long>(st[sv::kStatProposed]);
  out->drafts_accepted = static_cast<long long>(st[sv::kStatAccepted]);
  out->emitted = static_cast<long long>(st[sv::kStatEmitted]);
  out->spec_off = static_cast<long long>(st[sv::kStatSpecOff]);
  out->zero_residual = static_cast<long long>(st[sv::kStatZeroResidual]);
  out->error_sequences = static_cast<long long>(st[sv::kStatErrorSeqs]);
  out->error_bits = word;
  out->rows_skipped = static_cast<long long>(st[sv::kStatRowsSkipped]);
  if (out->sequences > 0) {
    out->mean_emitted = static_cast<double>(out->emitted) / static_cast<double>(out->sequences);
    out->mean_accepted = static_cast<double>(out->drafts_accepted) / static_cast<double>(out->sequences);
  }
  if (out->drafts_proposed > 0)
    out->accept_rate = static_cast<double>(out->drafts_accepted) / static_cast<double>(out->drafts_proposed);
  for (int code = SV_ERR_BAD_DRAFT_LEN; code <= SV_ERR_TIMEOUT; ++code)
    if (word & (1u << code)) return static_cast<sv_status>(code);
  return SV_OK;
}

sv_status spec_verify_reset_stats(sv_ctx* ctx, sv_stream_t stream) {
  if (!ctx) return SV_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ctx->ws.stats, 0, sizeof(unsigned long long) * sv::kStatCount, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(ctx->ws.err_word, 0, sizeof(unsigned int), s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "spec_verify_reset_stats");
  ctx->calls = 0;
  return SV_OK;
}

sv_status sv_set_pipeline(sv_ctx* ctx, int stages, int ctas_per_sm) {
  if (!ctx) return SV_ERR_INVALID_ARG;
  if (stages == 0 && ctas_per_sm == 0) return configure_auto(ctx);
  if (stages < 2 || stages > sv::kMaxStages || ctas_per_sm < 0) return SV_ERR_INVALID_ARG;
  const int prev_s = ctx->stages, prev_c = ctx->ctas_per_sm;
  sv_status s = configure(ctx, stages, ctas_per_sm);
  if (s != SV_OK) configure(ctx, prev_s, prev_c);
  return s;
}

sv_status sv_set_early_exit(sv_ctx* ctx, int on) {
  if (!ctx || (on != 0 && on != 1)) return SV_ERR_INVALID_ARG;
  ctx->early_exit = on;
  return SV_OK;
}

sv_status sv_set_diagnostics(sv_ctx* ctx, int on) {
  if (!ctx || (on != 0 && on != 1)) return SV_ERR_INVALID_ARG;
  ctx->diagnostics = on;
  return SV_OK;
}

sv_status sv_set_cluster(sv_ctx* ctx, int cluster) {
  if (!ctx) return SV_ERR_INVALID_ARG;
  if (cluster != 0 && cluster != 1 && cluster != 2 && cluster != 4 && cluster != 8) return SV_ERR_INVALID_ARG;
  if (cluster > 0 && ctx->max_clusters[__builtin_ctz(static_cast<unsigned>(cluster))] <= 0)
    return SV_ERR_UNSUPPORTED;
  ctx->cluster = cluster;
  return SV_OK;
}

sv_status sv_get_config(const sv_ctx* ctx, int* stages, int* ctas_per_sm, int* threads, int* smem_bytes,
                        int* grid_ctas, int* cluster) {
  if (!ctx) return SV_ERR_INVALID_ARG;
  if (stages) *stages = ctx->stages;
  if (ctas_per_sm) *ctas_per_sm = ctx->ctas_per_sm;
  if (threads) *threads = sv::kThreads;
  if (smem_bytes) *smem_bytes = ctx->smem_bytes;
  if (grid_ctas) *grid_ctas = ctx->num_sms * ctx->ctas_per_sm;
  if (cluster) *cluster = ctx->cluster;
  return SV_OK;
}

sv_status sv_launch_shape(const sv_ctx* ctx, int B, int* cluster, int* grid_ctas) {
  if (!ctx || B < 1 || B > ctx->max_B) return SV_ERR_INVALID_ARG;
  int cs = 0, ctas = 0;
  launch_shape(ctx, B, &cs, &ctas);
  if (cluster) *cluster = cs;
  if (grid_ctas) *grid_ctas = ctas;
  return SV_OK;
}

sv_status sv_rows_shape(const sv_ctx* ctx, int* threads, int* smem_bytes, int* grid_ctas) {
  if (!ctx) return SV_ERR_INVALID_ARG;
  if (!ctx->pw_mem || ctx->pieces_ctas <= 0) return SV_ERR_UNSUPPORTED;
  if (threads) *threads = sv::pieces_threads();
  if (smem_bytes) *smem_bytes = sv::pieces_smem_bytes();
  if (grid_ctas) *grid_ctas = ctx->pieces_ctas;
  return SV_OK;
}

sv_status sv_set_timeline(sv_ctx* ctx, unsigned long long* timeline, int capacity) {
  if (!ctx || capacity < 0 || (timeline && capacity == 0)) return SV_ERR_INVALID_ARG;
  ctx->timeline = timeline;
  ctx->timeline_cap = timeline ? capacity : 0;
  return SV_OK;
}

sv_status sv_set_kernel(sv_ctx* ctx, int kernel) {
  if (!ctx || kernel < SV_KERNEL_AUTO || kernel > SV_KERNEL_PIECES) return SV_ERR_INVALID_ARG;
  ctx->kernel = kernel;
  return SV_OK;
}

sv_status sv_kernel_for(const sv_ctx* ctx, int B, int* kernel) {
  if (!ctx || B < 1 || B > ctx->max_B || !kernel) return SV_ERR_INVALID_ARG;
  *kernel = use_pieces(ctx) ? SV_KERNEL_PIECES : SV_KERNEL_CLUSTER;
  return SV_OK;
}

sv_status sv_set_wait_limit_ns(sv_ctx* ctx, long long ns) {
  if (!ctx) return SV_ERR_INVALID_ARG;
  ctx->wait_limit_ns = ns < 0 ? sv::kDrainLimitNs : ns;
  return SV_OK;
}

}  // extern "C"
