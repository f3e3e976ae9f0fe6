// Acceptance-aware draft-length controller with the speculation toggle.
//
// "EfficientRollout: System-Aware Self-Speculative Decoding for RL
// Rollouts" (abstract) turns speculation on only where it pays for the
// system, and sets the draft budget from how well the drafter is doing;
// "ReSpec: Towards Optimizing Speculative Decoding in Reinforcement
// Learning Systems" (Adaptive Server) picks the SD configuration for the
// effective batch size from a performance model profiled offline, running
// without speculation while the batch is large.  Neither page gives
// formulas; this controller takes the plainest reading:
//
//   observe  a round of sequence b with draft length k_b > 0 and emitted
//            length a + 1 tested a + r drafts (r = 1 when a < k_b: the first
//            rejection); decayed counts A <- d A + a, N <- d N + (a + r);
//   estimate alpha_b = (A + alpha0 w0) / (N + w0), alpha0 without data;
//   expected tokens of a round of n drafts: E_n = sum_{j=0..n} alpha^j;
//   round time T(B, n): the caller's table at profiled batch sizes, linear
//            in B between two of them, the end row outside;
//   choose   batch mode: n* = argmax_n sum_b E_n(alpha_b) / T(B, n), the
//            smallest n on ties, for every row (n* = 0: speculation off);
//            per-sequence mode: n_b = argmax_n E_n(alpha_b) / T(B, n).
//
// The state (A, N per sequence slot) stays on the device, so a decode loop
// runs verify -> observe -> choose -> draft without a host round trip and
// can be captured in one CUDA graph.  The work is B rows of at most 32
// candidates, in fp64 with each multiply and add rounded on its own (no
// fused multiply-add), in the order stated above; a per-sequence rate is
// e_n * (1 / T(B, n)), which may differ from the quotient in the last bit.

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <new>
#include <utility>

#include "../../include/specverify.h"
#include "sv_internal.h"

namespace {

constexpr int kCtrlMaxK = 31;
constexpr int kCtrlMaxPoints = SV_CTRL_MAX_POINTS;
constexpr int kObserveThreads = 1024;
#ifndef SV_CTRL_CHOOSE_THREADS
#define SV_CTRL_CHOOSE_THREADS 128
#endif
constexpr int kChooseThreads = SV_CTRL_CHOOSE_THREADS;
constexpr int kChooseWarps = kChooseThreads / 32;
constexpr int kChooseMaxCtas = 1024;

// The round-time table travels by value in the launch parameters (3 KB).
struct CostTable {
  int n_points;
  int points[kCtrlMaxPoints];
  double time[kCtrlMaxPoints][kCtrlMaxK + 1];
};

struct ObserveParams {
  double* A;
  double* N;
  int* claim;                 // per slot, zero between calls
  unsigned int* err;          // error bits (1 << sv_status)
  const int32_t* seq_ids;
  const int32_t* draft_len;
  const int32_t* out_len;
  int B, n_slots, max_k;
  double decay;
};

struct ChooseParams {
  const double* A;
  const double* N;
  unsigned int* err;
  const int32_t* seq_ids;
  int32_t* next_len;
  int32_t* choice;
  double* alpha_out;          // spec_ctrl_alpha only
  double* cta_sums;           // [kChooseMaxCtas][kCtrlMaxK + 1]
  int* cta_max;               // [kChooseMaxCtas]
  unsigned int* ticket;       // zero between calls
  int B, n_slots, max_k, mode;
  double alpha0, w0;
  CostTable cost;
};

__device__ __forceinline__ double estimate(double A, double N, double alpha0, double w0) {
  const double den = __dadd_rn(N, w0);
  if (den == 0.0) return alpha0;
  return __ddiv_rn(__dadd_rn(A, __dmul_rn(alpha0, w0)), den);
}

__device__ double round_time(const CostTable& c, int B, int n) {
  const int last = c.n_points - 1;
  if (B <= c.points[0]) return c.time[0][n];
  if (B >= c.points[last]) return c.time[last][n];
  int j = 0;
  while (!(c.points[j] <= B && B < c.points[j + 1])) ++j;
  const double t0 = c.time[j][n], t1 = c.time[j + 1][n];
  const double f = __ddiv_rn(static_cast<double>(B - c.points[j]), static_cast<double>(c.points[j + 1] - c.points[j]));
  return __dadd_rn(t0, __dmul_rn(__dadd_rn(t1, -t0), f));
}

__device__ __forceinline__ bool bad_id(int id, int n_slots) { return id < 0 || id >= n_slots; }

// Programmatic dependent launch: a controller kernel may start while the
// kernel before it on the stream finishes; it waits here, before its first
// read of anything that kernel wrote, and lets the next kernel start early.
__device__ __forceinline__ void wait_for_predecessor() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void release_successor() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void raise_bits(unsigned int* err, unsigned int bits) {
  bits = __reduce_or_sync(0xffffffffu, bits);
  if ((threadIdx.x & 31) == 0 && bits) atomicOr(err, bits);
}

__global__ void __launch_bounds__(kObserveThreads) ctrl_observe_kernel(const ObserveParams P) {
  wait_for_predecessor();
  release_successor();
  // a slot named twice in one call is an error: count the claims first
  for (int b = threadIdx.x; b < P.B; b += blockDim.x) {
    const int id = P.seq_ids[b];
    if (!bad_id(id, P.n_slots)) atomicAdd(&P.claim[id], 1);
  }
  __syncthreads();
  unsigned int bits = 0;
  for (int b = threadIdx.x; b < P.B; b += blockDim.x) {
    const int id = P.seq_ids[b];
    if (bad_id(id, P.n_slots) || __ldcg(&P.claim[id]) != 1) {
      bits |= 1u << SV_ERR_INVALID_ARG;
      continue;
    }
    const int k = P.draft_len[b], len = P.out_len[b];
    if (k < 0 || k > P.max_k || len < 0 || len > k + 1) {
      bits |= 1u << SV_ERR_BAD_DRAFT_LEN;
      continue;
    }
    if (len == 0 || k == 0) continue;          // rejected by the verifier, or nothing tested
    const int a = len - 1;
    const int tested = a + (a < k ? 1 : 0);
    P.A[id] = __dadd_rn(__dmul_rn(P.decay, P.A[id]), static_cast<double>(a));
    P.N[id] = __dadd_rn(__dmul_rn(P.decay, P.N[id]), static_cast<double>(tested));
  }
  __syncthreads();
  for (int b = threadIdx.x; b < P.B; b += blockDim.x) {
    const int id = P.seq_ids[b];
    if (!bad_id(id, P.n_slots)) P.claim[id] = 0;
  }
  raise_bits(P.err, bits);
}

// One thread per row, rows spread over up to kChooseMaxCtas CTAs: fp64 runs at
// a small fraction of the fp32 rate, so the rows must use many SMs.  Batch
// mode sums E_n per CTA (fixed order), the last CTA to finish adds the CTA
// sums in CTA order, takes the first maximum of sum / T(B, n) and writes
// every row's length.
__global__ void __launch_bounds__(kChooseThreads) ctrl_choose_kernel(const ChooseParams P) {
  __shared__ double T[kCtrlMaxK + 1], invT[kCtrlMaxK + 1];
  __shared__ double tile[kCtrlMaxK + 1][kChooseThreads];   // batch mode: E_n of each thread's rows
  __shared__ double part[kChooseWarps][kCtrlMaxK + 1];
  __shared__ int wmax[kChooseWarps];
  __shared__ int best_s;
  __shared__ bool last_cta;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = P.max_k;
  if (tid <= K) {
    T[tid] = round_time(P.cost, P.B, tid);
    invT[tid] = __ddiv_rn(1.0, T[tid]);
  }
  wait_for_predecessor();
  release_successor();
  __syncthreads();

  const bool batch = (P.mode == SV_CTRL_BATCH) && !P.alpha_out;
  double acc[kCtrlMaxK + 1];
#pragma unroll
  for (int n = 0; n <= kCtrlMaxK; ++n) acc[n] = 0.0;
  unsigned int bits = 0;
  int top_n = 0;
  for (int b = blockIdx.x * kChooseThreads + tid; b < P.B; b += gridDim.x * kChooseThreads) {
    const int id = P.seq_ids[b];
    if (bad_id(id, P.n_slots)) {
      bits |= 1u << SV_ERR_INVALID_ARG;
      if (P.next_len) P.next_len[b] = 0;
      if (P.alpha_out) P.alpha_out[b] = __longlong_as_double(0x7ff8000000000000LL);
      continue;
    }
    const double alpha = estimate(P.A[id], P.N[id], P.alpha0, P.w0);
    if (P.alpha_out) {
      P.alpha_out[b] = alpha;
      continue;
    }
    // E_n built term by term: e_n = e_{n-1} + alpha^n
    double e = 0.0, pw = 1.0, best_rate = -1.0;
    int best = 0;
#pragma unroll
    for (int n = 0; n <= kCtrlMaxK; ++n) {
      if (n <= K) {
        e = __dadd_rn(e, pw);
        pw = __dmul_rn(pw, alpha);
        if (batch) {
          acc[n] = __dadd_rn(acc[n], e);
        } else {
          const double rate = __dmul_rn(e, invT[n]);
          if (rate > best_rate) {
            best_rate = rate;
            best = n;
          }
        }
      }
    }
    if (!batch) {
      P.next_len[b] = best;
      top_n = max(top_n, best);
    }
  }
  raise_bits(P.err, bits);
  if (P.alpha_out) return;

  // this CTA's part: the sums of E_n (batch) or the largest n_b.  Batch
  // sums go through shared memory so that each warp reduces only its own
  // share of the n (fp64 adds are the scarce resource here): warp w takes
  // n = w, w + W, ..., each lane first adds its column of the tile, then the
  // warp adds the 32 lane sums
  if (batch) {
#pragma unroll
    for (int n = 0; n <= kCtrlMaxK; ++n)
      if (n <= K) tile[n][tid] = acc[n];
  } else {
    top_n = __reduce_max_sync(0xffffffffu, top_n);
    if (lane == 0) wmax[warp] = top_n;
  }
  __syncthreads();
  if (batch) {
    for (int n = warp; n <= K; n += kChooseWarps) {
      double v = tile[n][lane];
#pragma unroll
      for (int i = 1; i < kChooseThreads / 32; ++i) v = __dadd_rn(v, tile[n][lane + 32 * i]);
      for (int o = 16; o > 0; o >>= 1) v = __dadd_rn(v, __shfl_down_sync(0xffffffffu, v, o));
      if (lane == 0) P.cta_sums[blockIdx.x * (kCtrlMaxK + 1) + n] = v;
    }
  }
  if (!batch && tid == 0) {
    int m = 0;
    for (int w = 0; w < kChooseWarps; ++w) m = max(m, wmax[w]);
    P.cta_max[blockIdx.x] = m;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) last_cta = (atomicAdd(P.ticket, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!last_cta) return;
  __threadfence();

  if (!batch) {
    if (tid == 0) {
      int m = 0;
      for (int c = 0; c < static_cast<int>(gridDim.x); ++c) m = max(m, __ldcg(&P.cta_max[c]));
      if (P.choice) *P.choice = m;
      *P.ticket = 0;
    }
    return;
  }
  if (tid <= K) {
    double v = 0.0;
#pragma unroll 8
    for (int c = 0; c < static_cast<int>(gridDim.x); ++c) v = __dadd_rn(v, __ldcg(&P.cta_sums[c * (kCtrlMaxK + 1) + tid]));
    part[0][tid] = __ddiv_rn(v, T[tid]);
  }
  __syncthreads();
  if (tid == 0) {
    double top = -1.0;
    int best = 0;
    for (int n = 0; n <= K; ++n) {
      if (part[0][n] > top) {
        top = part[0][n];
        best = n;
      }
    }
    best_s = best;
    if (P.choice) *P.choice = best;
    *P.ticket = 0;
  }
  __syncthreads();
  const int best = best_s;
  const bool vec = ((reinterpret_cast<uintptr_t>(P.seq_ids) | reinterpret_cast<uintptr_t>(P.next_len)) & 15u) == 0;
  const int B4 = vec ? (P.B & ~3) : 0;
  for (int b = 4 * tid; b < B4; b += 4 * kChooseThreads) {
    const int4 id = *reinterpret_cast<const int4*>(P.seq_ids + b);
    int4 o;
    o.x = bad_id(id.x, P.n_slots) ? 0 : best;
    o.y = bad_id(id.y, P.n_slots) ? 0 : best;
    o.z = bad_id(id.z, P.n_slots) ? 0 : best;
    o.w = bad_id(id.w, P.n_slots) ? 0 : best;
    *reinterpret_cast<int4*>(P.next_len + b) = o;
  }
  for (int b = B4 + tid; b < P.B; b += kChooseThreads)
    if (!bad_id(P.seq_ids[b], P.n_slots)) P.next_len[b] = best;
}

__global__ void ctrl_forget_kernel(double* A, double* N, const int32_t* ids, int n, int n_slots,
                                   unsigned int* err) {
  wait_for_predecessor();
  release_successor();
  unsigned int bits = 0;
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < n) {
    const int id = ids[b];
    if (bad_id(id, n_slots)) {
      bits = 1u << SV_ERR_INVALID_ARG;
    } else {
      A[id] = 0.0;
      N[id] = 0.0;
    }
  }
  raise_bits(err, bits);
}

}  // namespace

struct sv_ctrl {
  int n_slots = 0, max_k = 0;
  double* A = nullptr;
  double* N = nullptr;
  int* claim = nullptr;
  unsigned int* err = nullptr;
  double* cta_sums = nullptr;
  int* cta_max = nullptr;
  unsigned int* ticket = nullptr;
  double decay = 0.9, alpha0 = 0.5, w0 = 2.0;
  int mode = SV_CTRL_BATCH;
  bool has_cost = false;
  CostTable cost{};
};

namespace {

void release(sv_ctrl* c) {
  cudaFree(c->A);
  cudaFree(c->N);
  cudaFree(c->claim);
  cudaFree(c->err);
  cudaFree(c->cta_sums);
  cudaFree(c->cta_max);
  cudaFree(c->ticket);
  delete c;
}

// Launch with programmatic stream serialisation (see wait_for_predecessor).
template <typename... KArgs, typename... Args>
sv_status launch_pdl(const char* name, void (*kernel)(KArgs...), int ctas, int threads, cudaStream_t s,
                     Args&&... args) {
  sv::NvtxRange range(name);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...) == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // namespace

extern "C" {

sv_status spec_ctrl_create(sv_ctrl** out, int n_slots, int max_k) {
  if (!out) return SV_ERR_INVALID_ARG;
  *out = nullptr;
  if (n_slots < 1 || n_slots > (1 << 24) || max_k < 0 || max_k > kCtrlMaxK) return SV_ERR_INVALID_ARG;
  sv_ctrl* c = new (std::nothrow) sv_ctrl;
  if (!c) return SV_ERR_CUDA;
  c->n_slots = n_slots;
  c->max_k = max_k;
  const size_t n = static_cast<size_t>(n_slots);
  if (cudaMalloc(&c->A, n * sizeof(double)) != cudaSuccess || cudaMalloc(&c->N, n * sizeof(double)) != cudaSuccess ||
      cudaMalloc(&c->claim, n * sizeof(int)) != cudaSuccess || cudaMalloc(&c->err, sizeof(unsigned int)) != cudaSuccess ||
      cudaMemset(c->A, 0, n * sizeof(double)) != cudaSuccess || cudaMemset(c->N, 0, n * sizeof(double)) != cudaSuccess ||
      cudaMemset(c->claim, 0, n * sizeof(int)) != cudaSuccess || cudaMemset(c->err, 0, sizeof(unsigned int)) != cudaSuccess ||
      cudaMalloc(&c->cta_sums, sizeof(double) * kChooseMaxCtas * (kCtrlMaxK + 1)) != cudaSuccess ||
      cudaMalloc(&c->cta_max, sizeof(int) * kChooseMaxCtas) != cudaSuccess ||
      cudaMalloc(&c->ticket, sizeof(unsigned int)) != cudaSuccess ||
      cudaMemset(c->ticket, 0, sizeof(unsigned int)) != cudaSuccess) {
    cudaGetLastError();
    release(c);
    return SV_ERR_CUDA;
  }
  *out = c;
  return SV_OK;
}

sv_status spec_ctrl_destroy(sv_ctrl* c) {
  if (!c) return SV_ERR_INVALID_ARG;
  release(c);
  return SV_OK;
}

sv_status spec_ctrl_set_cost(sv_ctrl* c, int n_points, const int* batch_sizes, const double* round_time) {
  if (!c || !batch_sizes || !round_time || n_points < 1 || n_points > kCtrlMaxPoints) return SV_ERR_INVALID_ARG;
  const int K1 = c->max_k + 1;
  for (int j = 0; j < n_points; ++j) {
    if (batch_sizes[j] < 1 || (j > 0 && batch_sizes[j] <= batch_sizes[j - 1])) return SV_ERR_INVALID_ARG;
    for (int n = 0; n < K1; ++n) {
      const double t = round_time[static_cast<size_t>(j) * K1 + n];
      if (!(t > 0.0) || !std::isfinite(t)) return SV_ERR_INVALID_ARG;
    }
  }
  CostTable t{};
  t.n_points = n_points;
  for (int j = 0; j < n_points; ++j) {
    t.points[j] = batch_sizes[j];
    for (int n = 0; n < K1; ++n) t.time[j][n] = round_time[static_cast<size_t>(j) * K1 + n];
  }
  c->cost = t;
  c->has_cost = true;
  return SV_OK;
}

sv_status spec_ctrl_set_params(sv_ctrl* c, double decay, double prior_alpha, double prior_weight, sv_ctrl_mode mode) {
  if (!c) return SV_ERR_INVALID_ARG;
  if (!(decay > 0.0 && decay <= 1.0)) return SV_ERR_INVALID_ARG;
  if (!(prior_alpha >= 0.0 && prior_alpha <= 1.0)) return SV_ERR_INVALID_ARG;
  if (!(prior_weight >= 0.0) || !std::isfinite(prior_weight)) return SV_ERR_INVALID_ARG;
  if (mode != SV_CTRL_BATCH && mode != SV_CTRL_PER_SEQUENCE) return SV_ERR_INVALID_ARG;
  c->decay = decay;
  c->alpha0 = prior_alpha;
  c->w0 = prior_weight;
  c->mode = mode;
  return SV_OK;
}

sv_status spec_ctrl_reset(sv_ctrl* c, int n, const int32_t* seq_ids, sv_stream_t stream) {
  if (!c) return SV_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!seq_ids) {
    const size_t bytes = static_cast<size_t>(c->n_slots) * sizeof(double);
    cudaError_t e = cudaMemsetAsync(c->A, 0, bytes, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(c->N, 0, bytes, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(c->err, 0, sizeof(unsigned int), s);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
  }
  if (n < 0 || n > c->n_slots) return SV_ERR_INVALID_ARG;
  if (n == 0) return SV_OK;
  return launch_pdl("spec_ctrl_reset", ctrl_forget_kernel, (n + 255) / 256, 256, s, c->A, c->N, seq_ids, n, c->n_slots, c->err);
}

sv_status spec_ctrl_observe(sv_ctrl* c, int B, const int32_t* seq_ids, const int32_t* draft_len,
                            const int32_t* out_len, sv_stream_t stream) {
  if (!c || B < 0 || B > c->n_slots) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!seq_ids || !draft_len || !out_len) return SV_ERR_INVALID_ARG;
  ObserveParams p{c->A, c->N, c->claim, c->err, seq_ids, draft_len, out_len, B, c->n_slots, c->max_k, c->decay};
  return launch_pdl("spec_ctrl_observe", ctrl_observe_kernel, 1, kObserveThreads, reinterpret_cast<cudaStream_t>(stream), p);
}

static sv_status launch_choose(sv_ctrl* c, int B, const int32_t* seq_ids, int32_t* next_len, int32_t* choice,
                               double* alpha_out, sv_stream_t stream) {
  ChooseParams p{};
  p.A = c->A;
  p.N = c->N;
  p.err = c->err;
  p.seq_ids = seq_ids;
  p.next_len = next_len;
  p.choice = choice;
  p.alpha_out = alpha_out;
  p.B = B;
  p.n_slots = c->n_slots;
  p.max_k = c->max_k;
  p.mode = c->mode;
  p.alpha0 = c->alpha0;
  p.w0 = c->w0;
  p.cost = c->cost;
  p.cta_sums = c->cta_sums;
  p.cta_max = c->cta_max;
  p.ticket = c->ticket;
  const int ctas = B < 1 ? 1 : (B + kChooseThreads - 1) / kChooseThreads;
  return launch_pdl("spec_ctrl_choose", ctrl_choose_kernel, ctas < kChooseMaxCtas ? ctas : kChooseMaxCtas, kChooseThreads,
                    reinterpret_cast<cudaStream_t>(stream), p);
}

sv_status spec_ctrl_choose(sv_ctrl* c, int B, const int32_t* seq_ids, int32_t* next_draft_len, int32_t* choice,
                           sv_stream_t stream) {
  if (!c || !c->has_cost || B < 0 || B > c->n_slots) return SV_ERR_INVALID_ARG;
  if (B > 0 && (!seq_ids || !next_draft_len)) return SV_ERR_INVALID_ARG;
  if (B == 0 && !choice) return SV_OK;
  return launch_choose(c, B, seq_ids, next_draft_len, choice, nullptr, stream);
}

sv_status spec_ctrl_alpha(sv_ctrl* c, int B, const int32_t* seq_ids, double* alpha, sv_stream_t stream) {
  if (!c || B < 0 || B > c->n_slots) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!seq_ids || !alpha) return SV_ERR_INVALID_ARG;
  return launch_choose(c, B, seq_ids, nullptr, nullptr, alpha, stream);
}

sv_status spec_ctrl_status(sv_ctrl* c, sv_stream_t stream) {
  if (!c) return SV_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned int word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, c->err, sizeof word, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  if (word & (1u << SV_ERR_INVALID_ARG)) return SV_ERR_INVALID_ARG;
  if (word & (1u << SV_ERR_BAD_DRAFT_LEN)) return SV_ERR_BAD_DRAFT_LEN;
  return SV_OK;
}

}  // extern "C"
