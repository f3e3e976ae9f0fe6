// Speculative-sampling verification kernels for sm_103a.
//
// Work unit ("item"): a (target row i, draft row i) pair of sequence b with
// i < k_b, or the bonus target row k_b of sequence b.
//
// plan_kernel (one CTA) lists the items position-major (every sequence's
// position 0, then position 1, ..., then all bonus rows), resets the
// per-sequence words and the ticket counter, and handles sequences whose
// draft length is invalid.
//
// verify_kernel is persistent: each thread-block CLUSTER pulls items with an
// atomic ticket and its CTAs split the vocabulary.  Every CTA keeps `stages`
// shared-memory buffers; while it computes on one item, cp.async.bulk is
// already staging the rows of the next ones, so each needed logit crosses
// HBM exactly once and the copy engine never idles.  Per item:
//
//   local    slice maximum m_r and sum s_r = sum 2^(z c - fl(m_r c)),
//            c = log2(e)/T, plus the drafted token's logits
//   barrier  cluster combine through distributed shared memory:
//            M = max m_r, S = sum s_r 2^(fl(m_r c) - fl(M c))
//   test     alpha = min(1, p(x)/q(x)); accept iff u < alpha
//   draw     (rejected pair: w = max(0, p - q); bonus row: w = p)
//            per-warp totals -> barrier -> cluster scan in rank order ->
//            the CTA holding s*S walks its warp's chunk to the token
//
// Items of one sequence run in different clusters; the last one to finish
// (threadfence + atomic counter, no waiting) writes the sequence's outputs.
// A rejecting pair does atomicMin on its sequence's first-rejection word and
// skips its draw when an earlier position already rejected; the bonus row
// skips its draw when any rejection is known.  Position-major order makes
// earlier positions finish first, so most useless draws are skipped.
//
// The rule implemented (accept with min(1, p/q), stop at the first
// rejection, resample from max(0, p - q) or draw the bonus token from the
// last target row) is the standard speculative-sampling rule: the reading of
// "rejection sampling based on the verifier's probability distribution" in
// "Accelerating RL Post-Training Rollouts via System-Integrated Speculative
// Decoding", §2 core mechanism.

#include <cuda_runtime.h>
#include <cstdint>
#include <cmath>

#include "sv_internal.h"

namespace sv {
namespace {

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t remote_addr(const void* local, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_addr(local)), "r"(rank));
  return out;
}

__device__ __forceinline__ float ld_remote_f32(const void* local, uint32_t rank) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote_addr(local, rank)) : "memory");
  return v;
}

__device__ __forceinline__ double ld_remote_f64(const void* local, uint32_t rank) {
  double v;
  asm volatile("ld.shared::cluster.f64 %0, [%1];" : "=d"(v) : "r"(remote_addr(local, rank)) : "memory");
  return v;
}

__device__ __forceinline__ int ld_remote_s32(const void* local, uint32_t rank) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(remote_addr(local, rank)) : "memory");
  return v;
}

__device__ __forceinline__ void st_remote_s32(void* local, uint32_t rank, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" :: "r"(remote_addr(local, rank)), "r"(v) : "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile("{\n\t.reg .pred p;\n\t"
               "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(done) : "r"(smem_addr(bar)), "r"(parity) : "memory");
  return done != 0;
}

// Global -> shared bulk copy completing on `bar` (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Programmatic dependent launch: wait until the preceding grid's writes are
// visible / let the dependent grid start launching.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 2^x on the special-function unit (PTX ex2.approx; -inf -> +0, NaN -> NaN).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Bounded wait on an mbarrier phase.  Returns false if `limit_ns` passed
// before the phase completed.  A limit <= 0 is the error-path test hook: it
// always reports expiry (the caller then drains the copies with a 1 s wait).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, long long limit_ns) {
  if (limit_ns <= 0) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (static_cast<long long>(global_ns() - t0) >= limit_ns) return false;
  }
  return true;
}

// ---------------------------------------------------------------------------
// Logit vectors: 16 bytes = 8 bf16 or 4 fp32 values.
// ---------------------------------------------------------------------------

template <int ELT> struct Vec;
template <> struct Vec<2> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void load(const unsigned char* p, float (&v)[8]) {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[2 * j] = __uint_as_float(ws[j] << 16);
      v[2 * j + 1] = __uint_as_float(ws[j] & 0xffff0000u);
    }
  }
  __device__ __forceinline__ static float scalar(const unsigned char* base, int idx) {
    const uint16_t h = reinterpret_cast<const uint16_t*>(base)[idx];
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
  }
  __device__ __forceinline__ static void store_scalar(unsigned char* base, int idx, float v) {
    reinterpret_cast<uint16_t*>(base)[idx] = static_cast<uint16_t>(__float_as_uint(v) >> 16);
  }
};
template <> struct Vec<4> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void load(const unsigned char* p, float (&v)[4]) {
    const float4 w = *reinterpret_cast<const float4*>(p);
    v[0] = w.x; v[1] = w.y; v[2] = w.z; v[3] = w.w;
  }
  __device__ __forceinline__ static float scalar(const unsigned char* base, int idx) {
    return reinterpret_cast<const float*>(base)[idx];
  }
  __device__ __forceinline__ static void store_scalar(unsigned char* base, int idx, float v) {
    reinterpret_cast<float*>(base)[idx] = v;
  }
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ int warp_or(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v |= __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// (value, index) maximum, ties to the lower index.
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
  }
}

// ---------------------------------------------------------------------------
// Shared control block (first kCtrlBytes of dynamic shared memory).
// ---------------------------------------------------------------------------

// Values a CTA publishes to its cluster for one item.  Two copies alternate
// between consecutive items, so a CTA can publish item j+1 while another CTA
// is still reading item j.
struct Pub {
  float m_t, s_t, m_d, s_d;   // slice maximum and sum relative to fl(m c)
  float zt_x, zd_x;           // logits at the drafted token (owner CTA only)
  int arg_t;                  // greedy: first index of the slice maximum
  int flags;                  // bit0 wait timed out, bit1 non-finite seen (greedy)
  double W;                   // this CTA's total draw weight
  int skip;                   // this CTA skipped the draw
  int pad_;
};

struct Ctrl {
  uint64_t bar[kMaxStages];   // staging barrier per buffer
  int inbox[kMaxStages];      // tickets written by the cluster leader
  int2 desc[kMaxStages];      // item staged in each buffer ({-1, 0} = none)
  Pub pub[2];
  float red_f[64];
  int red_i[64];
  double warp_W[32];
  // cluster-wide values of the current item (same in every CTA)
  float g_Kt, g_Kd, g_Lt, g_Ld, g_zt_x, g_zd_x, g_Mt, g_Md;
  int g_arg_t, g_flags, g_accept, g_compute, g_skip, g_rstar, g_found_warp, g_y;
  double g_S, g_target;
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block too large");

// ---------------------------------------------------------------------------
// Sequence bookkeeping
// ---------------------------------------------------------------------------

// Sequence epilogue, run by the item that finishes last.
__device__ void finalize_sequence(const VerifyParams& P, int b, int kb) {
  const Workspace& ws = P.ws;
  const int err = __ldcg(ws.seq_err + b);
  const int rmin = __ldcg(ws.rej_min + b);
  int* ot = P.out_tokens + static_cast<size_t>(b) * (P.k + 1);
  if (err) {
    for (int j = 0; j <= P.k; ++j) ot[j] = -1;
    P.out_len[b] = 0;
    atomicAdd(ws.stats + kStatErrorSeqs, 1ull);
    return;
  }
  const int a = rmin < kb ? rmin : kb;
  const int y = __ldcg(ws.y_slot + static_cast<size_t>(b) * (P.k + 1) + a);
  const int* xt = P.tokens + static_cast<size_t>(b) * P.k;
  for (int j = 0; j < a; ++j) ot[j] = xt[j];
  ot[a] = y;
  for (int j = a + 1; j <= P.k; ++j) ot[j] = -1;
  P.out_len[b] = a + 1;
  atomicAdd(ws.stats + kStatSequences, 1ull);
  atomicAdd(ws.stats + kStatProposed, static_cast<unsigned long long>(kb));
  atomicAdd(ws.stats + kStatAccepted, static_cast<unsigned long long>(a));
  atomicAdd(ws.stats + kStatEmitted, static_cast<unsigned long long>(a + 1));
  if (kb == 0) atomicAdd(ws.stats + kStatSpecOff, 1ull);
}

// Report one finished item; the last of the sequence's k_b + 1 items
// finalises it.  `y` < -1 means "no token recorded".
__device__ void report_item(const VerifyParams& P, int b, int kb, int pos, int y) {
  if (y >= -1) P.ws.y_slot[static_cast<size_t>(b) * (P.k + 1) + pos] = y;
  __threadfence();
  const int prev = atomicAdd(P.ws.done + b, 1);
  if (prev == kb) {
    __threadfence();
    finalize_sequence(P, b, kb);
  }
}

__device__ void mark_error(const VerifyParams& P, int b, int code) {
  atomicOr(P.ws.seq_err + b, 1 << code);
  atomicOr(P.ws.err_word, 1u << code);
}

// ---------------------------------------------------------------------------
// plan_kernel: the work list and per-call resets (one CTA).
// ---------------------------------------------------------------------------
constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const VerifyParams P) {
  grid_dependents_launch();   // the verify grid may start its prologue now
  __shared__ int warp_cnt[32];
  __shared__ int base;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = P.B, k = P.k;
  const Workspace& ws = P.ws;
  // per-sequence resets, diagnostics cleared to NaN, invalid draft lengths
  for (int b = tid; b < B; b += kPlanThreads) {
    ws.done[b] = 0;
    ws.rej_min[b] = kNoReject;
    ws.seq_err[b] = 0;
    const int kb = P.draft_len[b];
    if (kb < 0 || kb > k) {
      int* ot = P.out_tokens + static_cast<size_t>(b) * (k + 1);
      for (int j = 0; j <= k; ++j) ot[j] = -1;
      P.out_len[b] = 0;
      atomicOr(ws.err_word, 1u << 2 /* SV_ERR_BAD_DRAFT_LEN */);
      atomicAdd(ws.stats + kStatErrorSeqs, 1ull);
    }
  }
  for (int i = tid; i < B * (k + 1); i += kPlanThreads) {
    ws.m_t[i] = NAN; ws.L_t[i] = NAN; ws.mass[i] = NAN;
  }
  for (int i = tid; i < B * k; i += kPlanThreads) {
    ws.m_d[i] = NAN; ws.L_d[i] = NAN; ws.alpha[i] = NAN;
  }
  if (tid == 0) { base = 0; *ws.ticket = 0; }
  __syncthreads();
  // position-major list: level L < k holds pairs (b, L) with k_b > L;
  // level k holds the bonus row (b, k_b) of every valid sequence
  for (int L = 0; L <= k; ++L) {
    for (int b0 = 0; b0 < B; b0 += kPlanThreads) {
      const int b = b0 + tid;
      int kb = -1;
      if (b < B) kb = P.draft_len[b];
      const bool valid = kb >= 0 && kb <= k;
      const bool take = valid && (L < k ? kb > L : true);
      const unsigned m = __ballot_sync(0xffffffffu, take);
      if (lane == 0) warp_cnt[warp] = __popc(m);
      __syncthreads();
      if (warp == 0) {
        const int c = warp_cnt[lane];
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int up = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += up;
        }
        warp_cnt[lane] = incl - c;
      }
      __syncthreads();
      if (take) {
        const int idx = base + warp_cnt[warp] + __popc(m & ((1u << lane) - 1u));
        const int pos = L < k ? L : kb;
        ws.items[idx] = make_int2(b, (pos << 1) | (L < k ? 1 : 0));
      }
      __syncthreads();
      if (tid == kPlanThreads - 1) base += warp_cnt[31] + __popc(m);
      __syncthreads();
    }
  }
  if (tid == 0) *ws.n_items = base;
}

// ---------------------------------------------------------------------------
// verify_kernel
// ---------------------------------------------------------------------------

template <int ELT>
__global__ void __launch_bounds__(kThreads)
verify_kernel(const VerifyParams P) {
  using V = Vec<ELT>;
  constexpr int NV = V::N;          // logits per 16-byte vector
  constexpr int NW = kThreads / 32;
  extern __shared__ __align__(128) unsigned char smem[];
  Ctrl& C = *reinterpret_cast<Ctrl*>(smem);

  const uint32_t CS = cluster_size();
  const uint32_t rank = cluster_rank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = P.k;
  const int S = P.stages;
  const float c2 = P.c2;

  // this CTA's slice of every row, and this warp's part of it
  const int lo = static_cast<int>(rank) * P.slice;
  const int hi = min(P.V, lo + P.slice);
  const int n = max(0, hi - lo);
  const int nvec = (n + NV - 1) / NV;
  const int vpw = (nvec + NW - 1) / NW;
  const int v0 = warp * vpw;
  const int v1 = min(nvec, v0 + vpw);
  const int row_pad = ((P.slice * ELT + 127) / 128) * 128;
  auto bufT = [&](int s) { return smem + kCtrlBytes + s * 2 * row_pad; };
  auto bufD = [&](int s) { return smem + kCtrlBytes + s * 2 * row_pad + row_pad; };

  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&C.bar[s], 1);
    mbar_fence_init();
  }
  grid_dependency_wait();           // the work list of plan_kernel is ready
  const int n_items = __ldcg(P.ws.n_items);
  const bool leader = (rank == 0 && tid == 0);

  // stage item `t` (a ticket) into buffer s; records the descriptor
  auto stage = [&](int s, int t) {
    int2 d = make_int2(-1, 0);
    if (t < n_items) d = __ldcg(P.ws.items + t);
    C.desc[s] = d;
    if (d.x < 0 || !P.bulk || n == 0) return;
    const int b = d.x, pos = d.y >> 1;
    const bool pair = (d.y & 1) && !P.greedy;
    const uint32_t bytes = static_cast<uint32_t>(n) * ELT;
    const unsigned char* gT = static_cast<const unsigned char*>(P.target) +
        ((static_cast<size_t>(b) * (k + 1) + pos) * P.V + lo) * ELT;
    mbar_expect_tx(&C.bar[s], pair ? 2 * bytes : bytes);
    constexpr uint32_t kChunk = 32768;
    for (uint32_t o = 0; o < bytes; o += kChunk)
      bulk_load(bufT(s) + o, gT + o, min(kChunk, bytes - o), &C.bar[s]);
    if (pair) {
      const unsigned char* gD = static_cast<const unsigned char*>(P.draft) +
          ((static_cast<size_t>(b) * k + pos) * P.V + lo) * ELT;
      for (uint32_t o = 0; o < bytes; o += kChunk)
        bulk_load(bufD(s) + o, gD + o, min(kChunk, bytes - o), &C.bar[s]);
    }
  };
  // plain-load staging (rows not 16-byte aligned): every thread helps; the
  // tail of the last vector is padded with -inf
  auto stage_plain = [&](int s) {
    const int2 d = C.desc[s];
    if (d.x < 0 || P.bulk) return;
    const int b = d.x, pos = d.y >> 1;
    const bool pair = (d.y & 1) && !P.greedy;
    const unsigned char* gT = static_cast<const unsigned char*>(P.target) +
        ((static_cast<size_t>(b) * (k + 1) + pos) * P.V + lo) * ELT;
    const unsigned char* gD = pair ? static_cast<const unsigned char*>(P.draft) +
        ((static_cast<size_t>(b) * k + pos) * P.V + lo) * ELT : nullptr;
    for (int e = tid; e < nvec * NV; e += kThreads) {
      V::store_scalar(bufT(s), e, e < n ? V::scalar(gT, e) : -INFINITY);
      if (pair) V::store_scalar(bufD(s), e, e < n ? V::scalar(gD, e) : -INFINITY);
    }
  };

  // prologue: the leader takes S tickets and hands them to every CTA
  if (leader) {
    const int t0 = atomicAdd(P.ws.ticket, S);
    for (uint32_t r = 0; r < CS; ++r)
      for (int s = 0; s < S; ++s) st_remote_s32(&C.inbox[s], r, t0 + s);
  }
  cluster_barrier();
  if (tid == 0)
    for (int s = 0; s < S; ++s) stage(s, C.inbox[s]);
  __syncthreads();
  for (int s = 0; s < S; ++s) stage_plain(s);
  __syncthreads();

  for (int j = 0;; ++j) {
    const int s = j % S;
    const int2 d = C.desc[s];
    if (d.x < 0) break;             // same ticket stream in every CTA: uniform
    const int pb = j & 1;
    const int b = d.x, pos = d.y >> 1;
    const bool pair = (d.y & 1) != 0;
    const int kb = __ldg(P.draft_len + b);
    const bool use_draft = pair && !P.greedy;
    const int x = pair ? __ldg(P.tokens + static_cast<size_t>(b) * k + pos) : -1;
    const bool bad_token = pair && (x < 0 || x >= P.V);
    const unsigned char* T_ = bufT(s);
    const unsigned char* D_ = bufD(s);

    // ---- wait for the staged slice ----------------------------------------
    int my_flags = 0;
    if (P.bulk && n > 0) {
      const uint32_t parity = static_cast<uint32_t>(j / S) & 1u;
      if (!mbar_wait_bounded(&C.bar[s], parity, P.wait_limit_ns)) {
        my_flags |= 1;
        mbar_wait_bounded(&C.bar[s], parity, kDrainLimitNs);
      }
    }
    my_flags = __syncthreads_or(my_flags);

    // ---- local pass: slice maximum and sum (or argmax when greedy) --------
    float mt = -INFINITY, md = -INFINITY, st = 0.f, sd = 0.f;
    int arg = 0x7fffffff;
    int bad = 0;
    if (!bad_token) {
      if (P.greedy) {
        for (int v = v0 + lane; v < v1; v += 32) {
          float z[NV];
          V::load(T_ + v * 16, z);
#pragma unroll
          for (int e = 0; e < NV; ++e) {
            bad |= (z[e] != z[e]) || (z[e] == INFINITY);
            if (z[e] > mt) { mt = z[e]; arg = lo + v * NV + e; }
          }
        }
        warp_argmax(mt, arg);
        bad = warp_or(bad);
      } else {
        for (int v = v0 + lane; v < v1; v += 32) {
          float z[NV];
          V::load(T_ + v * 16, z);
#pragma unroll
          for (int e = 0; e < NV; ++e) mt = fmaxf(mt, z[e]);
          if (use_draft) {
            V::load(D_ + v * 16, z);
#pragma unroll
            for (int e = 0; e < NV; ++e) md = fmaxf(md, z[e]);
          }
        }
        mt = warp_max(mt);
        md = warp_max(md);
      }
      if (lane == 0) { C.red_f[warp] = mt; C.red_f[NW + warp] = md; C.red_i[warp] = arg; C.red_i[NW + warp] = bad; }
      __syncthreads();
      if (P.greedy) {
        if (warp == 0) {
          float m = lane < NW ? C.red_f[lane] : -INFINITY;
          int a = lane < NW ? C.red_i[lane] : 0x7fffffff;
          warp_argmax(m, a);
          mt = m;
          arg = a;
          bad = warp_or(lane < NW ? C.red_i[NW + lane] : 0);
        }
      } else {
        mt = C.red_f[0];
        md = C.red_f[NW];
        for (int w = 1; w < NW; ++w) { mt = fmaxf(mt, C.red_f[w]); md = fmaxf(md, C.red_f[NW + w]); }
        // K = fl(m c), rounded once and used identically wherever this slice's
        // sum is rescaled (no contraction into an FMA)
        const float Kt = __fmul_rn(mt, c2), Kd = __fmul_rn(md, c2);
        for (int v = v0 + lane; v < v1; v += 32) {
          float z[NV];
          V::load(T_ + v * 16, z);
#pragma unroll
          for (int e = 0; e < NV; ++e) st += fast_exp2(fmaf(z[e], c2, -Kt));
          if (use_draft) {
            V::load(D_ + v * 16, z);
#pragma unroll
            for (int e = 0; e < NV; ++e) sd += fast_exp2(fmaf(z[e], c2, -Kd));
          }
        }
        st = warp_sum(st);
        sd = warp_sum(sd);
        __syncthreads();            // red_f is reused below
        if (lane == 0) { C.red_f[warp] = st; C.red_f[NW + warp] = sd; }
        __syncthreads();
        if (tid == 0) {
          st = 0.f; sd = 0.f;
          for (int w = 0; w < NW; ++w) { st += C.red_f[w]; sd += C.red_f[NW + w]; }
          if (mt == -INFINITY) st = 0.f;      // empty or fully masked slice
          if (md == -INFINITY) sd = 0.f;
        }
      }
    }

    // ---- publish, take the next ticket, cluster barrier A -------------------
    if (tid == 0) {
      Pub& pp = C.pub[pb];
      pp.m_t = mt; pp.s_t = st; pp.m_d = md; pp.s_d = sd; pp.arg_t = arg;
      pp.flags = my_flags | (bad ? 2 : 0);
      pp.zt_x = NAN; pp.zd_x = NAN;
      if (pair && !bad_token && x >= lo && x < hi) {
        pp.zt_x = V::scalar(T_, x - lo);
        if (use_draft) pp.zd_x = V::scalar(D_, x - lo);
      }
    }
    if (leader) {
      const int t = atomicAdd(P.ws.ticket, 1);
      for (uint32_t r = 0; r < CS; ++r) st_remote_s32(&C.inbox[s], r, t);
    }
    cluster_barrier();  // A

    // ---- cluster combine (warp 0, one lane per CTA) -------------------------
    int next_t = 0;
    if (warp == 0) {
      const bool in = lane < static_cast<int>(CS);
      const uint32_t r = in ? static_cast<uint32_t>(lane) : 0u;
      float rmt = in ? ld_remote_f32(&C.pub[pb].m_t, r) : -INFINITY;
      const float rst = in ? ld_remote_f32(&C.pub[pb].s_t, r) : 0.f;
      const float rmd = in ? ld_remote_f32(&C.pub[pb].m_d, r) : -INFINITY;
      const float rsd = in ? ld_remote_f32(&C.pub[pb].s_d, r) : 0.f;
      int rarg = in ? ld_remote_s32(&C.pub[pb].arg_t, r) : 0x7fffffff;
      const int rfl = in ? ld_remote_s32(&C.pub[pb].flags, r) : 0;
      int fl = warp_or(rfl);
      if (P.greedy) {
        warp_argmax(rmt, rarg);
        if (!(rmt > -INFINITY) && !bad_token) fl |= 2;
        if (lane == 0) { C.g_Mt = rmt; C.g_arg_t = rarg; C.g_flags = fl; }
      } else {
        const float Mt = warp_max(rmt);
        const float Md = warp_max(rmd);
        const float Kt = __fmul_rn(Mt, c2), Kd = __fmul_rn(Md, c2);
        // s_r was summed relative to fl(m_r c): rescale by 2^(fl(m_r c) - fl(M c))
        const float tt = (rmt == -INFINITY) ? 0.f : rst * fast_exp2(__fsub_rn(__fmul_rn(rmt, c2), Kt));
        const float td = (rmd == -INFINITY) ? 0.f : rsd * fast_exp2(__fsub_rn(__fmul_rn(rmd, c2), Kd));
        const float St = warp_sum(tt), Sd = warp_sum(td);
        if (lane == 0) {
          C.g_Mt = Mt; C.g_Md = Md;
          C.g_Kt = Kt; C.g_Kd = Kd;
          C.g_Lt = log2f(St);
          C.g_Ld = use_draft ? log2f(Sd) : 0.f;
          bool nonfinite = !(isfinite(Mt) && isfinite(St) && St > 0.f);
          if (use_draft) nonfinite |= !(isfinite(Md) && isfinite(Sd) && Sd > 0.f);
          if (nonfinite && !bad_token) fl |= 2;
          C.g_flags = fl;
        }
      }
      if (pair && !bad_token && lane == 0) {
        const uint32_t owner = static_cast<uint32_t>(x / P.slice);
        C.g_zt_x = ld_remote_f32(&C.pub[pb].zt_x, owner);
        C.g_zd_x = use_draft ? ld_remote_f32(&C.pub[pb].zd_x, owner) : 0.f;
      }
      if (lane == 0) next_t = C.inbox[s];
    }
    __syncthreads();

    const size_t slot_t = static_cast<size_t>(b) * (k + 1) + pos;
    const size_t slot_d = static_cast<size_t>(b) * k + pos;
    const int flags = C.g_flags;

    if (bad_token || flags) {
      // ---- errors: the sequence emits nothing ---------------------------
      if (leader) {
        if (bad_token) mark_error(P, b, 3 /* SV_ERR_BAD_TOKEN */);
        if (flags & 1) mark_error(P, b, 5 /* SV_ERR_TIMEOUT */);
        if (flags & 2) mark_error(P, b, 4 /* SV_ERR_NONFINITE */);
        report_item(P, b, kb, pos, -2);
      }
    } else if (P.greedy) {
      // ---- T == 0: accept iff x is the first argmax ---------------------
      if (leader) {
        P.ws.m_t[slot_t] = C.g_Mt;
        if (pair) {
          const bool acc = (x == C.g_arg_t);
          P.ws.alpha[slot_d] = acc ? 1.f : 0.f;
          if (!acc) atomicMin(P.ws.rej_min + b, pos);
        }
        report_item(P, b, kb, pos, C.g_arg_t);
      }
    } else {
      // ---- acceptance test (identical in every CTA) ---------------------
      const float Kt = C.g_Kt, Kd = C.g_Kd, Lt = C.g_Lt, Ld = C.g_Ld;
      if (tid == 0) {
        int accept = 0;
        float alpha = NAN;
        if (pair) {
          const float zt = C.g_zt_x, zd = C.g_zd_x;
          if (zt == -INFINITY) alpha = 0.f;               // p(x) = 0
          else if (zd == -INFINITY) alpha = 1.f;          // q(x) = 0 < p(x)
          else {
            const float log2r = (fmaf(zt, c2, -Kt) - Lt) - (fmaf(zd, c2, -Kd) - Ld);
            alpha = log2r >= 0.f ? 1.f : exp2f(log2r);
          }
          const float u = __ldg(P.uniforms + static_cast<size_t>(b) * (k + 1) + pos);
          accept = (u < alpha) ? 1 : 0;
        }
        C.g_accept = accept;
        if (rank == 0) {
          // debug: log-sum-exp(z/T) = m/T + L ln 2 (to within the rounding of fl(m c))
          P.ws.m_t[slot_t] = C.g_Mt;
          P.ws.L_t[slot_t] = Lt;
          if (pair) {
            P.ws.m_d[slot_d] = C.g_Md;
            P.ws.L_d[slot_d] = Ld;
            P.ws.alpha[slot_d] = alpha;
          }
        }
        int compute = 0;
        if (pair && !accept) compute = atomicMin(P.ws.rej_min + b, pos) >= pos;
        else if (!pair) compute = __ldcg(P.ws.rej_min + b) == kNoReject;
        C.g_compute = compute;
      }
      __syncthreads();

      if (pair && C.g_accept) {
        if (leader) report_item(P, b, kb, pos, -2);
      } else {
        // ---- the draw ----------------------------------------------------
        const float s_u = __ldg(P.uniforms + static_cast<size_t>(b) * (k + 1) + k);
        bool resid = pair;
        auto vec_weights = [&](int v, float (&w)[NV]) {
          float zt[NV], zd[NV];
          V::load(T_ + v * 16, zt);
          if (resid) V::load(D_ + v * 16, zd);
#pragma unroll
          for (int e = 0; e < NV; ++e) {
            const float p = fast_exp2(fmaf(zt[e], c2, -Kt) - Lt);
            w[e] = resid ? fmaxf(p - fast_exp2(fmaf(zd[e], c2, -Kd) - Ld), 0.f) : p;
          }
        };
        int zero_resid = 0, y = -2, reporter = 0;
        for (int attempt = 0; attempt < 2; ++attempt) {
          double wW = 0.0;
          if (C.g_compute) {
            float acc = 0.f;
            for (int v = v0 + lane; v < v1; v += 32) {
              float w[NV];
              vec_weights(v, w);
              float ls = 0.f;
#pragma unroll
              for (int e = 0; e < NV; ++e) ls += w[e];
              acc += ls;
            }
            wW = static_cast<double>(warp_sum(acc));
          }
          if (lane == 0) C.warp_W[warp] = wW;
          __syncthreads();
          if (tid == 0) {
            double t = 0.0;
            for (int w = 0; w < NW; ++w) t += C.warp_W[w];
            C.pub[pb].W = t;
            C.pub[pb].skip = C.g_compute ? 0 : 1;
          }
          cluster_barrier();  // B
          if (warp == 0) {
            const bool in = lane < static_cast<int>(CS);
            const double Wr = in ? ld_remote_f64(&C.pub[pb].W, static_cast<uint32_t>(lane)) : 0.0;
            const int sk = in ? ld_remote_s32(&C.pub[pb].skip, static_cast<uint32_t>(lane)) : 0;
            double incl = Wr;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const double up = __shfl_up_sync(0xffffffffu, incl, o);
              if (lane >= o) incl += up;
            }
            double excl = __shfl_up_sync(0xffffffffu, incl, 1);
            if (lane == 0) excl = 0.0;
            const double Stot = __shfl_sync(0xffffffffu, incl, 31);
            const double tgt = static_cast<double>(s_u) * Stot;
            const unsigned hit = __ballot_sync(0xffffffffu, in && tgt < incl);
            const unsigned pos_w = __ballot_sync(0xffffffffu, in && Wr > 0.0);
            const int rstar = hit ? (__ffs(hit) - 1) : (pos_w ? 31 - __clz(pos_w) : -1);
            const double before = __shfl_sync(0xffffffffu, excl, rstar < 0 ? 0 : rstar);
            const int skip = warp_or(sk);
            if (lane == 0) {
              C.g_skip = skip;
              C.g_rstar = rstar;
              C.g_S = Stot;
              C.g_target = tgt - before;
            }
          }
          __syncthreads();
          if (C.g_skip) break;           // an earlier position rejected: never used
          if (!(C.g_S > 0.0)) {
            if (resid) {
              // exact arithmetic rules this out (a rejection implies p > q
              // somewhere); draw from p_a instead and count it
              zero_resid = 1;
              resid = false;
              cluster_barrier();         // pub W read everywhere before it is rewritten
              continue;
            }
            break;
          }
          reporter = C.g_rstar;
          if (static_cast<int>(rank) == C.g_rstar) {
            if (tid == 0) {
              const double t = C.g_target;
              double run = 0.0, last_run = 0.0;
              int wstar = -1, wlast = 0;
              for (int w = 0; w < NW; ++w) {
                const double Ww = C.warp_W[w];
                if (Ww > 0.0) { wlast = w; last_run = run; }
                if (wstar < 0 && t < run + Ww) { wstar = w; C.g_target = t - run; }
                run += Ww;
              }
              if (wstar < 0) { wstar = wlast; C.g_target = t - last_run; }
              C.g_found_warp = wstar;
              C.g_y = -1;
            }
            __syncthreads();
            if (warp == C.g_found_warp) {
              // walk the chunk 32 vectors at a time with a warp inclusive scan
              const double t = C.g_target;
              double base = 0.0;
              int found = -1, last_positive = -1;
              for (int vb = v0; vb < v1 && found < 0; vb += 32) {
                const int v = vb + lane;
                float w[NV];
                float ls = 0.f;
                if (v < v1) {
                  vec_weights(v, w);
#pragma unroll
                  for (int e = 0; e < NV; ++e) ls += w[e];
                } else {
#pragma unroll
                  for (int e = 0; e < NV; ++e) w[e] = 0.f;
                }
                float incl = ls;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                  const float up = __shfl_up_sync(0xffffffffu, incl, o);
                  if (lane >= o) incl += up;
                }
                float excl = __shfl_up_sync(0xffffffffu, incl, 1);
                if (lane == 0) excl = 0.f;
                const float step_total = __shfl_sync(0xffffffffu, incl, 31);
                const bool mine = ls > 0.f && t < base + static_cast<double>(incl) &&
                                  !(t < base + static_cast<double>(excl));
                const unsigned hit = __ballot_sync(0xffffffffu, mine);
                int lp = -1;
#pragma unroll
                for (int e = 0; e < NV; ++e) if (w[e] > 0.f) lp = lo + v * NV + e;
                const unsigned anyp = __ballot_sync(0xffffffffu, lp >= 0);
                if (anyp) last_positive = __shfl_sync(0xffffffffu, lp, 31 - __clz(anyp));
                if (hit) {
                  const int hl = __ffs(hit) - 1;
                  int pick = -1;
                  if (lane == hl) {
                    double c = base + static_cast<double>(excl);
                    int lastp = -1;
#pragma unroll
                    for (int e = 0; e < NV; ++e) {
                      if (w[e] > 0.f) lastp = lo + v * NV + e;
                      c += static_cast<double>(w[e]);
                      if (pick < 0 && w[e] > 0.f && t < c) pick = lo + v * NV + e;
                    }
                    if (pick < 0) pick = lastp;
                  }
                  found = __shfl_sync(0xffffffffu, pick, hl);
                }
                base += static_cast<double>(step_total);
              }
              if (found < 0) found = last_positive;
              if (lane == 0) C.g_y = found;
            }
            __syncthreads();
            y = C.g_y;
          }
          break;
        }
        if (static_cast<int>(rank) == reporter && tid == 0) {
          P.ws.mass[slot_t] = C.g_skip ? NAN : static_cast<float>(C.g_S);
          if (zero_resid && !C.g_skip) atomicAdd(P.ws.stats + kStatZeroResidual, 1ull);
          report_item(P, b, kb, pos, y);
        }
      }
    }

    // ---- buffer s is free: stage the item S positions ahead ---------------
    __syncthreads();
    if (tid == 0) stage(s, next_t);
    if (!P.bulk) {
      __syncthreads();
      stage_plain(s);
    }
    __syncthreads();
  }
  cluster_barrier();  // no CTA leaves while others may still read its shared memory
}

// ---------------------------------------------------------------------------
// Packed outputs: offsets = exclusive scan of out_len, then a gather of the
// emitted tokens.  One CTA walks the batch in chunks of its width.
// ---------------------------------------------------------------------------
constexpr int kCompactThreads = 1024;

__global__ void __launch_bounds__(kCompactThreads)
compact_kernel(int B, int k, const int* __restrict__ out_tokens, const int* __restrict__ out_len,
               int* __restrict__ packed, int* __restrict__ offsets) {
  __shared__ int warp_tot[32];
  __shared__ int carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < B; base += kCompactThreads) {
    const int b = base + tid;
    const int len = b < B ? out_len[b] : 0;
    int incl = len;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int up = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += up;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int t = warp_tot[lane];
      int ti = t;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int up = __shfl_up_sync(0xffffffffu, ti, o);
        if (lane >= o) ti += up;
      }
      warp_tot[lane] = ti - t;   // exclusive prefix of the warp totals
    }
    __syncthreads();
    const int off = carry + warp_tot[warp] + incl - len;
    if (b < B) {
      offsets[b] = off;
      const int* src = out_tokens + static_cast<size_t>(b) * (k + 1);
      for (int j = 0; j < len; ++j) packed[off + j] = src[j];
    }
    __syncthreads();
    if (tid == kCompactThreads - 1) carry = off + len;
    __syncthreads();
  }
  if (tid == 0) offsets[B] = carry;
}

// Diagnostics of the last verify launch, widened to double.
// log-sum-exp of z/T = (m c + L) ln 2 with c = log2(e)/T, i.e. m/T + L ln 2.
__global__ void debug_kernel(Workspace ws, int B, int k, int greedy, float inv_T,
                             double* lse_t, double* lse_d, double* accept_prob, double* mass) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  const double ln2 = 0.69314718055994530942;
  if (i < B * (k + 1)) {
    const double m = ws.m_t[i], L = ws.L_t[i];
    if (lse_t) lse_t[i] = greedy ? NAN : m * static_cast<double>(inv_T) + L * ln2;
    if (mass) mass[i] = ws.mass[i];
  }
  if (i < B * k) {
    const double m = ws.m_d[i], L = ws.L_d[i];
    if (lse_d) lse_d[i] = greedy ? NAN : m * static_cast<double>(inv_T) + L * ln2;
    if (accept_prob) accept_prob[i] = ws.alpha[i];
  }
}

__global__ void init_workspace_kernel(Workspace ws, int max_B) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < max_B) {
    ws.done[i] = 0;
    ws.rej_min[i] = kNoReject;
    ws.seq_err[i] = 0;
  }
  if (i < kStatCount) ws.stats[i] = 0ull;
  if (i == 0) { *ws.err_word = 0u; *ws.n_items = 0; *ws.ticket = 0; }
}

}  // namespace

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------

cudaError_t prepare_verify_kernel(int smem_bytes, int cluster) {
  const void* fns[2] = {reinterpret_cast<const void*>(&verify_kernel<2>),
                        reinterpret_cast<const void*>(&verify_kernel<4>)};
  for (const void* f : fns) {
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    if (cluster > 8) {
      e = cudaFuncSetAttribute(f, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

static cudaLaunchConfig_t verify_config(int nclusters, int cluster, int smem_bytes, cudaStream_t s,
                                        cudaLaunchAttribute* attr, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(nclusters) * static_cast<unsigned>(cluster), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cfg;
}

cudaError_t query_max_active_clusters(int cluster, int smem_bytes, int* out) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = verify_config(1, cluster, smem_bytes, nullptr, attr, false);
  return cudaOccupancyMaxActiveClusters(out, reinterpret_cast<const void*>(&verify_kernel<2>), &cfg);
}

cudaError_t launch_verify(const VerifyParams& p, int cluster, int clusters, int smem_bytes, cudaStream_t s) {
  plan_kernel<<<1, kPlanThreads, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = verify_config(clusters, cluster, smem_bytes, s, attr, true);
  if (p.elt == 2) return cudaLaunchKernelEx(&cfg, verify_kernel<2>, p);
  return cudaLaunchKernelEx(&cfg, verify_kernel<4>, p);
}

cudaError_t launch_compact(int B, int k, const int* out_tokens, const int* out_len,
                           int* packed, int* offsets, cudaStream_t s) {
  compact_kernel<<<1, kCompactThreads, 0, s>>>(B, k, out_tokens, out_len, packed, offsets);
  return cudaGetLastError();
}

cudaError_t launch_debug(const Workspace& ws, int B, int k, int greedy, float inv_T, double* lse_t,
                         double* lse_d, double* accept_prob, double* mass, cudaStream_t s) {
  const int n = B * (k + 1);
  debug_kernel<<<(n + 255) / 256, 256, 0, s>>>(ws, B, k, greedy, inv_T, lse_t, lse_d, accept_prob, mass);
  return cudaGetLastError();
}

cudaError_t launch_init_workspace(const Workspace& ws, int max_B, cudaStream_t s) {
  const int n = max_B > kStatCount ? max_B : kStatCount;
  init_workspace_kernel<<<(n + 255) / 256, 256, 0, s>>>(ws, max_B);
  return cudaGetLastError();
}

}  // namespace sv
