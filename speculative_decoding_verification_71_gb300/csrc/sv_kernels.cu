// Speculative-sampling verification kernels for sm_103a.
//
// One thread-block CLUSTER verifies one "item": either a (target row i,
// draft row i) pair of sequence b with i < k_b, or the bonus target row k_b.
// The cluster's CTAs split the vocabulary; each CTA stages its slice of the
// item's row(s) into shared memory once with cp.async.bulk and keeps it there
// for every later pass, so each needed logit crosses HBM exactly once:
//
//   pass 1  slice maximum (and the drafted token's logits)   -> cluster max
//   pass 2  sum of 2^((z - m) c), c = log2(e)/T               -> cluster sum
//   test    alpha = min(1, p(x)/q(x)); accept iff u < alpha
//   pass 3  (rejected pair, or bonus row) weights w = max(0, p - q) or p,
//           per-warp totals -> cluster exclusive scan -> the CTA holding
//           s*S walks its warp chunk to the sampled token
//
// Cross-CTA values move through distributed shared memory between hardware
// cluster barriers.  Items of one sequence run in different clusters; the
// last one to finish (a threadfence + atomic counter, no waiting) writes the
// sequence's outputs.  A rejecting pair first does atomicMin on the
// sequence's first-rejection word and skips its draw when an earlier
// position has already rejected; clusters are numbered position-major so
// that earlier positions usually finish first.
//
// The rule implemented (accept with min(1, p/q), stop at the first
// rejection, resample from max(0, p - q) or draw the bonus token from the
// last target row) is the standard speculative-sampling rule, the reading of
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

// 2^x on the special-function unit (PTX ex2.approx; -inf -> +0, NaN -> NaN).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Non-blocking probe of an mbarrier phase.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile("{\n\t.reg .pred p;\n\t"
               "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(done) : "r"(smem_addr(bar)), "r"(parity) : "memory");
  return done != 0;
}

// Bounded wait on an mbarrier phase.  Returns false if `limit_ns` passed
// before the phase completed (a limit <= 0 only probes, without blocking).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, long long limit_ns) {
  if (limit_ns <= 0) return mbar_test_wait(bar, parity);
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
};

// ---------------------------------------------------------------------------
// Shared control block (first kCtrlBytes of dynamic shared memory).
// Fields read by other CTAs of the cluster are written before a cluster
// barrier and read after it.
// ---------------------------------------------------------------------------

struct Ctrl {
  uint64_t bar[2];        // staging barriers: target slice, draft slice
  // published to the cluster
  float pub_max_t, pub_max_d;
  float pub_zt_x, pub_zd_x;   // logits at the drafted token (owner CTA only)
  float pub_sum_t, pub_sum_d;
  int pub_arg_t;              // greedy: first index of the slice maximum
  int pub_flags;              // bit0 wait timed out, bit1 non-finite seen (greedy), bit2 skipped draw
  double pub_W;               // this CTA's total draw weight
  // CTA-local scratch
  float red_f[32];
  int red_i[32];
  double warp_W[32];
  // values agreed by the whole cluster
  float g_max_t, g_max_d, g_zt_x, g_zd_x, g_L_t, g_L_d;
  int g_arg_t;
  int g_flags;
  int g_accept;
  int g_compute;              // this CTA computes the draw
  int g_found_warp;
  int g_y;
  int g_skip;                 // some CTA skipped the draw (earlier rejection known)
  int g_rstar;                // CTA whose slice holds s*S
  double g_S;                 // total weight of the draw
  double g_target;            // s*S - (mass before this CTA / warp)
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block too large");

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
// (value, index) maximum, ties to the lower index.
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
  }
}

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
  } else {
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
  // leave the per-sequence words ready for the next launch
  ws.done[b] = 0;
  ws.rej_min[b] = kNoReject;
  ws.seq_err[b] = 0;
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
// The verify kernel.
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
  const int cid = static_cast<int>(blockIdx.x / CS);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = P.B, k = P.k;
  const int level = cid / B;
  const int b = cid - level * B;
  const int kb = P.draft_len[b];
  const bool root = (rank == 0 && tid == 0);

  // ---- which item is this cluster? --------------------------------------
  if (kb < 0 || kb > k) {
    if (level == k && root) {
      int* ot = P.out_tokens + static_cast<size_t>(b) * (k + 1);
      for (int j = 0; j <= k; ++j) ot[j] = -1;
      P.out_len[b] = 0;
      // only the sticky word: this sequence has no items, so nothing would
      // clear a per-sequence flag before the next launch
      atomicOr(P.ws.err_word, 1u << 2 /* SV_ERR_BAD_DRAFT_LEN */);
      atomicAdd(P.ws.stats + kStatErrorSeqs, 1ull);
    }
    return;
  }
  int pos;
  bool pair;
  if (level < kb) { pos = level; pair = true; }
  else if (level == k) { pos = kb; pair = false; }
  else {
    // padding position: clear its diagnostics and leave
    if (root) {
      const size_t st = static_cast<size_t>(b) * (k + 1) + level + 1;
      P.ws.m_t[st] = NAN; P.ws.L_t[st] = NAN; P.ws.mass[st] = NAN;
      const size_t sd = static_cast<size_t>(b) * k + level;
      P.ws.m_d[sd] = NAN; P.ws.L_d[sd] = NAN; P.ws.alpha[sd] = NAN;
    }
    return;
  }
  const bool use_draft = pair && !P.greedy;
  int x = -1;
  if (pair) {
    x = P.tokens[static_cast<size_t>(b) * k + pos];
    if (x < 0 || x >= P.V) {
      if (root) {
        mark_error(P, b, 3 /* SV_ERR_BAD_TOKEN */);
        report_item(P, b, kb, pos, -2);
      }
      return;
    }
  }

  // ---- stage this CTA's slice of the row(s) ------------------------------
  const int lo = static_cast<int>(rank) * P.slice;
  const int hi = min(P.V, lo + P.slice);
  const int n = max(0, hi - lo);
  const int nvec = (n + NV - 1) / NV;
  const int row_bytes_pad = ((P.slice * ELT + 127) / 128) * 128;
  unsigned char* bufT = smem + kCtrlBytes;
  unsigned char* bufD = bufT + row_bytes_pad;
  const unsigned char* gT = static_cast<const unsigned char*>(P.target) +
      ((static_cast<size_t>(b) * (k + 1) + pos) * P.V + lo) * ELT;
  const unsigned char* gD = use_draft ? static_cast<const unsigned char*>(P.draft) +
      ((static_cast<size_t>(b) * k + pos) * P.V + lo) * ELT : nullptr;

  int my_flags = 0;
  if (P.bulk) {
    if (tid == 0) {
      mbar_init(&C.bar[0], 1);
      mbar_init(&C.bar[1], 1);
      mbar_fence_init();
    }
    __syncthreads();
    if (tid == 0 && n > 0) {
      const uint32_t bytes = static_cast<uint32_t>(n) * ELT;
      constexpr uint32_t kChunk = 32768;
      mbar_expect_tx(&C.bar[0], bytes);
      for (uint32_t o = 0; o < bytes; o += kChunk)
        bulk_load(bufT + o, gT + o, min(kChunk, bytes - o), &C.bar[0]);
      if (use_draft) {
        mbar_expect_tx(&C.bar[1], bytes);
        for (uint32_t o = 0; o < bytes; o += kChunk)
          bulk_load(bufD + o, gD + o, min(kChunk, bytes - o), &C.bar[1]);
      }
    }
  } else {
    // plain loads (unaligned rows); pad the last vector with -inf
    const int npad = nvec * NV;
    for (int e = tid; e < npad; e += kThreads) {
      float vt = -INFINITY, vd = -INFINITY;
      if (e < n) {
        vt = V::scalar(gT, e);
        if (use_draft) vd = V::scalar(gD, e);
      }
      if (ELT == 2) {
        reinterpret_cast<uint16_t*>(bufT)[e] = static_cast<uint16_t>(__float_as_uint(vt) >> 16);
        if (use_draft) reinterpret_cast<uint16_t*>(bufD)[e] = static_cast<uint16_t>(__float_as_uint(vd) >> 16);
      } else {
        reinterpret_cast<float*>(bufT)[e] = vt;
        if (use_draft) reinterpret_cast<float*>(bufD)[e] = vd;
      }
    }
    __syncthreads();
  }

  // vectors [v0, v1) of this CTA's slice belong to this warp
  const int vpw = (nvec + NW - 1) / NW;
  const int v0 = warp * vpw;
  const int v1 = min(nvec, v0 + vpw);

  // ---- pass 1: maxima (+ argmax when greedy) ------------------------------
  float mx_t = -INFINITY, mx_d = -INFINITY;
  int arg_t = 0x7fffffff;
  bool bad = false;
  if (P.bulk && n > 0) {
    if (!mbar_wait_bounded(&C.bar[0], 0, P.wait_limit_ns)) {
      my_flags |= 1;
      mbar_wait_bounded(&C.bar[0], 0, kDrainLimitNs);
    }
    if (use_draft && !mbar_wait_bounded(&C.bar[1], 0, P.wait_limit_ns)) {
      my_flags |= 1;
      mbar_wait_bounded(&C.bar[1], 0, kDrainLimitNs);
    }
  }
  my_flags = __syncthreads_or(my_flags);
  if (P.greedy) {
    for (int v = v0 + lane; v < v1; v += 32) {
      float z[NV];
      V::load(bufT + v * 16, z);
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        bad |= (z[j] != z[j]) || (z[j] == INFINITY);
        if (z[j] > mx_t) { mx_t = z[j]; arg_t = lo + v * NV + j; }
      }
    }
    warp_argmax(mx_t, arg_t);
    bad = __any_sync(0xffffffffu, bad);
  } else {
    for (int v = v0 + lane; v < v1; v += 32) {
      float z[NV];
      V::load(bufT + v * 16, z);
#pragma unroll
      for (int j = 0; j < NV; ++j) mx_t = fmaxf(mx_t, z[j]);
      if (use_draft) {
        V::load(bufD + v * 16, z);
#pragma unroll
        for (int j = 0; j < NV; ++j) mx_d = fmaxf(mx_d, z[j]);
      }
    }
    mx_t = warp_max(mx_t);
    mx_d = warp_max(mx_d);
  }
  if (lane == 0) { C.red_f[warp] = mx_t; C.red_f[NW + warp] = mx_d; C.red_i[warp] = arg_t; C.red_i[NW + warp] = bad; }
  __syncthreads();
  if (tid == 0) {
    float mt = -INFINITY, md = -INFINITY;
    int at = 0x7fffffff, anybad = 0;
    for (int w = 0; w < NW; ++w) {
      const float vt = C.red_f[w];
      if (vt > mt || (vt == mt && C.red_i[w] < at)) { mt = vt; at = C.red_i[w]; }
      md = fmaxf(md, C.red_f[NW + w]);
      anybad |= C.red_i[NW + w];
    }
    C.pub_max_t = mt;
    C.pub_max_d = md;
    C.pub_arg_t = at;
    // the drafted token's logits, from the CTA whose slice holds x
    C.pub_zt_x = NAN;
    C.pub_zd_x = NAN;
    if (pair && x >= lo && x < hi) {
      C.pub_zt_x = V::scalar(bufT, x - lo);
      if (use_draft) C.pub_zd_x = V::scalar(bufD, x - lo);
    }
    C.pub_flags = my_flags | (anybad ? 2 : 0);
  }
  cluster_barrier();  // #1
  if (tid == 0) {
    float mt = -INFINITY, md = -INFINITY;
    int at = 0x7fffffff, fl = 0;
    for (uint32_t r = 0; r < CS; ++r) {
      const float vt = ld_remote_f32(&C.pub_max_t, r);
      const int it = ld_remote_s32(&C.pub_arg_t, r);
      if (vt > mt || (vt == mt && it < at)) { mt = vt; at = it; }
      md = fmaxf(md, ld_remote_f32(&C.pub_max_d, r));
      fl |= ld_remote_s32(&C.pub_flags, r);
    }
    C.g_max_t = mt;
    C.g_max_d = md;
    C.g_arg_t = at;
    C.g_flags = fl;
    if (pair) {
      const uint32_t owner = static_cast<uint32_t>(x / P.slice);
      C.g_zt_x = ld_remote_f32(&C.pub_zt_x, owner);
      C.g_zd_x = use_draft ? ld_remote_f32(&C.pub_zd_x, owner) : 0.f;
    }
  }
  __syncthreads();

  const size_t slot_t = static_cast<size_t>(b) * (k + 1) + pos;
  const size_t slot_d = static_cast<size_t>(b) * k + pos;

  // ---- greedy (T == 0): accept iff x is the first argmax ------------------
  if (P.greedy) {
    if (root) {
      if (C.g_flags & 1) mark_error(P, b, 5 /* SV_ERR_TIMEOUT */);
      if ((C.g_flags & 2) || !(C.g_max_t > -INFINITY)) mark_error(P, b, 4 /* SV_ERR_NONFINITE */);
      P.ws.m_t[slot_t] = C.g_max_t; P.ws.L_t[slot_t] = NAN; P.ws.mass[slot_t] = NAN;
      int y = C.g_arg_t;
      if (pair) {
        const bool acc = (x == C.g_arg_t);
        P.ws.alpha[slot_d] = acc ? 1.f : 0.f;
        P.ws.m_d[slot_d] = NAN; P.ws.L_d[slot_d] = NAN;
        if (!acc) atomicMin(P.ws.rej_min + b, pos);
      }
      report_item(P, b, kb, pos, y);
    }
    cluster_barrier();  // final: no CTA leaves while others may read its shared memory
    return;
  }

  // ---- pass 2: sums of 2^((z - m) c) ---------------------------------------
  const float c2 = P.c2;
  const float mt = C.g_max_t, md = C.g_max_d;
  {
    float st = 0.f, sd = 0.f;
    for (int v = v0 + lane; v < v1; v += 32) {
      float z[NV];
      V::load(bufT + v * 16, z);
#pragma unroll
      for (int j = 0; j < NV; ++j) st += fast_exp2((z[j] - mt) * c2);
      if (use_draft) {
        V::load(bufD + v * 16, z);
#pragma unroll
        for (int j = 0; j < NV; ++j) sd += fast_exp2((z[j] - md) * c2);
      }
    }
    st = warp_sum(st);
    sd = warp_sum(sd);
    if (lane == 0) { C.red_f[warp] = st; C.red_f[NW + warp] = sd; }
    __syncthreads();
    if (tid == 0) {
      float a = 0.f, d = 0.f;
      for (int w = 0; w < NW; ++w) { a += C.red_f[w]; d += C.red_f[NW + w]; }
      C.pub_sum_t = a;
      C.pub_sum_d = d;
    }
  }
  cluster_barrier();  // #2
  if (tid == 0) {
    float st = 0.f, sd = 0.f;
    for (uint32_t r = 0; r < CS; ++r) {
      st += ld_remote_f32(&C.pub_sum_t, r);
      sd += ld_remote_f32(&C.pub_sum_d, r);
    }
    const float Lt = log2f(st);
    const float Ld = use_draft ? log2f(sd) : 0.f;
    C.g_L_t = Lt;
    C.g_L_d = Ld;
    bool nonfinite = !(isfinite(mt) && isfinite(st));
    if (use_draft) nonfinite |= !(isfinite(md) && isfinite(sd));
    int fl = C.g_flags;
    if (nonfinite) fl |= 2;
    C.g_flags = fl;
    // acceptance test
    int accept = 0;
    float alpha = NAN;
    if (pair) {
      const float zt = C.g_zt_x, zd = C.g_zd_x;
      if (zt == -INFINITY) alpha = 0.f;               // p(x) = 0
      else if (zd == -INFINITY) alpha = 1.f;          // q(x) = 0 < p(x)
      else {
        const float log2r = ((zt - mt) * c2 - Lt) - ((zd - md) * c2 - Ld);
        alpha = log2r >= 0.f ? 1.f : exp2f(log2r);
      }
      const float u = P.uniforms[static_cast<size_t>(b) * (k + 1) + pos];
      accept = (u < alpha) ? 1 : 0;
    }
    C.g_accept = accept;
    if (rank == 0) {
      P.ws.m_t[slot_t] = mt; P.ws.L_t[slot_t] = Lt; P.ws.mass[slot_t] = NAN;
      if (pair) { P.ws.m_d[slot_d] = md; P.ws.L_d[slot_d] = Ld; P.ws.alpha[slot_d] = alpha; }
    }
    // does this CTA compute a draw?
    int compute = 0;
    if (!fl) {
      if (pair && !accept) compute = atomicMin(P.ws.rej_min + b, pos) >= pos;
      else if (!pair) compute = __ldcg(P.ws.rej_min + b) == kNoReject;
    }
    C.g_compute = compute;
    C.pub_flags = compute ? 0 : 4;
  }
  __syncthreads();

  const int flags = C.g_flags;
  if (flags) {
    if (root) {
      if (flags & 1) mark_error(P, b, 5 /* SV_ERR_TIMEOUT */);
      if (flags & 2) mark_error(P, b, 4 /* SV_ERR_NONFINITE */);
      report_item(P, b, kb, pos, -2);
    }
    cluster_barrier();  // final
    return;
  }
  if (pair && C.g_accept) {
    if (root) report_item(P, b, kb, pos, -2);
    cluster_barrier();  // final
    return;
  }

  // ---- pass 3: the draw (rejected pair: max(0, p - q); bonus: p) ----------
  const float Lt = C.g_L_t, Ld = C.g_L_d;
  const float s = P.uniforms[static_cast<size_t>(b) * (k + 1) + k];
  bool resid = pair;
  // weights of the logits of vector v
  auto vec_weights = [&](int v, float (&w)[NV]) {
    float zt[NV], zd[NV];
    V::load(bufT + v * 16, zt);
    if (resid) V::load(bufD + v * 16, zd);
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const float p = fast_exp2((zt[j] - mt) * c2 - Lt);
      w[j] = resid ? fmaxf(p - fast_exp2((zd[j] - md) * c2 - Ld), 0.f) : p;
    }
  };

  int zero_resid = 0;
  int y = -2;
  int reporter = 0;
  for (int attempt = 0; attempt < 2; ++attempt) {
    // totals: per warp chunk, then per CTA
    double wW = 0.0;
    if (C.g_compute) {
      float acc = 0.f;
      for (int v = v0 + lane; v < v1; v += 32) {
        float w[NV];
        vec_weights(v, w);
        float ls = 0.f;
#pragma unroll
        for (int j = 0; j < NV; ++j) ls += w[j];
        acc += ls;
      }
      wW = static_cast<double>(warp_sum(acc));
    }
    if (lane == 0) C.warp_W[warp] = wW;
    __syncthreads();
    if (tid == 0) {
      double t = 0.0;
      for (int w = 0; w < NW; ++w) t += C.warp_W[w];
      C.pub_W = t;
    }
    cluster_barrier();  // #3
    // every CTA derives the same cluster-wide picture, in rank order
    if (tid == 0) {
      int skip = 0;
      double S = 0.0;
      for (uint32_t r = 0; r < CS; ++r) {
        skip |= ld_remote_s32(&C.pub_flags, r) & 4;
        S += ld_remote_f64(&C.pub_W, r);
      }
      int rstar = -1;
      double before = 0.0;
      const double tgt = static_cast<double>(s) * S;
      if (!skip && S > 0.0) {
        double run = 0.0, last_before = 0.0;
        int last_pos = 0;
        for (uint32_t r = 0; r < CS; ++r) {
          const double Wr = ld_remote_f64(&C.pub_W, r);
          if (Wr > 0.0) { last_pos = static_cast<int>(r); last_before = run; }
          if (rstar < 0 && tgt < run + Wr) { rstar = static_cast<int>(r); before = run; }
          run += Wr;
        }
        if (rstar < 0) { rstar = last_pos; before = last_before; }
      }
      C.g_skip = skip;
      C.g_rstar = rstar;
      C.g_S = S;
      C.g_target = tgt - before;
    }
    __syncthreads();
    if (C.g_skip) break;             // an earlier position rejected: this draw is never used
    if (!(C.g_S > 0.0)) {
      if (resid) {
        // exact arithmetic rules this out (a rejection implies p > q
        // somewhere); draw from p_a instead and count it
        zero_resid = 1;
        resid = false;
        cluster_barrier();           // everyone has read pub_W before it is rewritten
        continue;
      }
      break;
    }
    reporter = C.g_rstar;
    if (static_cast<int>(rank) == C.g_rstar) {
      // the warp whose chunk holds the target
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
            for (int j = 0; j < NV; ++j) ls += w[j];
          } else {
#pragma unroll
            for (int j = 0; j < NV; ++j) w[j] = 0.f;
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
          for (int j = 0; j < NV; ++j) if (w[j] > 0.f) lp = lo + v * NV + j;
          const unsigned anyp = __ballot_sync(0xffffffffu, lp >= 0);
          if (anyp) last_positive = __shfl_sync(0xffffffffu, lp, 31 - __clz(anyp));
          if (hit) {
            const int hl = __ffs(hit) - 1;
            int pick = -1;
            if (lane == hl) {
              double c = base + static_cast<double>(excl);
              int lastp = -1;
#pragma unroll
              for (int j = 0; j < NV; ++j) {
                if (w[j] > 0.f) lastp = lo + v * NV + j;
                c += static_cast<double>(w[j]);
                if (pick < 0 && w[j] > 0.f && t < c) pick = lo + v * NV + j;
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
  cluster_barrier();  // final: no CTA leaves while others may read its shared memory
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
      int t = warp_tot[lane];
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
  if (i == 0) *ws.err_word = 0u;
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
                                        cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(nclusters) * static_cast<unsigned>(cluster), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

cudaError_t query_max_active_clusters(int cluster, int smem_bytes, int* out) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = verify_config(1, cluster, smem_bytes, nullptr, attr);
  return cudaOccupancyMaxActiveClusters(out, reinterpret_cast<const void*>(&verify_kernel<2>), &cfg);
}

cudaError_t launch_verify(const VerifyParams& p, int cluster, int smem_bytes, cudaStream_t s) {
  const int nclusters = p.B * (p.k + 1);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = verify_config(nclusters, cluster, smem_bytes, s, attr);
  if (p.elt == 2) return cudaLaunchKernelEx(&cfg, verify_kernel<2>, p);
  return cudaLaunchKernelEx(&cfg, verify_kernel<4>, p);
}

cudaError_t launch_compact(int B, int k, const int* out_tokens, const int* out_len,
                           int* packed, int* offsets, cudaStream_t s) {
  compact_kernel<<<1, kCompactThreads, 0, s>>>(B, k, out_tokens, out_len, packed, offsets);
  return cudaGetLastError();
}

cudaError_t launch_debug(const Workspace& ws, int B, int k, const int* /*unused*/, int greedy,
                         float inv_T, double* lse_t, double* lse_d, double* accept_prob,
                         double* mass, cudaStream_t s) {
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
