// Speculative-sampling verification kernels for sm_103a.
//
// verify_kernel is persistent and warp-specialised.  Each CTA verifies whole
// sequences, one after another, taking them from a work list ordered longest
// first (plan_kernel) with an atomic ticket:
//
//   producer warp   streams the sequence's rows in position order (target 0,
//                   draft 0, target 1, draft 1, ..., target k_b) through a
//                   ring of 16 KB shared-memory slots with cp.async.bulk, and
//                   runs ahead into the next sequence while the consumers
//                   are busy, so HBM reads never wait on arithmetic;
//   8 consumer warps  fold every 16 KB chunk into per-warp running maxima and
//                   sums of 2^(z c - fl(m c)), c = log2(e)/T (one ex2 per
//                   logit), pick up the drafted token's logit, and at each
//                   row end combine the warps into the row's log-sum-exp.
//
// Because one CTA sees the positions of a sequence in order, the first
// rejection is known exactly:
//   * after draft row i: alpha_i = min(1, p_i(x_i) / q_i(x_i)); accept iff
//     u_i < alpha_i (every position's alpha is kept for diagnostics);
//   * at the first rejection a: the pair (target a, draft a), read moments
//     ago and still in L2, is read again to get exact per-segment masses of
//     max(0, p - q); a warp scan finds the segment holding s*S and one warp
//     walks that segment to the drawn token;
//   * if every draft is accepted, the bonus row needs no second read at
//     all: its per-segment sums were kept while streaming, so only the one
//     segment holding s*S is read again.
// Every needed logit crosses HBM once; the only extra reads are the rejected
// pair (from L2) and one segment.  The CTA writes the sequence's outputs
// itself: no atomics on the data path and no waiting on other CTAs.
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

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_addr(bar)) : "memory");
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
  asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

// The same with an L2 eviction-priority policy (for rows never read again).
__device__ __forceinline__ void bulk_load_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                               uint64_t policy) {
  asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
               :: "r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy) : "memory");
}

__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Programmatic dependent launch: wait for the preceding grid's results / let
// the dependent grid start its prologue.
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

// Packed pairs of fp32 (Blackwell f32x2 arithmetic: two lanes, one
// instruction, each lane rounded exactly as the scalar operation).
typedef unsigned long long f2;
__device__ __forceinline__ f2 pack2(float a, float b) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void unpack2(f2 r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
  f2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ f2 add2(f2 a, f2 b) {
  f2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f2 sub2(f2 a, f2 b) {
  f2 r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f2 exp2_2(f2 t) {
  float a, b;
  unpack2(t, a, b);
  return pack2(fast_exp2(a), fast_exp2(b));
}

// Bounded wait on an mbarrier phase.  Returns false if `limit_ns` passed
// before the phase completed.  A limit <= 0 is the error-path test hook: it
// always reports expiry (the caller then drains with a 1 s wait).
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
  __device__ __forceinline__ static void unpack(const uint4 w, float (&v)[8]) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[2 * j] = __uint_as_float(ws[j] << 16);
      v[2 * j + 1] = __uint_as_float(ws[j] & 0xffff0000u);
    }
  }
  __device__ __forceinline__ static float scalar(const void* base, long long idx) {
    const unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(base) + idx);
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
  }
  __device__ __forceinline__ static void store_scalar(unsigned char* base, int idx, float v) {
    reinterpret_cast<uint16_t*>(base)[idx] = static_cast<uint16_t>(__float_as_uint(v) >> 16);
  }
  __device__ __forceinline__ static uint4 neg_inf() { return make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u); }
  // the four fp32 pairs of a vector (element order within a pair: low, high)
  __device__ __forceinline__ static void pairs(const uint4 w, f2 (&z)[4]) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) z[i] = pack2(__uint_as_float(ws[i] << 16), __uint_as_float(ws[i] & 0xffff0000u));
  }
  // packed maximum of two bf16 pairs (NaN loses to a number, as with fmaxf)
  __device__ __forceinline__ static uint32_t max2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
  }
  template <int N>
  __device__ __forceinline__ static float vmax(const uint4 (&r)[N]) {
    uint32_t m[4] = {r[0].x, r[0].y, r[0].z, r[0].w};
#pragma unroll
    for (int j = 1; j < N; ++j) {
      m[0] = max2(m[0], r[j].x); m[1] = max2(m[1], r[j].y);
      m[2] = max2(m[2], r[j].z); m[3] = max2(m[3], r[j].w);
    }
    const uint32_t w = max2(max2(m[0], m[1]), max2(m[2], m[3]));
    return fmaxf(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
};
template <> struct Vec<4> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void unpack(const uint4 w, float (&v)[4]) {
    v[0] = __uint_as_float(w.x); v[1] = __uint_as_float(w.y);
    v[2] = __uint_as_float(w.z); v[3] = __uint_as_float(w.w);
  }
  __device__ __forceinline__ static float scalar(const void* base, long long idx) {
    return __ldg(reinterpret_cast<const float*>(base) + idx);
  }
  __device__ __forceinline__ static void store_scalar(unsigned char* base, int idx, float v) {
    reinterpret_cast<float*>(base)[idx] = v;
  }
  __device__ __forceinline__ static uint4 neg_inf() { return make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u); }
  __device__ __forceinline__ static void pairs(const uint4 w, f2 (&z)[2]) {
    z[0] = pack2(__uint_as_float(w.x), __uint_as_float(w.y));
    z[1] = pack2(__uint_as_float(w.z), __uint_as_float(w.w));
  }
  template <int N>
  __device__ __forceinline__ static float vmax(const uint4 (&r)[N]) {
    float m[4] = {__uint_as_float(r[0].x), __uint_as_float(r[0].y), __uint_as_float(r[0].z), __uint_as_float(r[0].w)};
#pragma unroll
    for (int j = 1; j < N; ++j) {
      m[0] = fmaxf(m[0], __uint_as_float(r[j].x)); m[1] = fmaxf(m[1], __uint_as_float(r[j].y));
      m[2] = fmaxf(m[2], __uint_as_float(r[j].z)); m[3] = fmaxf(m[3], __uint_as_float(r[j].w));
    }
    return fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
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
__device__ __forceinline__ double warp_incl_scan(double v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double up = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += up;
  }
  return v;
}
__device__ __forceinline__ float warp_incl_scan(float v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float up = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += up;
  }
  return v;
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

// ---------------------------------------------------------------------------
// Shared control block
// ---------------------------------------------------------------------------

// What a staging slot holds.
//   kind 0 / 1: chunk `chunk` of the target / draft row at position pos;
//   kind 2:     chunk `chunk` of the re-read of the pair at pos for its draw:
//               the first half of the slot holds target logits, the second
//               half the draft logits of the same vocabulary range; x holds
//               the draw mode (1: residual max(0, p - q), 2: p alone) and
//               K0, L0, K1, L1 the pair's normalisers;
//   kind -1:    no more work.
struct Desc {
  int b, kb, pos, kind;
  int chunk, nchunks, x, rec;  // x: drafted token at pos (rows of pairs, else -1); rec: sequence record
  float u, s;                  // accept uniform at pos, sampling uniform of b
  float K0, L0, K1, L1;
};

// A finished row, published by the consumer warps for the control warp.
struct RowBuf {
  Desc d;
  float wK[kConsumerWarps], wS[kConsumerWarps], wM[kConsumerWarps];
  int wArg[kConsumerWarps], wBad[kConsumerWarps];
  float zx;                                  // logit of the drafted token
  float segK[kMaxChunks * kConsumerWarps];   // bonus rows: per-segment fl(m c)
  float segS[kMaxChunks * kConsumerWarps];   // bonus rows: per-segment sum
};

// One sequence in flight (control warp only).  Its stream and its draw can
// finish in either order; the outputs are written when both are done.
struct SeqRec {
  int b, kb, a, err, y, zero_resid;
  int pending;                 // events left before the outputs can be written
  float s;                     // sampling uniform
};

// A re-read request as the control warp remembers it.
struct DrawReq {
  int b, pos, rec, mode;
  float Kt, Lt, Kd, Ld;
};

constexpr int kRecs = 8;       // sequence records (ring)
constexpr int kReqs = 8;       // re-read requests (ring)
constexpr int kRowBufs = 4;    // row buffers (ring)
constexpr int kHalfBytes = kChunkBytes / 2;                          // one row's part of a draw chunk
constexpr int kDrawVecsPerWarp = kHalfBytes / 16 / kConsumerWarps;   // 128
constexpr int kDrawVecsPerLane = kDrawVecsPerWarp / 32;              // 4
constexpr int kMaxDrawSegs = 2 * kMaxChunks * kConsumerWarps;

enum : int { kErrBadToken = 1 << 3, kErrNonfinite = 1 << 4, kErrTimeout = 1 << 5 };

struct Ctrl {
  uint64_t full[kMaxStages];        // slot filled (producer -> consumers)
  uint64_t empty[kMaxStages];       // slot released (one arrival per consumer warp)
  uint64_t row_ready[kRowBufs];     // row published (one arrival per consumer warp)
  uint64_t row_free[kRowBufs];      // row consumed by the control warp
  uint64_t draw_ready[2];           // draw masses complete (one arrival per consumer warp)
  uint64_t draw_free[2];            // draw masses consumed by the control warp
  Desc desc[kMaxStages];
  RowBuf rows[kRowBufs];
  double rmass[2][kMaxDrawSegs];    // per-segment weights of a re-read draw
  int draw_err[2];
  // re-read requests: the control warp pushes, the producer pops
  DrawReq req[kReqs];
  volatile int req_head, req_tail;
  volatile int seqs_finished;       // sequences whose outputs are written
  // control warp state
  SeqRec rec[kRecs];
  DrawReq ctl_req[kReqs];           // every pushed request, by push order, until its draw is done
  int pushed;                       // requests pushed so far
  float pairK, pairL, pairZx;       // target row of the current pair
  double bmass[kMaxChunks * kConsumerWarps];
};

constexpr int kCtrlBytes = ((static_cast<int>(sizeof(Ctrl)) + 1023) / 1024) * 1024;

// ---------------------------------------------------------------------------
// plan_kernel: the work list (valid sequences, longest first) and resets.
// ---------------------------------------------------------------------------
constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const VerifyParams P) {
  grid_dependents_launch();   // the verify grid may start its prologue now
  __shared__ int warp_cnt[32];
  __shared__ int base;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = P.B, k = P.k;
  const Workspace& ws = P.ws;
  for (int b = tid; b < B; b += kPlanThreads) {
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
  // counting sort by k_b, largest first, stable in b
  for (int L = k; L >= 0; --L) {
    for (int b0 = 0; b0 < B; b0 += kPlanThreads) {
      const int b = b0 + tid;
      const int kb = b < B ? P.draft_len[b] : -1;
      const bool take = (kb == L);
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
      if (take) ws.seqs[base + warp_cnt[warp] + __popc(m & ((1u << lane) - 1u))] = make_int2(b, kb);
      __syncthreads();
      if (tid == kPlanThreads - 1) base += warp_cnt[31] + __popc(m);
      __syncthreads();
    }
  }
  if (tid == 0) *ws.n_seqs = base;
}

// ---------------------------------------------------------------------------
// verify_kernel
// ---------------------------------------------------------------------------

template <int ELT>
struct Verifier {
  using V = Vec<ELT>;
  static constexpr int NV = V::N;                          // logits per vector
  static constexpr int kSegElems = kVecsPerWarp * NV;      // logits per stream segment (chunk, warp)

  const VerifyParams& P;
  Ctrl& C;
  unsigned char* ring;
  const int lane, warp;
  const long long row_bytes;    // V * ELT
  const int nchunks;            // stream chunks per row
  const int ndraw;              // draw chunks per row
  const int nvec_row;           // 16-byte vectors per row (last one padded)

  __device__ Verifier(const VerifyParams& p, Ctrl& c, unsigned char* r, int ln, int wp)
      : P(p), C(c), ring(r), lane(ln), warp(wp),
        row_bytes(static_cast<long long>(p.V) * ELT),
        nchunks(static_cast<int>((static_cast<long long>(p.V) * ELT + kChunkBytes - 1) / kChunkBytes)),
        ndraw(static_cast<int>((static_cast<long long>(p.V) * ELT + kHalfBytes - 1) / kHalfBytes)),
        nvec_row(static_cast<int>((static_cast<long long>(p.V) * ELT + 15) / 16)) {}

  __device__ const unsigned char* row_ptr(int b, int pos, int kind) const {
    if (kind == 0)
      return static_cast<const unsigned char*>(P.target) +
             (static_cast<size_t>(b) * (P.k + 1) + pos) * static_cast<size_t>(row_bytes);
    return static_cast<const unsigned char*>(P.draft) +
           (static_cast<size_t>(b) * P.k + pos) * static_cast<size_t>(row_bytes);
  }

  // Vector v of a row read straight from global memory, -inf beyond V.
  __device__ uint4 load_global_raw(const unsigned char* row, int v) const {
    if (v >= nvec_row) return V::neg_inf();
    if (P.bulk) return __ldg(reinterpret_cast<const uint4*>(row) + v);
    unsigned char buf[16];
#pragma unroll
    for (int e = 0; e < NV; ++e) {
      const int x = v * NV + e;
      V::store_scalar(buf, e, x < P.V ? V::scalar(row, x) : -INFINITY);
    }
    return *reinterpret_cast<const uint4*>(buf);
  }

  // Bounded wait by lane 0 for the whole warp; false (and the error word
  // set) if nothing happened for 1 s.
  __device__ bool warp_wait(uint64_t* bar, uint32_t parity) const {
    int ok = 1;
    if (lane == 0) ok = mbar_wait_bounded(bar, parity, kDrainLimitNs) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok && lane == 0) atomicOr(P.ws.err_word, 1u << 5 /* SV_ERR_TIMEOUT */);
    __syncwarp();
    return ok != 0;
  }

  // ======================= producer ==========================================

  // Copy `bytes` of a row starting at byte `off` into dst (bulk or plain).
  __device__ void fill(unsigned char* dst, const unsigned char* src, long long off, int bytes,
                       uint64_t* bar, bool hint, uint64_t policy) {
    if (P.bulk) {
      if (lane == 0) {
        if (hint) bulk_load_hint(dst, src + off, static_cast<uint32_t>(bytes), bar, policy);
        else bulk_load(dst, src + off, static_cast<uint32_t>(bytes), bar);
      }
    } else {
      // plain loads (rows not 16-byte aligned); pad the last vector with -inf
      const int e0 = static_cast<int>(off / ELT);
      const int n = (bytes + ELT - 1) / ELT;
      const int npad = ((n + NV - 1) / NV) * NV;
      for (int e = lane; e < npad; e += 32) {
        const int xg = e0 + e;
        V::store_scalar(dst, e, xg < P.V ? V::scalar(src, xg) : -INFINITY);
      }
    }
  }

  __device__ bool acquire_slot(int q) {
    const int S = P.stages;
    return warp_wait(&C.empty[q % S], ((q / S) & 1) ^ 1);
  }

  // Issue the draw chunks of every queued re-read request.
  __device__ bool service_requests(int& q) {
    const int S = P.stages;
    while (true) {
      int head = 0, tail = 0;
      if (lane == 0) { head = C.req_head; tail = C.req_tail; }
      head = __shfl_sync(0xffffffffu, head, 0);
      tail = __shfl_sync(0xffffffffu, tail, 0);
      if (head == tail) return true;
      const DrawReq r = C.req[head % kReqs];
      __syncwarp();
      if (lane == 0) { __threadfence_block(); C.req_head = head + 1; }
      const unsigned char* srcT = row_ptr(r.b, r.pos, 0);
      const unsigned char* srcD = row_ptr(r.b, r.pos, 1);
      for (int c = 0; c < ndraw; ++c) {
        if (!acquire_slot(q)) return false;
        const int slot = q % S;
        const long long off = static_cast<long long>(c) * kHalfBytes;
        const long long rem = row_bytes - off;
        const int bytes = static_cast<int>(rem < kHalfBytes ? rem : kHalfBytes);
        unsigned char* dst = ring + static_cast<size_t>(slot) * kChunkBytes;
        if (lane == 0) {
          Desc& d = C.desc[slot];
          d.b = r.b; d.kb = 0; d.pos = r.pos; d.kind = 2;
          d.chunk = c; d.nchunks = ndraw; d.x = r.mode; d.rec = r.rec;
          d.u = 0.f; d.s = 0.f;
          d.K0 = r.Kt; d.L0 = r.Lt; d.K1 = r.Kd; d.L1 = r.Ld;
          if (P.bulk) mbar_expect_tx(&C.full[slot], static_cast<uint32_t>(r.mode == 1 ? 2 * bytes : bytes));
        }
        fill(dst, srcT, off, bytes, &C.full[slot], false, 0);
        if (r.mode == 1) fill(dst + kHalfBytes, srcD, off, bytes, &C.full[slot], false, 0);
        if (!P.bulk) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&C.full[slot]);
        }
        ++q;
      }
    }
  }

  __device__ void produce() {
    const int S = P.stages;
    const int k = P.k;
    const int n_seqs = __ldcg(P.ws.n_seqs);
    const uint64_t evict_first = evict_first_policy();
    int q = 0, streamed = 0;
    // the next sequence's work-list entry, tokens and uniforms are fetched one
    // sequence ahead so that a sequence start never waits on global memory
    int t = 0;
    if (lane == 0) t = atomicAdd(P.ws.ticket, 1);
    t = __shfl_sync(0xffffffffu, t, 0);
    int2 sq = make_int2(-1, 0);
    int xj = -1;
    float uj = 0.f;
    auto fetch = [&](int tt, int2& s_, int& x_, float& u_) {
      s_ = make_int2(-1, 0);
      x_ = -1;
      u_ = 0.f;
      if (tt < n_seqs) {
        s_ = __ldcg(P.ws.seqs + tt);
        x_ = lane < s_.y ? __ldg(P.tokens + static_cast<size_t>(s_.x) * k + lane) : -1;
        u_ = (!P.greedy && lane <= k) ? __ldg(P.uniforms + static_cast<size_t>(s_.x) * (k + 1) + lane) : 0.f;
      }
    };
    fetch(t, sq, xj, uj);
    bool ok = true;
    while (ok && t < n_seqs) {
      const int b = sq.x, kb = sq.y;
      const int rec = streamed % kRecs;
      // the next ticket is taken when this sequence's last row starts: late
      // enough that sequences keep going to whichever CTA frees up first
      // (longest first), early enough to hide the fetch behind that row
      int t_next = 0;
      int2 sq_next = make_int2(-1, 0);
      int xj_next = -1;
      float uj_next = 0.f;
      bool fetched = false;
      const float s_samp = __shfl_sync(0xffffffffu, uj, k);
      const int nrows = P.greedy ? kb + 1 : 2 * kb + 1;
      for (int r = 0; r < nrows && ok; ++r) {
        int pos, kind;
        if (P.greedy) { pos = r; kind = 0; }
        else if (r < 2 * kb) { pos = r >> 1; kind = r & 1; }
        else { pos = kb; kind = 0; }
        const int x = __shfl_sync(0xffffffffu, xj, pos < kb ? pos : 0);
        const float u = __shfl_sync(0xffffffffu, uj, pos < kb ? pos : 0);
        const unsigned char* src = row_ptr(b, pos, kind);
        for (int c = 0; c < nchunks && ok; ++c) {
          if (!(ok = acquire_slot(q))) break;
          const int slot = q % S;
          const long long off = static_cast<long long>(c) * kChunkBytes;
          const long long rem = row_bytes - off;
          const int bytes = static_cast<int>(rem < kChunkBytes ? rem : kChunkBytes);
          if (lane == 0) {
            Desc& d = C.desc[slot];
            d.b = b; d.kb = kb; d.pos = pos; d.kind = kind;
            d.chunk = c; d.nchunks = nchunks;
            d.x = pos < kb ? x : -1; d.rec = rec;
            d.u = u; d.s = s_samp;
            if (P.bulk) mbar_expect_tx(&C.full[slot], static_cast<uint32_t>(bytes));
          }
          // the bonus row is never read in full again: first out of L2
          fill(ring + static_cast<size_t>(slot) * kChunkBytes, src, off, bytes, &C.full[slot],
               pos == kb, evict_first);
          if (!P.bulk) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&C.full[slot]);
          }
          ++q;
          if (!fetched && r == nrows - 1) {
            if (lane == 0) t_next = atomicAdd(P.ws.ticket, 1);
            t_next = __shfl_sync(0xffffffffu, t_next, 0);
            fetch(t_next, sq_next, xj_next, uj_next);
            fetched = true;
          }
          ok = service_requests(q);
        }
      }
      if (!fetched) {
        if (lane == 0) t_next = atomicAdd(P.ws.ticket, 1);
        t_next = __shfl_sync(0xffffffffu, t_next, 0);
        fetch(t_next, sq_next, xj_next, uj_next);
      }
      ++streamed;
      t = t_next;
      sq = sq_next;
      xj = xj_next;
      uj = uj_next;
    }
    // no more sequences: keep serving re-reads until every streamed sequence
    // is finished, then signal the end (bounded: 1 s without progress)
    unsigned long long t0 = global_ns();
    int last_done = -1;
    while (ok) {
      ok = service_requests(q);
      int done = 0;
      if (lane == 0) done = C.seqs_finished;
      done = __shfl_sync(0xffffffffu, done, 0);
      if (done >= streamed) break;
      if (done != last_done) { last_done = done; t0 = global_ns(); }
      if (static_cast<long long>(global_ns() - t0) > kDrainLimitNs) {
        if (lane == 0) atomicOr(P.ws.err_word, 1u << 5 /* SV_ERR_TIMEOUT */);
        break;
      }
      __nanosleep(256);
    }
    if (acquire_slot(q)) {
      if (lane == 0) {
        C.desc[q % S].kind = -1;
        mbar_arrive(&C.full[q % S]);
      }
    }
  }

  // ======================= consumers =========================================
  // They never wait on each other: a finished row is published into a ring
  // of row buffers, a re-read's weights into a pair of mass arrays, and the
  // control warp takes it from there.

  __device__ void consume() {
    const int S = P.stages;
    const float c2 = P.c2;
    float rK = -INFINITY, rS = 0.f, rM = -INFINITY;   // running state of the current row
    int rArg = 0x7fffffff, rBad = 0;
    int q = 0, rr = 0, dr = 0;                        // slots, rows, re-reads seen
    while (true) {
      const int slot = q % S;
      const uint32_t par = static_cast<uint32_t>(q / S) & 1u;
      int timed_out = 0;
      if (!mbar_wait_bounded(&C.full[slot], par, P.wait_limit_ns)) {
        timed_out = 1;
        if (!mbar_wait_bounded(&C.full[slot], par, kDrainLimitNs)) {
          if (lane == 0) atomicOr(P.ws.err_word, 1u << 5 /* SV_ERR_TIMEOUT */);
          return;   // the producer is gone
        }
      }
      const Desc d = C.desc[slot];
      if (d.kind < 0) {
        // tell the control warp that the work is over
        const int buf = rr % kRowBufs;
        if (!warp_wait(&C.row_free[buf], ((rr / kRowBufs) & 1) ^ 1)) return;
        if (warp == 0 && lane == 0) C.rows[buf].d.kind = -1;
        __syncwarp();
        if (lane == 0) mbar_arrive(&C.row_ready[buf]);
        return;
      }

      if (d.kind == 2) {
        // ---- a chunk of a pair's re-read: per-segment draw weights --------
        const int dp = dr & 1;
        if (d.chunk == 0 && !warp_wait(&C.draw_free[dp], ((dr >> 1) & 1) ^ 1)) return;
        const bool resid = (d.x == 1);
        const unsigned char* data = ring + static_cast<size_t>(slot) * kChunkBytes;
        const long long off = static_cast<long long>(d.chunk) * kHalfBytes;
        const long long rem = row_bytes - off;
        const int nvec = static_cast<int>(((rem < kHalfBytes ? rem : kHalfBytes) + 15) / 16);
        uint4 rt[kDrawVecsPerLane], rd[kDrawVecsPerLane];
#pragma unroll
        for (int j = 0; j < kDrawVecsPerLane; ++j) {
          const int v = warp * kDrawVecsPerWarp + j * 32 + lane;
          const bool in = v < nvec;
          rt[j] = in ? *reinterpret_cast<const uint4*>(data + static_cast<size_t>(v) * 16) : V::neg_inf();
          rd[j] = (in && resid) ? *reinterpret_cast<const uint4*>(data + kHalfBytes + static_cast<size_t>(v) * 16)
                                : V::neg_inf();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&C.empty[slot]);
        const f2 cc = pack2(c2, c2), nkt = pack2(-d.K0, -d.K0), nlt = pack2(-d.L0, -d.L0);
        const f2 nkd = pack2(-d.K1, -d.K1), nld = pack2(-d.L1, -d.L1);
        f2 acc[NV / 2];
#pragma unroll
        for (int i = 0; i < NV / 2; ++i) acc[i] = 0ull;
#pragma unroll
        for (int j = 0; j < kDrawVecsPerLane; ++j) {
          f2 zt[NV / 2], zd[NV / 2];
          V::pairs(rt[j], zt);
          V::pairs(rd[j], zd);
#pragma unroll
          for (int i = 0; i < NV / 2; ++i) {
            // the same roundings as the scalar fmaf(z, c, -K) - L of the walk
            const f2 p = exp2_2(add2(fma2(zt[i], cc, nkt), nlt));
            if (resid) {
              float d0, d1;
              unpack2(sub2(p, exp2_2(add2(fma2(zd[i], cc, nkd), nld))), d0, d1);
              acc[i] = add2(acc[i], pack2(fmaxf(d0, 0.f), fmaxf(d1, 0.f)));
            } else {
              acc[i] = add2(acc[i], p);
            }
          }
        }
        float a0, a1, sum = 0.f;
#pragma unroll
        for (int i = 0; i < NV / 2; ++i) { unpack2(acc[i], a0, a1); sum += a0 + a1; }
        const float ws = warp_sum(sum);
        if (lane == 0) {
          C.rmass[dp][d.chunk * kConsumerWarps + warp] = static_cast<double>(ws);
          if (timed_out) atomicOr(&C.draw_err[dp], 1);
        }
        if (d.chunk == d.nchunks - 1) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&C.draw_ready[dp]);
          ++dr;
        }
        ++q;
        continue;
      }

      // ---- a chunk of a streamed row ----------------------------------------
      const int buf = rr % kRowBufs;
      RowBuf& RB = C.rows[buf];
      if (d.chunk == 0) {
        if (!warp_wait(&C.row_free[buf], ((rr / kRowBufs) & 1) ^ 1)) return;
        rK = -INFINITY; rS = 0.f; rM = -INFINITY; rArg = 0x7fffffff; rBad = 0;
      }
      const unsigned char* data = ring + static_cast<size_t>(slot) * kChunkBytes;
      const long long off = static_cast<long long>(d.chunk) * kChunkBytes;
      const long long rem = row_bytes - off;
      const int nvec = static_cast<int>(((rem < kChunkBytes ? rem : kChunkBytes) + 15) / 16);
      uint4 raw[kVecsPerLane];
#pragma unroll
      for (int j = 0; j < kVecsPerLane; ++j) {
        const int v = warp * kVecsPerWarp + j * 32 + lane;
        raw[j] = v < nvec ? *reinterpret_cast<const uint4*>(data + static_cast<size_t>(v) * 16) : V::neg_inf();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&C.empty[slot]);   // the slot is free again

      const int seg = d.chunk * kConsumerWarps + warp;
      const int seg_base = seg * kSegElems;
      if (timed_out) rBad |= 2;
      // the drafted token's logit
      if (d.x >= 0 && d.x < P.V && !P.greedy) {
        const int rel = d.x - seg_base;
        if (rel >= 0 && rel < kSegElems && ((rel / NV) & 31) == lane) {
          const int vv = rel / NV;
          const int j = vv >> 5, e = rel - vv * NV;
#pragma unroll
          for (int jj = 0; jj < kVecsPerLane; ++jj) {
            if (jj == j) {
              float z[NV];
              V::unpack(raw[jj], z);
#pragma unroll
              for (int ee = 0; ee < NV; ++ee)
                if (ee == e) RB.zx = z[ee];
            }
          }
        }
      }
      if (P.greedy) {
        float lm = -INFINITY;
        int li = 0x7fffffff, bad = 0;
#pragma unroll
        for (int j = 0; j < kVecsPerLane; ++j) {
          float z[NV];
          V::unpack(raw[j], z);
#pragma unroll
          for (int e = 0; e < NV; ++e) {
            bad |= (z[e] != z[e]) || (z[e] == INFINITY);
            if (z[e] > lm) { lm = z[e]; li = seg_base + (j * 32 + lane) * NV + e; }
          }
        }
        warp_argmax(lm, li);
        bad = warp_or(bad);
        if (lm > rM) { rM = lm; rArg = li; }
        rBad |= bad;
      } else {
        const float wm = warp_max(V::vmax(raw));
        float Ks = -INFINITY, ss = 0.f;
        if (wm > -INFINITY) {
          Ks = __fmul_rn(wm, c2);      // fl(m c), used identically wherever rescaled
          const f2 cc = pack2(c2, c2), nk = pack2(-Ks, -Ks);
          f2 acc[NV / 2];
#pragma unroll
          for (int i = 0; i < NV / 2; ++i) acc[i] = 0ull;
#pragma unroll
          for (int j = 0; j < kVecsPerLane; ++j) {
            f2 z[NV / 2];
            V::pairs(raw[j], z);
#pragma unroll
            for (int i = 0; i < NV / 2; ++i) acc[i] = add2(acc[i], exp2_2(fma2(z[i], cc, nk)));
          }
          float a0, a1, sum = 0.f;
#pragma unroll
          for (int i = 0; i < NV / 2; ++i) { unpack2(acc[i], a0, a1); sum += a0 + a1; }
          ss = warp_sum(sum);   // NaN logits make this NaN: caught at the row end
          if (Ks > rK) { rS = rS * fast_exp2(__fsub_rn(rK, Ks)) + ss; rK = Ks; }
          else         { rS += ss * fast_exp2(__fsub_rn(Ks, rK)); }
        } else {
          // no finite logit in the segment: only NaN can still hide here
          int nan_seen = 0;
#pragma unroll
          for (int j = 0; j < kVecsPerLane; ++j) {
            float z[NV];
            V::unpack(raw[j], z);
#pragma unroll
            for (int e = 0; e < NV; ++e) nan_seen |= (z[e] != z[e]);
          }
          rBad |= warp_or(nan_seen);
        }
        rM = fmaxf(rM, wm);
        if (d.kind == 0 && d.pos == d.kb && lane == 0 && seg < kMaxChunks * kConsumerWarps) {
          RB.segK[seg] = Ks;
          RB.segS[seg] = ss;
        }
      }

      if (d.chunk == d.nchunks - 1) {
        // publish the row: this warp's state, the descriptor (warp 0)
        if (lane == 0) {
          RB.wK[warp] = rK; RB.wS[warp] = rS; RB.wM[warp] = rM; RB.wArg[warp] = rArg; RB.wBad[warp] = rBad;
          if (warp == 0) RB.d = d;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&C.row_ready[buf]);
        ++rr;
      }
      ++q;
    }
  }

  // ======================= control warp ======================================

  __device__ void push_request(const DrawReq& r) {
    // the control warp (lane 0) produces, the producer warp consumes
    unsigned long long t0 = 0;
    while (C.req_tail - C.req_head >= kReqs) {
      if (!t0) t0 = global_ns();
      if (static_cast<long long>(global_ns() - t0) > kDrainLimitNs) {
        atomicOr(P.ws.err_word, 1u << 5 /* SV_ERR_TIMEOUT */);
        C.rec[r.rec].err |= kErrTimeout;
        return;
      }
    }
    const int tail = C.req_tail;
    C.req[tail % kReqs] = r;
    C.ctl_req[C.pushed % kReqs] = r;
    C.pushed = C.pushed + 1;
    __threadfence_block();
    C.req_tail = tail + 1;
  }

  // The segment holding s * S among `nseg` masses (index order).
  __device__ void locate(const double* mass, int nseg, float s, double& Stot, int& seg, double& seg_t) const {
    const int per = (nseg + 31) / 32;
    const int g0 = min(nseg, lane * per), g1 = min(nseg, g0 + per);
    double gs = 0.0;
    for (int i = g0; i < g1; ++i) gs += mass[i];
    const double incl = warp_incl_scan(gs, lane);
    const double excl = incl - gs;
    Stot = __shfl_sync(0xffffffffu, incl, 31);
    const double tgt = static_cast<double>(s) * Stot;
    const unsigned hit = __ballot_sync(0xffffffffu, gs > 0.0 && tgt < incl);
    const unsigned posg = __ballot_sync(0xffffffffu, gs > 0.0);
    const int owner = hit ? (__ffs(hit) - 1) : (posg ? 31 - __clz(posg) : -1);
    seg = -1;
    seg_t = 0.0;
    if (owner >= 0 && lane == owner) {
      double run = excl, last_run = excl;
      int last = -1;
      for (int i = g0; i < g1; ++i) {
        const double m = mass[i];
        if (m > 0.0) { last = i; last_run = run; }
        if (seg < 0 && m > 0.0 && tgt < run + m) { seg = i; seg_t = tgt - run; }
        run += m;
      }
      if (seg < 0) { seg = last; seg_t = tgt - last_run; }
    }
    if (owner >= 0) {
      seg = __shfl_sync(0xffffffffu, seg, owner);
      seg_t = __shfl_sync(0xffffffffu, seg_t, owner);
    }
  }

  // Walk NSTEPS x 32 vectors starting at vector v0, a warp inclusive scan
  // per step, to the token where the running weight passes t.
  // RESID: weights max(0, p - q); else p.
  template <int NSTEPS, bool RESID>
  __device__ int walk(int v0, double t, const unsigned char* rowT, const unsigned char* rowD,
                      float Kt, float Lt, float Kd, float Ld) const {
    uint4 rt[NSTEPS], rd[RESID ? NSTEPS : 1];
#pragma unroll
    for (int j = 0; j < NSTEPS; ++j) {
      rt[j] = load_global_raw(rowT, v0 + j * 32 + lane);
      if (RESID) rd[RESID ? j : 0] = load_global_raw(rowD, v0 + j * 32 + lane);
    }
    double base = 0.0;
    int found = -1, last_positive = -1;
#pragma unroll
    for (int j = 0; j < NSTEPS; ++j) {
      float w[NV], zt[NV], zd[NV];
      V::unpack(rt[j], zt);
      if (RESID) V::unpack(rd[RESID ? j : 0], zd);
      float ls = 0.f;
#pragma unroll
      for (int e = 0; e < NV; ++e) {
        const float p = fast_exp2(fmaf(zt[e], P.c2, -Kt) - Lt);
        w[e] = RESID ? fmaxf(p - fast_exp2(fmaf(zd[e], P.c2, -Kd) - Ld), 0.f) : p;
        ls += w[e];
      }
      const float incl = warp_incl_scan(ls, lane);
      float excl = __shfl_up_sync(0xffffffffu, incl, 1);
      if (lane == 0) excl = 0.f;
      const float step_total = __shfl_sync(0xffffffffu, incl, 31);
      const int x0 = (v0 + j * 32 + lane) * NV;
      const bool mine = found < 0 && ls > 0.f && t < base + static_cast<double>(incl) &&
                        !(t < base + static_cast<double>(excl));
      const unsigned hit = __ballot_sync(0xffffffffu, mine);
      int lp = -1;
#pragma unroll
      for (int e = 0; e < NV; ++e) if (w[e] > 0.f) lp = x0 + e;
      const unsigned anyp = __ballot_sync(0xffffffffu, lp >= 0);
      if (found < 0 && anyp) last_positive = __shfl_sync(0xffffffffu, lp, 31 - __clz(anyp));
      if (hit) {
        const int hl = __ffs(hit) - 1;
        int pick = -1;
        if (lane == hl) {
          double c = base + static_cast<double>(excl);
          int lastp = -1;
#pragma unroll
          for (int e = 0; e < NV; ++e) {
            if (w[e] > 0.f) lastp = x0 + e;
            c += static_cast<double>(w[e]);
            if (pick < 0 && w[e] > 0.f && t < c) pick = x0 + e;
          }
          if (pick < 0) pick = lastp;
        }
        found = __shfl_sync(0xffffffffu, pick, hl);
      }
      base += static_cast<double>(step_total);
    }
    return found >= 0 ? found : last_positive;
  }

  // Outputs of a sequence whose stream and draw are both done.
  __device__ void finish_sequence(int rec) {
    const SeqRec& R = C.rec[rec];
    const int k = P.k;
    const size_t b = static_cast<size_t>(R.b);
    int* ot = P.out_tokens + b * (k + 1);
    const int err = R.err;
    const int a = R.a < 0 ? R.kb : R.a;
    const int y = R.y;
    const bool ok = !err && y >= 0;
    for (int j = lane; j <= k; j += 32) {
      int v = -1;
      if (ok) v = j < a ? __ldg(P.tokens + b * k + j) : (j == a ? y : -1);
      ot[j] = v;
    }
    if (lane == 0) {
      P.out_len[b] = ok ? a + 1 : 0;
      if (ok) {
        atomicAdd(P.ws.stats + kStatSequences, 1ull);
        atomicAdd(P.ws.stats + kStatProposed, static_cast<unsigned long long>(R.kb));
        atomicAdd(P.ws.stats + kStatAccepted, static_cast<unsigned long long>(a));
        atomicAdd(P.ws.stats + kStatEmitted, static_cast<unsigned long long>(a + 1));
        if (R.kb == 0) atomicAdd(P.ws.stats + kStatSpecOff, 1ull);
        if (R.zero_resid) atomicAdd(P.ws.stats + kStatZeroResidual, 1ull);
      } else {
        atomicAdd(P.ws.stats + kStatErrorSeqs, 1ull);
        unsigned bits = static_cast<unsigned>(err & (kErrBadToken | kErrNonfinite | kErrTimeout));
        if (!bits) bits = kErrNonfinite;   // no token could be drawn
        atomicOr(P.ws.err_word, bits);
      }
      __threadfence_block();
      C.seqs_finished = C.seqs_finished + 1;
    }
    __syncwarp();
  }

  // A finished row: combine the warps, decide, draw the bonus token.
  // Returns false at the end of the work.
  __device__ bool control_row(int buf) {
    const float c2 = P.c2;
    RowBuf& RB = C.rows[buf];
    const Desc d = RB.d;
    if (d.kind < 0) return false;
    // combine the consumer warps, one lane per warp
    const bool in = lane < kConsumerWarps;
    float M = in ? RB.wM[lane] : -INFINITY;
    int arg = in ? RB.wArg[lane] : 0x7fffffff;
    warp_argmax(M, arg);
    const float wk = in ? RB.wK[lane] : -INFINITY;
    const float K = warp_max(wk);
    const int bad = warp_or(in ? RB.wBad[lane] : 0);
    const float Ssum = warp_sum((in && wk > -INFINITY) ? RB.wS[lane] * fast_exp2(__fsub_rn(wk, K)) : 0.f);
    const float L = log2f(Ssum);
    SeqRec& R = C.rec[d.rec];
    const size_t b = static_cast<size_t>(d.b);
    int bonus = 0;
    if (lane == 0) {
      if (d.pos == 0 && d.kind == 0) {
        // first row of the sequence: open its record (free unless the ring of
        // records has wrapped onto a sequence still waiting for its draw)
        if (R.pending != 0) atomicOr(P.ws.err_word, 1u << 5 /* SV_ERR_TIMEOUT */);
        R.b = d.b; R.kb = d.kb; R.a = -1; R.err = 0; R.y = -1; R.zero_resid = 0;
        R.pending = 1; R.s = d.s;
      }
      if (bad & 2) R.err |= kErrTimeout;
      if (d.pos < d.kb && (d.x < 0 || d.x >= P.V)) R.err |= kErrBadToken;
      if (P.greedy) {
        if ((bad & 1) || !(M > -INFINITY)) R.err |= kErrNonfinite;
        P.ws.m_t[b * (P.k + 1) + d.pos] = M;
        if (d.pos < d.kb) {
          const bool acc = (d.x == arg);
          P.ws.alpha[b * P.k + d.pos] = acc ? 1.f : 0.f;
          if (!acc && R.a < 0) { R.a = d.pos; R.y = arg; }
        } else if (R.a < 0) {
          R.y = arg;
        }
      } else {
        if ((bad & 1) || !(isfinite(M) && isfinite(Ssum) && Ssum > 0.f)) R.err |= kErrNonfinite;
        if (d.kind == 0) {
          P.ws.m_t[b * (P.k + 1) + d.pos] = M;
          P.ws.L_t[b * (P.k + 1) + d.pos] = L;
          C.pairK = K; C.pairL = L; C.pairZx = RB.zx;
        } else {
          P.ws.m_d[b * P.k + d.pos] = M;
          P.ws.L_d[b * P.k + d.pos] = L;
        }
        if (d.kind == 1 && !R.err) {
          // the pair is complete: acceptance test of draft d.pos
          const float zt = C.pairZx, zd = RB.zx;
          float alpha;
          if (zt == -INFINITY) alpha = 0.f;               // p(x) = 0
          else if (zd == -INFINITY) alpha = 1.f;          // q(x) = 0 < p(x)
          else {
            const float log2r = (fmaf(zt, c2, -C.pairK) - C.pairL) - (fmaf(zd, c2, -K) - L);
            alpha = log2r >= 0.f ? 1.f : exp2f(log2r);
          }
          P.ws.alpha[b * P.k + d.pos] = alpha;
          if (!(d.u < alpha) && R.a < 0) {
            // first rejection: the producer re-reads this pair for the draw
            R.a = d.pos;
            R.pending += 1;
            DrawReq rq;
            rq.b = d.b; rq.pos = d.pos; rq.rec = d.rec; rq.mode = 1;
            rq.Kt = C.pairK; rq.Lt = C.pairL; rq.Kd = K; rq.Ld = L;
            push_request(rq);
          }
        } else if (d.kind == 0 && d.pos == d.kb && R.a < 0 && !R.err) {
          bonus = 1;   // every draft accepted: the bonus draw
        }
      }
    }
    bonus = __shfl_sync(0xffffffffu, bonus, 0);
    __syncwarp();
    if (bonus) {
      // masses of the stream segments from the sums kept while streaming,
      // then one segment of the bonus row is read again
      const int nseg = nchunks * kConsumerWarps;
      for (int sg = lane; sg < nseg; sg += 32) {
        const float ks = RB.segK[sg];
        C.bmass[sg] = ks == -INFINITY ? 0.0
                      : static_cast<double>(RB.segS[sg]) * static_cast<double>(fast_exp2(__fsub_rn(ks, K) - L));
      }
      __syncwarp();
      double S;
      int seg;
      double seg_t;
      locate(C.bmass, nseg, R.s, S, seg, seg_t);
      int y = -1;
      if (seg >= 0)
        y = walk<kVecsPerLane, false>(seg * kVecsPerWarp, seg_t, row_ptr(d.b, d.kb, 0), nullptr, K, L, 0.f, 0.f);
      if (lane == 0) {
        R.y = y;
        P.ws.mass[b * (P.k + 1) + d.kb] = static_cast<float>(S);
      }
      __syncwarp();
    }
    if (d.pos == d.kb && d.kind == 0) {
      // the sequence's stream is done
      int fin = 0;
      if (lane == 0) fin = (--R.pending == 0) ? 1 : 0;
      fin = __shfl_sync(0xffffffffu, fin, 0);
      if (fin) finish_sequence(d.rec);
    }
    return true;
  }

  // A re-read draw whose segment weights are complete.
  __device__ void control_draw(int di) {
    const int dp = di & 1;
    const DrawReq r = C.ctl_req[di % kReqs];
    SeqRec& R = C.rec[r.rec];
    const int nseg = ndraw * kConsumerWarps;
    const bool resid = (r.mode == 1);
    double S;
    int seg;
    double seg_t;
    locate(C.rmass[dp], nseg, R.s, S, seg, seg_t);
    int fin = 0;
    if (lane == 0 && C.draw_err[dp]) { R.err |= kErrTimeout; C.draw_err[dp] = 0; }
    if (S > 0.0 || !resid) {
      int y = -1;
      if (seg >= 0) {
        if (resid)
          y = walk<kDrawVecsPerLane, true>(seg * kDrawVecsPerWarp, seg_t, row_ptr(r.b, r.pos, 0),
                                           row_ptr(r.b, r.pos, 1), r.Kt, r.Lt, r.Kd, r.Ld);
        else
          y = walk<kDrawVecsPerLane, false>(seg * kDrawVecsPerWarp, seg_t, row_ptr(r.b, r.pos, 0),
                                            nullptr, r.Kt, r.Lt, r.Kd, r.Ld);
      }
      if (lane == 0) {
        R.y = y;
        P.ws.mass[static_cast<size_t>(r.b) * (P.k + 1) + r.pos] = static_cast<float>(S);
        fin = (--R.pending == 0) ? 1 : 0;
      }
    } else if (lane == 0) {
      // exact arithmetic rules a zero residual out (a rejection implies
      // p > q somewhere); draw from p_a instead and count it
      R.zero_resid = 1;
      DrawReq rq = r;
      rq.mode = 2;
      push_request(rq);
    }
    fin = __shfl_sync(0xffffffffu, fin, 0);
    __syncwarp();
    if (fin) finish_sequence(r.rec);
  }

  __device__ void control() {
    int ri = 0, di = 0;
    unsigned long long idle_since = 0;
    while (true) {
      bool progressed = false;
      const int buf = ri % kRowBufs;
      int ready = 0;
      if (lane == 0) ready = mbar_test_wait(&C.row_ready[buf], static_cast<uint32_t>(ri / kRowBufs) & 1u) ? 1 : 0;
      ready = __shfl_sync(0xffffffffu, ready, 0);
      if (ready) {
        const bool more = control_row(buf);
        __syncwarp();
        if (lane == 0) mbar_arrive(&C.row_free[buf]);
        ++ri;
        if (!more) return;
        progressed = true;
      }
      int pushed = 0;
      if (lane == 0) pushed = C.pushed;
      pushed = __shfl_sync(0xffffffffu, pushed, 0);
      if (di < pushed) {
        const int dp = di & 1;
        int dready = 0;
        if (lane == 0) dready = mbar_test_wait(&C.draw_ready[dp], static_cast<uint32_t>(di >> 1) & 1u) ? 1 : 0;
        dready = __shfl_sync(0xffffffffu, dready, 0);
        if (dready) {
          control_draw(di);
          __syncwarp();
          if (lane == 0) mbar_arrive(&C.draw_free[dp]);
          ++di;
          progressed = true;
        }
      }
      if (progressed) {
        idle_since = 0;
      } else {
        if (!idle_since) idle_since = global_ns();
        if (static_cast<long long>(global_ns() - idle_since) > 4 * kDrainLimitNs) {
          if (lane == 0) atomicOr(P.ws.err_word, 1u << 5 /* SV_ERR_TIMEOUT */);
          return;
        }
        __nanosleep(64);
      }
    }
  }
};

template <int ELT>
__global__ void __launch_bounds__(kThreads, 1)
verify_kernel(const VerifyParams P) {
  extern __shared__ __align__(1024) unsigned char smem[];
  Ctrl& C = *reinterpret_cast<Ctrl*>(smem);
  unsigned char* ring = smem + kCtrlBytes;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < P.stages; ++s) {
      mbar_init(&C.full[s], 1);
      mbar_init(&C.empty[s], kConsumerWarps);
    }
    for (int r = 0; r < kRowBufs; ++r) {
      mbar_init(&C.row_ready[r], kConsumerWarps);
      mbar_init(&C.row_free[r], 1);
    }
    for (int r = 0; r < 2; ++r) {
      mbar_init(&C.draw_ready[r], kConsumerWarps);
      mbar_init(&C.draw_free[r], 1);
      C.draw_err[r] = 0;
    }
    C.req_head = 0;
    C.req_tail = 0;
    C.pushed = 0;
    C.seqs_finished = 0;
    for (int r = 0; r < kRecs; ++r) C.rec[r].pending = 0;
    fence_mbar_init();
  }
  __syncthreads();
  grid_dependency_wait();           // the work list of plan_kernel is ready
  Verifier<ELT> v(P, C, ring, lane, warp);
  if (warp < kConsumerWarps) v.consume();
  else if (warp == kConsumerWarps) v.produce();
  else v.control();
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

__global__ void init_workspace_kernel(Workspace ws) {
  const int i = threadIdx.x;
  if (i < kStatCount) ws.stats[i] = 0ull;
  if (i == 0) { *ws.err_word = 0u; *ws.n_seqs = 0; *ws.ticket = 0; }
}

}  // namespace

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------

int verify_smem_bytes(int stages) { return kCtrlBytes + stages * kChunkBytes; }

cudaError_t prepare_verify_kernel(int smem_bytes) {
  const void* fns[2] = {reinterpret_cast<const void*>(&verify_kernel<2>),
                        reinterpret_cast<const void*>(&verify_kernel<4>)};
  for (const void* f : fns) {
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t query_ctas_per_sm(int smem_bytes, int* out) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, verify_kernel<2>, kThreads,
                                                       static_cast<size_t>(smem_bytes));
}

cudaError_t launch_verify(const VerifyParams& p, int ctas, int smem_bytes, cudaStream_t s) {
  plan_kernel<<<1, kPlanThreads, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
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

cudaError_t launch_init_workspace(const Workspace& ws, cudaStream_t s) {
  init_workspace_kernel<<<1, 32, 0, s>>>(ws);
  return cudaGetLastError();
}

}  // namespace sv
