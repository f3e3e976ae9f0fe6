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

// Barrier of the consumer warps only (the producer never joins it).
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" :: "n"(kConsumerWarps * 32) : "memory");
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

// ---------------------------------------------------------------------------
// Shared control block
// ---------------------------------------------------------------------------

// What a staging slot holds.
//   kind 0 / 1: chunk `chunk` of the target / draft row at position pos;
//   kind 2:     chunk `chunk` of the re-read of the pair at pos for its draw:
//               the first half of the slot holds target logits, the second
//               half the draft logits of the same vocabulary range (x holds
//               the draw mode: 1 residual max(0, p - q), 2 p alone);
//   kind -1:    no more work.
struct Desc {
  int b, kb, pos, kind;
  int chunk, nchunks, x, rec;  // x: drafted token at pos (rows of pairs, else -1); rec: sequence record
  float u, s;                  // accept uniform at pos, sampling uniform of b
};

// One sequence in flight.  Its stream and its draw can finish in either
// order; the outputs are written when both are done.
struct SeqRec {
  int b, kb, a, err, y, zero_resid;
  int pending;                 // events left before the outputs can be written
  float Kt, Lt, Kd, Ld;        // normalisers of the pair being drawn from
  float s;                     // sampling uniform
};

constexpr int kRecs = 8;       // sequence records (ring)
constexpr int kReqs = 8;       // re-read requests (ring)
constexpr int kHalfBytes = kChunkBytes / 2;                   // one row's part of a draw chunk
constexpr int kDrawVecsPerWarp = kHalfBytes / 16 / kConsumerWarps;   // 128
constexpr int kDrawVecsPerLane = kDrawVecsPerWarp / 32;              // 4
constexpr int kMaxDrawSegs = 2 * kMaxChunks * kConsumerWarps;

enum : int { kErrBadToken = 1 << 3, kErrNonfinite = 1 << 4, kErrTimeout = 1 << 5 };

struct Ctrl {
  uint64_t full[kMaxStages];   // slot filled (producer -> consumers)
  uint64_t empty[kMaxStages];  // slot released (one arrival per consumer warp)
  Desc desc[kMaxStages];
  // per-warp row state published at a row end
  float wK[kConsumerWarps], wS[kConsumerWarps], wM[kConsumerWarps];
  int wArg[kConsumerWarps], wBad[kConsumerWarps];
  // the current pair: [0] target row, [1] draft row
  float zx[2];
  float rowK[2], rowL[2];
  SeqRec rec[kRecs];
  // re-read requests: consumer thread 0 pushes, the producer pops
  int req_b[kReqs], req_pos[kReqs], req_rec[kReqs], req_mode[kReqs];
  volatile int req_head, req_tail;
  volatile int seqs_finished;  // sequences whose outputs are written
  // broadcasts from consumer thread 0 / warp 0 to the consumer warps
  int flag_bonus, flag_finish;
  // the draw being located
  int seg;
  double seg_t, S;
  float segK[kMaxChunks * kConsumerWarps];   // bonus row: per-segment fl(m c)
  float segS[kMaxChunks * kConsumerWarps];   // bonus row: per-segment sum
  double bmass[kMaxChunks * kConsumerWarps]; // bonus draw: weight per stream segment
  double rmass[kMaxDrawSegs];                // re-read draws: weight per draw segment
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

  // ======================= producer ==========================================

  // Wait for slot q%S to be free (lane 0 waits, the warp follows).
  __device__ bool acquire_slot(int q) {
    const int S = P.stages;
    int ok = 1;
    if (lane == 0) ok = mbar_wait_bounded(&C.empty[q % S], ((q / S) & 1) ^ 1, kDrainLimitNs) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok && lane == 0) atomicOr(P.ws.err_word, 1u << 5 /* SV_ERR_TIMEOUT */);
    __syncwarp();
    return ok != 0;
  }

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

  // Issue the draw chunks of every queued re-read request.
  __device__ bool service_requests(int& q) {
    const int S = P.stages;
    while (true) {
      int head = 0, tail = 0;
      if (lane == 0) { head = C.req_head; tail = C.req_tail; }
      head = __shfl_sync(0xffffffffu, head, 0);
      tail = __shfl_sync(0xffffffffu, tail, 0);
      if (head == tail) return true;
      const int r = head % kReqs;
      const int b = C.req_b[r], pos = C.req_pos[r], rec = C.req_rec[r], mode = C.req_mode[r];
      __syncwarp();
      if (lane == 0) { __threadfence_block(); C.req_head = head + 1; }
      const unsigned char* srcT = row_ptr(b, pos, 0);
      const unsigned char* srcD = row_ptr(b, pos, 1);
      for (int c = 0; c < ndraw; ++c) {
        if (!acquire_slot(q)) return false;
        const int slot = q % S;
        const long long off = static_cast<long long>(c) * kHalfBytes;
        const long long rem = row_bytes - off;
        const int bytes = static_cast<int>(rem < kHalfBytes ? rem : kHalfBytes);
        unsigned char* dst = ring + static_cast<size_t>(slot) * kChunkBytes;
        if (lane == 0) {
          Desc& d = C.desc[slot];
          d.b = b; d.kb = 0; d.pos = pos; d.kind = 2;
          d.chunk = c; d.nchunks = ndraw; d.x = mode; d.rec = rec;
          d.u = 0.f; d.s = 0.f;
          if (P.bulk) mbar_expect_tx(&C.full[slot], static_cast<uint32_t>(mode == 1 ? 2 * bytes : bytes));
        }
        fill(dst, srcT, off, bytes, &C.full[slot], false, 0);
        if (mode == 1) fill(dst + kHalfBytes, srcD, off, bytes, &C.full[slot], false, 0);
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
    int t = 0;
    if (lane == 0) t = atomicAdd(P.ws.ticket, 1);
    t = __shfl_sync(0xffffffffu, t, 0);
    bool ok = true;
    while (ok && t < n_seqs) {
      const int2 sq = __ldcg(P.ws.seqs + t);
      const int b = sq.x, kb = sq.y;
      const int rec = streamed % kRecs;
      int t_next = 0;
      if (lane == 0) t_next = atomicAdd(P.ws.ticket, 1);
      // the sequence's drafted tokens and uniforms, one per lane
      const int xj = lane < kb ? __ldg(P.tokens + static_cast<size_t>(b) * k + lane) : -1;
      const float uj = (!P.greedy && lane <= k) ? __ldg(P.uniforms + static_cast<size_t>(b) * (k + 1) + lane) : 0.f;
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
          ok = service_requests(q);
        }
      }
      ++streamed;
      t = __shfl_sync(0xffffffffu, t_next, 0);
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
      __nanosleep(200);
    }
    if (acquire_slot(q)) {
      if (lane == 0) {
        C.desc[q % S].kind = -1;
        mbar_arrive(&C.full[q % S]);
      }
    }
  }

  // ======================= consumers =========================================

  __device__ void consume() {
    const int S = P.stages;
    const float c2 = P.c2;
    // warp-uniform running state of the current row
    float rK = -INFINITY, rS = 0.f, rM = -INFINITY;
    int rArg = 0x7fffffff, rBad = 0;
    int q = 0;
    while (true) {
      const int slot = q % S;
      const uint32_t par = static_cast<uint32_t>(q / S) & 1u;
      int timed_out = 0;
      if (!mbar_wait_bounded(&C.full[slot], par, P.wait_limit_ns)) {
        timed_out = 1;
        if (!mbar_wait_bounded(&C.full[slot], par, kDrainLimitNs)) {
          if (warp == 0 && lane == 0) atomicOr(P.ws.err_word, 1u << 5 /* SV_ERR_TIMEOUT */);
          return;   // the producer is gone; nothing is left in flight for this slot
        }
      }
      const Desc d = C.desc[slot];
      if (d.kind < 0) return;
      if (d.kind == 2) {
        draw_chunk(d, slot, timed_out);
        ++q;
        continue;
      }

      // this lane's vectors of the chunk (raw 16-byte words)
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
      if (d.chunk == 0) { rK = -INFINITY; rS = 0.f; rM = -INFINITY; rArg = 0x7fffffff; rBad = 0; }
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
                if (ee == e) C.zx[d.kind] = z[ee];
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
          C.segK[seg] = Ks;
          C.segS[seg] = ss;
        }
      }

      if (d.chunk == d.nchunks - 1) row_end(d, rK, rS, rM, rArg, rBad);
      ++q;
    }
  }

  // Row end: combine the warps, then the decisions that need the row.
  __device__ void row_end(const Desc& d, float rK, float rS, float rM, int rArg, int rBad) {
    const int ctid = warp * 32 + lane;
    const float c2 = P.c2;
    if (lane == 0) {
      C.wK[warp] = rK; C.wS[warp] = rS; C.wM[warp] = rM; C.wArg[warp] = rArg; C.wBad[warp] = rBad;
    }
    consumer_sync();
    // warp 0 combines the warps' states, one lane per warp
    float M = -INFINITY, K = -INFINITY, Ssum = 0.f;
    int arg = 0x7fffffff, bad = 0;
    if (warp == 0) {
      const bool in = lane < kConsumerWarps;
      M = in ? C.wM[lane] : -INFINITY;
      arg = in ? C.wArg[lane] : 0x7fffffff;
      warp_argmax(M, arg);
      const float wk = in ? C.wK[lane] : -INFINITY;
      K = warp_max(wk);
      bad = warp_or(in ? C.wBad[lane] : 0);
      if (!P.greedy) Ssum = warp_sum(wk > -INFINITY ? C.wS[lane] * fast_exp2(__fsub_rn(wk, K)) : 0.f);
    }
    int bonus_draw = 0;
    if (ctid == 0) {
      SeqRec& R = C.rec[d.rec];
      const int kind = d.kind;
      const size_t b = static_cast<size_t>(d.b);
      if (d.pos == 0 && kind == 0) {
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
        const float L = log2f(Ssum);
        C.rowK[kind] = K;
        C.rowL[kind] = L;
        if ((bad & 1) || !(isfinite(M) && isfinite(Ssum) && Ssum > 0.f)) R.err |= kErrNonfinite;
        if (kind == 0) {
          P.ws.m_t[b * (P.k + 1) + d.pos] = M;
          P.ws.L_t[b * (P.k + 1) + d.pos] = L;
        } else {
          P.ws.m_d[b * P.k + d.pos] = M;
          P.ws.L_d[b * P.k + d.pos] = L;
        }
        if (kind == 1 && !R.err) {
          // the pair is complete: acceptance test of draft d.pos
          const float zt = C.zx[0], zd = C.zx[1];
          float alpha;
          if (zt == -INFINITY) alpha = 0.f;               // p(x) = 0
          else if (zd == -INFINITY) alpha = 1.f;          // q(x) = 0 < p(x)
          else {
            const float log2r = (fmaf(zt, c2, -C.rowK[0]) - C.rowL[0]) - (fmaf(zd, c2, -C.rowK[1]) - C.rowL[1]);
            alpha = log2r >= 0.f ? 1.f : exp2f(log2r);
          }
          P.ws.alpha[b * P.k + d.pos] = alpha;
          if (!(d.u < alpha) && R.a < 0) {
            // first rejection: the producer re-reads this pair for the draw
            R.a = d.pos;
            R.Kt = C.rowK[0]; R.Lt = C.rowL[0]; R.Kd = C.rowK[1]; R.Ld = C.rowL[1];
            R.pending += 1;
            push_request(d.b, d.pos, d.rec, 1);
          }
        } else if (kind == 0 && d.pos == d.kb && R.a < 0 && !R.err) {
          bonus_draw = 1;   // every draft accepted: the bonus draw
          R.Kt = K; R.Lt = L;
        }
      }
      C.flag_bonus = bonus_draw;   // broadcast through the barrier below
    }
    consumer_sync();
    if (C.flag_bonus) this->bonus_draw(d);
    if (d.pos == d.kb && d.kind == 0) {
      // the sequence's stream is done
      if (ctid == 0) C.flag_finish = (--C.rec[d.rec].pending == 0) ? 1 : 0;
      consumer_sync();
      if (C.flag_finish) finish_sequence(d.rec);
    }
  }

  __device__ void push_request(int b, int pos, int rec, int mode) {
    // single producer (this thread) / single consumer (the producer warp) ring
    unsigned long long t0 = 0;
    while (C.req_tail - C.req_head >= kReqs) {
      if (!t0) t0 = global_ns();
      if (static_cast<long long>(global_ns() - t0) > kDrainLimitNs) {
        atomicOr(P.ws.err_word, 1u << 5 /* SV_ERR_TIMEOUT */);
        C.rec[rec].err |= kErrTimeout;
        return;
      }
    }
    const int tail = C.req_tail;
    const int r = tail % kReqs;
    C.req_b[r] = b; C.req_pos[r] = pos; C.req_rec[r] = rec; C.req_mode[r] = mode;
    __threadfence_block();
    C.req_tail = tail + 1;
  }

  // Warp 0: the segment holding s * S among `nseg` masses (index order).
  // Writes C.S, C.seg, C.seg_t.
  __device__ void locate(const double* mass, int nseg, float s) {
    const int per = (nseg + 31) / 32;
    const int g0 = min(nseg, lane * per), g1 = min(nseg, g0 + per);
    double gs = 0.0;
    for (int i = g0; i < g1; ++i) gs += mass[i];
    const double incl = warp_incl_scan(gs, lane);
    const double excl = incl - gs;
    const double Stot = __shfl_sync(0xffffffffu, incl, 31);
    const double tgt = static_cast<double>(s) * Stot;
    const unsigned hit = __ballot_sync(0xffffffffu, gs > 0.0 && tgt < incl);
    const unsigned posg = __ballot_sync(0xffffffffu, gs > 0.0);
    const int owner = hit ? (__ffs(hit) - 1) : (posg ? 31 - __clz(posg) : -1);
    int seg = -1;
    double seg_t = 0.0;
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
    if (lane == 0) { C.S = Stot; C.seg = seg; C.seg_t = seg_t; }
  }

  // Warp 0: walk `nsteps` x 32 vectors starting at vector v0 of the row(s),
  // a warp inclusive scan per step, to the token where the running weight
  // passes t.  resid: weights max(0, p - q); else p.
  template <int NSTEPS, bool RESID>
  __device__ int walk(int v0, double t, const unsigned char* rowT, const unsigned char* rowD,
                      float Kt, float Lt, float Kd, float Ld) const {
    // all loads first (raw), then the scan
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

  // The bonus draw of the sequence whose last row just ended (blocking; the
  // producer keeps the ring full meanwhile): masses from the sums kept while
  // streaming, then one stream segment of the bonus row is read again.
  __device__ void bonus_draw(const Desc& d) {
    const int ctid = warp * 32 + lane;
    SeqRec& R = C.rec[d.rec];
    const float Kt = R.Kt, Lt = R.Lt;
    const int nseg = nchunks * kConsumerWarps;
    for (int sg = ctid; sg < nseg; sg += kConsumerWarps * 32) {
      const float ks = C.segK[sg];
      C.bmass[sg] = ks == -INFINITY ? 0.0
                    : static_cast<double>(C.segS[sg]) * static_cast<double>(fast_exp2(__fsub_rn(ks, Kt) - Lt));
    }
    consumer_sync();
    if (warp == 0) {
      locate(C.bmass, nseg, R.s);
      __syncwarp();
      const int seg = C.seg;
      int y = -1;
      if (seg >= 0)
        y = walk<kVecsPerLane, false>(seg * kVecsPerWarp, C.seg_t, row_ptr(d.b, d.kb, 0), nullptr, Kt, Lt, 0.f, 0.f);
      if (lane == 0) {
        R.y = y;
        P.ws.mass[static_cast<size_t>(d.b) * (P.k + 1) + d.kb] = static_cast<float>(C.S);
      }
    }
    consumer_sync();
  }

  // One chunk of a pair's re-read: per-segment weights of the draw; the last
  // chunk locates the token.
  __device__ void draw_chunk(const Desc& d, int slot, int timed_out) {
    SeqRec& R = C.rec[d.rec];
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
    if (timed_out && lane == 0) atomicOr(&R.err, kErrTimeout);
    const float c2 = P.c2;
    const float Kt = R.Kt, Lt = R.Lt, Kd = R.Kd, Ld = R.Ld;
    const f2 cc = pack2(c2, c2), nkt = pack2(-Kt, -Kt), nlt = pack2(-Lt, -Lt);
    const f2 nkd = pack2(-Kd, -Kd), nld = pack2(-Ld, -Ld);
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
    const int sg = d.chunk * kConsumerWarps + warp;
    if (lane == 0) C.rmass[sg] = static_cast<double>(ws);
    if (d.chunk != d.nchunks - 1) return;

    // last chunk: the total, the segment, the token
    consumer_sync();
    const int nseg = d.nchunks * kConsumerWarps;
    if (warp == 0) {
      locate(C.rmass, nseg, R.s);
      __syncwarp();
      if (C.S > 0.0 || !resid) {
        const int seg = C.seg;
        int y = -1;
        if (seg >= 0) {
          if (resid)
            y = walk<kDrawVecsPerLane, true>(seg * kDrawVecsPerWarp, C.seg_t, row_ptr(d.b, d.pos, 0),
                                             row_ptr(d.b, d.pos, 1), Kt, Lt, Kd, Ld);
          else
            y = walk<kDrawVecsPerLane, false>(seg * kDrawVecsPerWarp, C.seg_t, row_ptr(d.b, d.pos, 0),
                                              nullptr, Kt, Lt, Kd, Ld);
        }
        if (lane == 0) {
          R.y = y;
          P.ws.mass[static_cast<size_t>(d.b) * (P.k + 1) + d.pos] = static_cast<float>(C.S);
          C.flag_finish = (--R.pending == 0) ? 1 : 0;
        }
      } else if (lane == 0) {
        // exact arithmetic rules a zero residual out (a rejection implies
        // p > q somewhere); draw from p_a instead and count it
        R.zero_resid = 1;
        push_request(d.b, d.pos, d.rec, 2);
        C.flag_finish = 0;
      }
    }
    consumer_sync();
    if (C.flag_finish) finish_sequence(d.rec);
  }

  // Outputs of a sequence whose stream and draw are both done.
  __device__ void finish_sequence(int rec) {
    if (warp == 0) {
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
    C.req_head = 0;
    C.req_tail = 0;
    C.seqs_finished = 0;
    for (int r = 0; r < kRecs; ++r) C.rec[r].pending = 0;
    fence_mbar_init();
  }
  __syncthreads();
  grid_dependency_wait();           // the work list of plan_kernel is ready
  Verifier<ELT> v(P, C, ring, lane, warp);
  if (warp == kConsumerWarps) v.produce();
  else v.consume();
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
