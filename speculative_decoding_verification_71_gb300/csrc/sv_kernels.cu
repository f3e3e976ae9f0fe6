// Speculative-sampling verification kernels for sm_103a.
//
// verify_kernel is persistent and warp-specialised.  A cluster of cs CTAs
// (1, 2, 4 or 8) verifies whole sequences, one after another, taken from a
// work list ordered longest first (plan_kernel) with an atomic ticket.  Each
// CTA of the cluster owns one slice of the vocabulary (a 1/cs share of every
// row, in 128-byte-aligned pieces) and runs four roles:
//
//   producer warp    streams its slice of the sequence's rows in position
//                    order (target 0, draft 0, target 1, ..., target k_b)
//                    through a ring of 64 KB shared-memory slots with
//                    cp.async.bulk, and runs ahead into the next sequence;
//   16 consumer warps  fold every chunk into per-warp running maxima and sums
//                    of 2^(z c - fl(m c)), c = log2(e)/T (one ex2 per logit),
//                    and pick up the drafted token's logit;
//   control warp     combines the warps into the slice's part of the row,
//                    sends it to every CTA of the cluster (st.async into their
//                    shared memory, counted on their mbarriers), combines the
//                    parts into the row's log-sum-exp and decides: after draft
//                    row i, alpha_i = min(1, p_i(x_i) / q_i(x_i)) and accept iff
//                    u_i < alpha_i, up to the first rejection;
//   walker warp      walks the one segment that holds the drawn token and
//                    writes the sequence's outputs.
//
// Because every CTA of a cluster sees the positions of a sequence in order,
// the first rejection is known exactly, identically everywhere:
//   * at the first rejection a, the pair (target a, draft a) is read again
//     (each CTA its slice) for exact per-segment masses of max(0, p - q) and
//     of p; the slice, then the segment, holding s*S is found and the walker
//     of the CTA that owns it finds the token;
//   * if every draft is accepted, the bonus row needs no second pass: its
//     per-segment sums were kept while streaming, so only the one segment
//     holding s*S is read again.
// Every CTA of a cluster inserts the re-reads at the same place in its
// stream, so the CTAs see one common order of events and each waits only for
// events that come earlier in it; every wait is bounded.
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
#include "sv_device.cuh"

namespace sv {
namespace {

// ---------------------------------------------------------------------------
// Shared control block
// ---------------------------------------------------------------------------

// What a staging slot holds.
//   kind 0 / 1: chunk `chunk` of this CTA's slice of the target / draft row
//               at position pos of sequence b;
//   kind 2:     chunk `chunk` of the re-read of this CTA's slice of the
//               rejected pair at pos: the first half of the slot holds target
//               logits, the second half the draft logits of the same range;
//               K0, L0 are the target row's normaliser, G0 + G1 the log2
//               ratio of the target's to the draft's normaliser;
//   kind 3:     end of a sequence cut short (early exit): no data;
//   kind -1:    no more work; x = draws inserted in all.
struct Desc {
  int b, kb, pos, kind;
  int chunk, nchunks, x, rec;  // x: drafted token at pos (rows of pairs, else -1); rec: record slot
  int seq, pad;                // seq: sequences streamed before this one
  float u, s;                  // accept uniform at pos, sampling uniform of b
  float K0, L0, G0, G1;
};

// A finished row, published by the consumer warps for the control warp.
struct RowBuf {
  Desc d;
  float wK[kConsumerWarps], wS[kConsumerWarps], wM[kConsumerWarps];
  int wArg[kConsumerWarps], wBad[kConsumerWarps];
  float zx;                                  // logit of the drafted token (if in this slice)
  float segK[kMaxChunks * kConsumerWarps];   // bonus rows: per-segment fl(m c)
  float segS[kMaxChunks * kConsumerWarps];   // bonus rows: per-segment sum
};

// One CTA's reduction of its slice of a row, sent to every CTA of the cluster.
struct alignas(16) RowPart {
  float M, K, S, zx;           // max logit, fl(M c), sum 2^(z c - K), drafted logit
  int arg, bad, has_zx, pad;   // argmax, error bits, zx present
};

// One CTA's masses of its slice of a re-read pair.
struct alignas(16) DrawPart {
  double r, p;                 // sum max(0, p - q), sum p
  int err, pad[3];
};

// One sequence in flight, kept identically by every CTA of the cluster.
struct SeqRec {
  int b, kb, a, err, y, zero_resid;
  int open;                    // from the first row until the outputs are settled
  int draw;                    // a residual draw follows (final once resolved)
  volatile int resolved;       // seq + 1 once `draw` and the normalisers are final
  volatile int seq_tag;        // seq of the sequence the record holds (set when opened)
  volatile int decided;        // pairs decided so far (early exit)
  volatile int stop;           // a rejection or an error: later rows are not needed
  float s;                     // sampling uniform
  float Kt, Lt;                // target normaliser of the rejected pair
  float Gh, Gl;                // log2 (target / draft normaliser) of that pair, as Gh + Gl
  int tok[32];                 // drafted tokens, taken from the rows as they pass
};

// An inverse-CDF walk over one segment, handed from the control warp to the
// walker warp (which reads the logits and writes the sequence's outputs).
struct WalkReq {
  int rec, mode;               // mode 0: p over a stream segment; 1: max(0, p - q) / 2: p over a draw segment
  int v0, b, pos;              // first vector of the segment (-1: nothing to walk), row
  int pad;
  double t;                    // target weight left at the segment's start
  float K0, L0;                // normaliser of the target row
  float Gh, Gl;                // residual walks: log2 (target / draft normaliser) as Gh + Gl
};

constexpr int kRecs = 32;          // sequence records (ring)
constexpr int kWalkReqs = 16;      // walk requests (ring)
constexpr int kRowBufs = 4;        // row buffers (ring)
constexpr int kXRing = 4;          // exchange slots of rows and of draws
constexpr int kDrawLagChunks = 6;  // a draw is inserted about this many chunks after its sequence ends ...
constexpr int kExitLagChunks = 32; // early exit in a cluster: a decision spares the rows this many chunks later
constexpr int kMaxPending = 24;    // ... or when this many sequences wait for theirs
constexpr int kHalfBytes = kChunkBytes / 2;                          // one row's part of a draw chunk
constexpr int kDrawVecsPerWarp = kHalfBytes / 16 / kConsumerWarps;   // 128
constexpr int kDrawVecsPerLane = kDrawVecsPerWarp / 32;              // 4
constexpr int kMaxDrawSegs = 2 * kMaxChunks * kConsumerWarps;
constexpr int kSliceAlign = 64;    // slice boundaries in logits (128 B of bf16)

static_assert(sizeof(RowPart) == 32 && sizeof(DrawPart) == 32, "parts travel as two 16-byte stores");
static_assert(kMaxPending + 4 <= kRecs, "records must outlive the pending window");

enum : int { kErrBadToken = 1 << 3, kErrNonfinite = 1 << 4, kErrTimeout = 1 << 5 };

struct Ctrl {
  uint64_t full[kMaxStages];        // slot filled (producer -> consumers)
  uint64_t empty[kMaxStages];       // slot released (one arrival per consumer warp)
  uint64_t row_ready[kRowBufs];     // row published (one arrival per consumer warp)
  uint64_t row_free[kRowBufs];      // row consumed by the control warp
  uint64_t draw_ready[2];           // draw masses complete (one arrival per consumer warp)
  uint64_t draw_free[2];            // draw masses consumed by the control warp
  uint64_t xrow_ready[kXRing];      // every CTA's part of a row has arrived here
  uint64_t xrow_free[kXRing];       // every CTA has read this CTA's part of a row
  uint64_t xdraw_ready[kXRing];     // the same for draws
  uint64_t xdraw_free[kXRing];
  uint64_t tk_full[2];              // a ticket was delivered (by the first CTA)
  uint64_t tk_empty[2];             // first CTA: every CTA has read the ticket
  RowPart xrow[kXRing][kMaxCluster];
  DrawPart xdraw[kXRing][kMaxCluster];
  Desc desc[kMaxStages];
  RowBuf rows[kRowBufs];
  float rmass[2][kMaxDrawSegs];     // per-segment sum max(0, p - q) of a re-read
  float pmass[2][kMaxDrawSegs];     // per-segment sum p of a re-read
  int draw_rec[2];
  int draw_err[2];
  volatile int tk[2];
  int pend_end[kRecs];              // producer: rows streamed when a sequence ended
  SeqRec rec[kRecs];
  double bmass[kMaxChunks * kConsumerWarps];
  WalkReq wreq[kWalkers][kWalkReqs];   // control warp -> walker warps (one ring each, taken in turn)
  volatile int wreq_head[kWalkers], wreq_tail[kWalkers];
  volatile int ctl_done;            // the control warp has left
  float pairK, pairL, pairZx, pairS;     // target row of the current pair (pairS: its sum of 2^(z c - K))
};

constexpr int kCtrlBytes = ((static_cast<int>(sizeof(Ctrl)) + 1023) / 1024) * 1024;
static_assert(kCtrlBytes + 3 * kChunkBytes <= 227 * 1024, "three staging slots must fit in one CTA");

// ---------------------------------------------------------------------------
// plan_kernel: the work list (valid sequences, longest first) and resets.
// ---------------------------------------------------------------------------
constexpr int kPlanThreads = 1024;

constexpr int kPlanCached = 8;   // k_b values a thread keeps in registers (B <= 8192)

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const VerifyParams P) {
  if (P.timeline && threadIdx.x == 0) P.timeline[static_cast<size_t>(P.ctas) * kTimelineSlots] = global_ns();
  grid_dependents_launch();   // the verify grid may start its prologue now
  __shared__ int warp_cnt[32];
  __shared__ int base;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = P.B, k = P.k;
  const Workspace& ws = P.ws;
  // one read of the lengths; invalid ones are answered here
  int kbc[kPlanCached];
#pragma unroll
  for (int c = 0; c < kPlanCached; ++c) {
    const int b = c * kPlanThreads + tid;
    kbc[c] = b < B ? __ldg(P.draft_len + b) : -1;
  }
  for (int b = tid; b < B; b += kPlanThreads) {
    const int kb = b < kPlanCached * kPlanThreads ? kbc[b / kPlanThreads] : P.draft_len[b];
    if (kb < 0 || kb > k) {
      int* ot = P.out_tokens + static_cast<size_t>(b) * (k + 1);
      for (int j = 0; j <= k; ++j) ot[j] = -1;
      P.out_len[b] = 0;
      atomicOr(ws.err_word, 1u << 2 /* SV_ERR_BAD_DRAFT_LEN */);
      atomicAdd(ws.stats + kStatErrorSeqs, 1ull);
    }
  }
  if (P.diag) {
    for (int i = tid; i < B * (k + 1); i += kPlanThreads) {
      ws.m_t[i] = NAN; ws.L_t[i] = NAN; ws.mass[i] = NAN;
    }
    for (int i = tid; i < B * k; i += kPlanThreads) {
      ws.m_d[i] = NAN; ws.L_d[i] = NAN; ws.alpha[i] = NAN;
    }
  }
  // the first sequence of cluster i is entry i of the work list (no atomic
  // needed); the shared counter hands out the rest
  if (tid == 0) { base = 0; *ws.ticket = P.ctas / max(1, P.cluster); }
  __syncthreads();
  // counting sort by k_b, largest first, stable in b
  for (int L = k; L >= 0; --L) {
    for (int b0 = 0, c = 0; b0 < B; b0 += kPlanThreads, ++c) {
      const int b = b0 + tid;
      int kb = -1;
      if (b < B) {
        if (c < kPlanCached) {
#pragma unroll
          for (int cc = 0; cc < kPlanCached; ++cc)
            if (cc == c) kb = kbc[cc];
        } else {
          kb = P.draft_len[b];
        }
      }
      const bool take = (kb == L);
      const unsigned m = __ballot_sync(0xffffffffu, take);
      if (lane == 0) warp_cnt[warp] = __popc(m);
      __syncthreads();
      if (warp == 0) {
        const int cnt = warp_cnt[lane];
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int up = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += up;
        }
        warp_cnt[lane] = incl - cnt;
      }
      __syncthreads();
      if (take) ws.seqs[base + warp_cnt[warp] + __popc(m & ((1u << lane) - 1u))] = make_int2(b, kb);
      __syncthreads();
      if (tid == kPlanThreads - 1) base += warp_cnt[31] + __popc(m);
      __syncthreads();
    }
  }
  if (tid == 0) {
    *ws.n_seqs = base;
    if (P.timeline) P.timeline[static_cast<size_t>(P.ctas) * kTimelineSlots + 1] = global_ns();
  }
}

// ---------------------------------------------------------------------------
// verify_kernel
// ---------------------------------------------------------------------------

template <int ELT, bool GREEDY>
struct Verifier {
  using V = Vec<ELT>;
  static constexpr int NV = V::N;                          // logits per vector
  static constexpr int kSegElems = kVecsPerWarp * NV;      // logits per stream segment (chunk, warp)

  const VerifyParams& P;
  Ctrl& C;
  unsigned char* ring;
  const int lane, warp;
  const int cs, rank;           // CTAs in the cluster, this CTA's rank
  const long long row_bytes;    // V * ELT
  int slice_lo, slice_n;        // this CTA's logits [slice_lo, slice_lo + slice_n) of every row
  int slice_bytes;
  int nchunks;                  // stream chunks per slice (at least one)
  int ndraw;                    // draw chunks per slice (at least one)
  int v_lo, v_hi;               // 16-byte vectors of the row covering the slice
  int chunks0;                  // stream chunks per row of the first (largest) slice
  int lag_rows;                 // rows between a sequence's end and its re-read (same in every CTA)
  int exit_lag;                 // early exit: pairs between a decision and the rows it can spare

  __device__ Verifier(const VerifyParams& p, Ctrl& c, unsigned char* r, int ln, int wp, int ncta, int rk)
      : P(p), C(c), ring(r), lane(ln), warp(wp), cs(ncta), rank(rk),
        row_bytes(static_cast<long long>(p.V) * ELT) {
    const int per = ((p.V + cs - 1) / cs + kSliceAlign - 1) / kSliceAlign * kSliceAlign;
    slice_lo = min(p.V, rank * per);
    const int hi = min(p.V, slice_lo + per);
    slice_n = hi - slice_lo;
    slice_bytes = slice_n * ELT;
    nchunks = max(1, (slice_bytes + kChunkBytes - 1) / kChunkBytes);
    ndraw = max(1, (slice_bytes + kHalfBytes - 1) / kHalfBytes);
    v_lo = slice_lo / NV;                       // slice_lo is a multiple of kSliceAlign
    v_hi = (hi * ELT + 15) / 16;
    // counted in chunks of the first (largest) slice so that every CTA agrees
    chunks0 = max(1, (min(p.V, per) * ELT + kChunkBytes - 1) / kChunkBytes);
    lag_rows = max(1, (kDrawLagChunks + chunks0 - 1) / chunks0);
    const int pair_chunks = (GREEDY ? 1 : 2) * chunks0;
    exit_lag = max(1, (kExitLagChunks + pair_chunks - 1) / pair_chunks);
  }

  __device__ const unsigned char* row_ptr(int b, int pos, int kind) const {
    if (kind == 0)
      return static_cast<const unsigned char*>(P.target) +
             (static_cast<size_t>(b) * (P.k + 1) + pos) * static_cast<size_t>(row_bytes);
    return static_cast<const unsigned char*>(P.draft) +
           (static_cast<size_t>(b) * P.k + pos) * static_cast<size_t>(row_bytes);
  }

  // Vector v of a row read straight from global memory, -inf outside the slice.
  __device__ uint4 load_global_raw(const unsigned char* row, int v) const {
    if (v < v_lo || v >= v_hi) return V::neg_inf();
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

  // One look at a phase (lane 0 looks, every lane learns the answer and, if
  // it completed, takes its own acquire).
  __device__ bool probe(uint64_t* bar, uint32_t parity) const {
    int r = 0;
    if (lane == 0) r = mbar_test_wait(bar, parity) ? 1 : 0;
    r = __shfl_sync(0xffffffffu, r, 0);
    if (r) mbar_test_wait(bar, parity);
    return r != 0;
  }

  // ======================= producer ==========================================
  // Every CTA of a cluster streams its slice of the same rows and inserts the
  // same re-reads at the same places, so the CTAs see one common order of
  // events and each waits only for events that come earlier in it.

  // Copy `bytes` of a row starting at byte `off` into dst (bulk or plain).
  __device__ void fill(unsigned char* dst, const unsigned char* src, long long off, int bytes,
                       uint64_t* bar, bool hint, uint64_t policy) {
    if (P.bulk) {
      if (lane == 0 && bytes > 0) {
        if (hint) bulk_load_hint(dst, src + off, static_cast<uint32_t>(bytes), bar, policy);
        else bulk_load(dst, src + off, static_cast<uint32_t>(bytes), bar);
      }
    } else {
      // plain loads (rows not 16-byte aligned); pad the last vector with -inf
      const int e0 = static_cast<int>(off / ELT);
      const int n = bytes / ELT;
      const int npad = ((n + NV - 1) / NV) * NV;
      for (int e = lane; e < npad; e += 32)
        V::store_scalar(dst, e, e < n ? V::scalar(src, e0 + e) : -INFINITY);
    }
  }

  __device__ bool acquire_slot(int q) {
    const int S = P.stages;
    return warp_wait(&C.empty[q % S], ((q / S) & 1) ^ 1);
  }

  // The next work-list entry: the first CTA of the cluster takes it and
  // hands it to every CTA (itself included).
  __device__ int take_ticket(int& tki, bool& ok) {
    const int slot = tki & 1;
    const uint32_t ph = static_cast<uint32_t>(tki >> 1) & 1u;
    ++tki;
    if (rank == 0) {
      if (!(ok = warp_wait(&C.tk_empty[slot], ph ^ 1u))) return 0x7fffffff;
      int t = 0;
      if (lane == 0) t = atomicAdd(P.ws.ticket, 1);
      t = __shfl_sync(0xffffffffu, t, 0);
      if (lane < cs) st_async(peer(&C.tk[slot], lane), t, peer(&C.tk_full[slot], lane));
    }
    if (!(ok = warp_wait(&C.tk_full[slot], ph))) return 0x7fffffff;
    int t = 0;
    if (lane == 0) {
      t = C.tk[slot];
      mbar_expect_tx(&C.tk_full[slot], 4u);              // armed for the slot's next ticket
      mbar_arrive_peer(peer(&C.tk_empty[slot], 0));
    }
    return __shfl_sync(0xffffffffu, t, 0);
  }

  // Issue the re-reads of the waiting sequences whose turn has come: lag_rows
  // rows after the sequence ended (long enough for the control warp to have
  // decided, normally), when kMaxPending sequences wait, or (all) at the end.
  __device__ bool insert_due(int& q, int& pend, int streamed, int rows, int& draws, bool all) {
    const int S = P.stages;
    while (pend < streamed) {
      const int rc = pend % kRecs;
      if (!all && rows - C.pend_end[rc] < lag_rows && streamed - pend < kMaxPending) return true;
      int res = 0, drw = 0, b = 0, pos = 0;
      float Kt = 0.f, Lt = 0.f, Gh = 0.f, Gl = 0.f;
      if (lane == 0) {
        const unsigned long long t0 = global_ns();
        while (true) {
          if (C.rec[rc].resolved == pend + 1) { res = 1; break; }
          if (static_cast<long long>(global_ns() - t0) > kDrainLimitNs) break;
          __nanosleep(64);
        }
        if (res) {
          __threadfence_block();
          const SeqRec& R = C.rec[rc];
          drw = R.draw; b = R.b; pos = R.a;
          Kt = R.Kt; Lt = R.Lt; Gh = R.Gh; Gl = R.Gl;
        } else {
          atomicOr(P.ws.err_word, 1u << 5 /* SV_ERR_TIMEOUT */);
        }
      }
      res = __shfl_sync(0xffffffffu, res, 0);
      if (!res) return false;
      drw = __shfl_sync(0xffffffffu, drw, 0);
      if (drw) {
        b = __shfl_sync(0xffffffffu, b, 0);
        pos = __shfl_sync(0xffffffffu, pos, 0);
        const unsigned char* srcT = row_ptr(b, pos, 0);
        const unsigned char* srcD = row_ptr(b, pos, 1);
        for (int c = 0; c < ndraw; ++c) {
          if (!acquire_slot(q)) return false;
          const int slot = q % S;
          const int rem = slice_bytes - c * kHalfBytes;
          const int bytes = rem < kHalfBytes ? max(rem, 0) : kHalfBytes;
          const long long off = static_cast<long long>(slice_lo) * ELT + static_cast<long long>(c) * kHalfBytes;
          unsigned char* dst = ring + static_cast<size_t>(slot) * kChunkBytes;
          if (lane == 0) {
            Desc& d = C.desc[slot];
            d.b = b; d.kb = 0; d.pos = pos; d.kind = 2;
            d.chunk = c; d.nchunks = ndraw; d.x = -1; d.rec = rc; d.seq = pend;
            d.u = 0.f; d.s = 0.f;
            d.K0 = Kt; d.L0 = Lt; d.G0 = Gh; d.G1 = Gl;
            if (P.bulk) mbar_expect_tx(&C.full[slot], static_cast<uint32_t>(2 * bytes));
          }
          fill(dst, srcT, off, bytes, &C.full[slot], false, 0);
          fill(dst + kHalfBytes, srcD, off, bytes, &C.full[slot], false, 0);
          if (!P.bulk) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&C.full[slot]);
          }
          ++q;
        }
        ++draws;
      }
      ++pend;
    }
    return true;
  }

  __device__ void produce() {
    const int S = P.stages;
    const int k = P.k;
    const int n_seqs = __ldcg(P.ws.n_seqs);
    const uint64_t evict_first = evict_first_policy();
    int q = 0, tki = 0, streamed = 0, rows = 0, draws = 0, pend = 0;
    bool ok = true;
    // the next sequence's work-list entry, tokens and uniforms are fetched one
    // sequence ahead so that a sequence start never waits on global memory
    auto fetch = [&](int tt, int2& s_, int& x_, float& u_) {
      s_ = make_int2(-1, 0);
      x_ = -1;
      u_ = 0.f;
      if (tt < n_seqs) {
        s_ = __ldcg(P.ws.seqs + tt);
        x_ = lane < s_.y ? __ldg(P.tokens + static_cast<size_t>(s_.x) * k + lane) : -1;
        u_ = (!GREEDY && lane <= k) ? __ldg(P.uniforms + static_cast<size_t>(s_.x) * (k + 1) + lane) : 0.f;
      }
    };
    // the first sequence of cluster i is entry i of the work list (the
    // shared counter starts after them): no ticket to wait for
    int t = static_cast<int>(blockIdx.x) / cs;
    int2 sq;
    int xj;
    float uj;
    fetch(t, sq, xj, uj);
    while (ok && t < n_seqs) {
      const int b = sq.x, kb = sq.y;
      const int rc = streamed % kRecs;
      // the next ticket is taken when this sequence's last row starts: late
      // enough that sequences keep going to whichever cluster frees up first
      // (longest first; taking it rows earlier measured slower), early enough
      // to hide the fetch behind that row
      int t_next = 0x7fffffff;
      int2 sq_next = make_int2(-1, 0);
      int xj_next = -1;
      float uj_next = 0.f;
      bool fetched = false;
      const float s_samp = __shfl_sync(0xffffffffu, uj, k);
      const int nrows = GREEDY ? kb + 1 : 2 * kb + 1;
      for (int r = 0; r < nrows && ok; ++r) {
        if (!(ok = insert_due(q, pend, streamed, rows, draws, false))) break;
        int pos, kind;
        if (GREEDY) { pos = r; kind = 0; }
        else if (r < 2 * kb) { pos = r >> 1; kind = r & 1; }
        else { pos = kb; kind = 0; }
        if (P.early_exit && cs == 1 && r > 0) {
          // early exit, one CTA per sequence: no peer to stay in step with, so
          // the rest of the sequence is dropped as soon as a rejection (or an
          // error) is known, without waiting for it
          int stop = 0;
          if (lane == 0) {
            const SeqRec& R = C.rec[rc];
            stop = (R.seq_tag == streamed && R.stop) ? 1 : 0;
          }
          if (__shfl_sync(0xffffffffu, stop, 0)) {
            if (!(ok = acquire_slot(q))) break;
            const int slot = q % S;
            if (lane == 0) {
              Desc& d = C.desc[slot];
              d.b = b; d.kb = kb; d.pos = pos; d.kind = 3;
              d.chunk = 0; d.nchunks = 1; d.x = -1; d.rec = rc; d.seq = streamed;
              d.u = 0.f; d.s = s_samp;
              mbar_arrive(&C.full[slot]);
              atomicAdd(P.ws.stats + kStatRowsSkipped, static_cast<unsigned long long>(nrows - r));
            }
            ++q;
            ++rows;
            break;
          }
        }
        if (P.early_exit && cs > 1 && kind == 0 && pos >= exit_lag) {
          // early exit in a cluster, decided the same way in every CTA: wait
          // for the control warp's decision on pair pos - exit_lag; if the
          // first rejection is at or before that pair, the rest of the
          // sequence is not read.  The test looks at the rejection's pair,
          // not at whether one has been seen by now, which would depend on
          // each CTA's timing.
          int stop = 0, seen = 0;
          if (lane == 0) {
            const unsigned long long t0 = global_ns();
            while (true) {
              const SeqRec& R = C.rec[rc];
              if (R.seq_tag == streamed && R.decided > pos - exit_lag) {
                __threadfence_block();
                stop = (R.a >= 0 && R.a <= pos - exit_lag) ? 1 : 0;
                seen = 1;
                break;
              }
              if (static_cast<long long>(global_ns() - t0) > kDrainLimitNs) break;
              __nanosleep(64);
            }
            if (!seen) atomicOr(P.ws.err_word, 1u << 5 /* SV_ERR_TIMEOUT */);
          }
          seen = __shfl_sync(0xffffffffu, seen, 0);
          stop = __shfl_sync(0xffffffffu, stop, 0);
          if (!(ok = seen != 0)) break;
          if (stop) {
            // the end marker: no data, it closes the sequence downstream
            if (!(ok = acquire_slot(q))) break;
            const int slot = q % S;
            if (lane == 0) {
              Desc& d = C.desc[slot];
              d.b = b; d.kb = kb; d.pos = pos; d.kind = 3;
              d.chunk = 0; d.nchunks = 1; d.x = -1; d.rec = rc; d.seq = streamed;
              d.u = 0.f; d.s = s_samp;
              mbar_arrive(&C.full[slot]);
              if (rank == 0)   // every CTA of the cluster skips the same rows: counted once
                atomicAdd(P.ws.stats + kStatRowsSkipped, static_cast<unsigned long long>(nrows - r));
            }
            ++q;
            ++rows;
            break;
          }
        }
        const int x = __shfl_sync(0xffffffffu, xj, pos < kb ? pos : 0);
        const float u = __shfl_sync(0xffffffffu, uj, pos < kb ? pos : 0);
        const unsigned char* src = row_ptr(b, pos, kind);
        for (int c = 0; c < nchunks && ok; ++c) {
          if (!(ok = acquire_slot(q))) break;
          const int slot = q % S;
          const int rem = slice_bytes - c * kChunkBytes;
          const int bytes = rem < kChunkBytes ? max(rem, 0) : kChunkBytes;
          const long long off = static_cast<long long>(slice_lo) * ELT + static_cast<long long>(c) * kChunkBytes;
          if (lane == 0) {
            Desc& d = C.desc[slot];
            d.b = b; d.kb = kb; d.pos = pos; d.kind = kind;
            d.chunk = c; d.nchunks = nchunks;
            d.x = pos < kb ? x : -1; d.rec = rc; d.seq = streamed;
            d.u = u; d.s = s_samp;
            if (P.bulk) mbar_expect_tx(&C.full[slot], static_cast<uint32_t>(bytes));
          }
          // streamed rows are marked first out of L2: keeping the pairs
          // (whose rejected one is read again a few chunks later) measured no
          // faster, the re-read mostly finding its lines either way
          fill(ring + static_cast<size_t>(slot) * kChunkBytes, src, off, bytes, &C.full[slot], true, evict_first);
          if (!P.bulk) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&C.full[slot]);
          }
          ++q;
          if (!fetched && r == nrows - 1) {
            t_next = take_ticket(tki, ok);
            fetch(t_next, sq_next, xj_next, uj_next);
            fetched = true;
          }
        }
        ++rows;
      }
      if (!ok) break;
      if (!fetched) {
        t_next = take_ticket(tki, ok);
        fetch(t_next, sq_next, xj_next, uj_next);
      }
      if (lane == 0) C.pend_end[rc] = rows;
      __syncwarp();
      ++streamed;
      t = t_next;
      sq = sq_next;
      xj = xj_next;
      uj = uj_next;
    }
    if (ok) insert_due(q, pend, streamed, rows, draws, true);
    // the end of the work (also after an error, so that every warp stops)
    if (acquire_slot(q)) {
      if (lane == 0) {
        C.desc[q % S].kind = -1;
        C.desc[q % S].x = draws;
        mbar_arrive(&C.full[q % S]);
      }
    }
  }

  // ======================= consumers =========================================
  // They never wait on each other: a finished row is published into a ring
  // of row buffers, a re-read's weights into a pair of mass arrays, and the
  // control warp takes it from there.

  // Timeline (consumer warp 0, lane 0): first and last chunk, chunks seen.
  __device__ void stamp_chunk(bool& first, unsigned long long& n) const {
    if (!P.timeline || warp != 0 || lane != 0) return;
    unsigned long long* t = P.timeline + static_cast<size_t>(blockIdx.x) * kTimelineSlots;
    const unsigned long long now = global_ns();
    if (!first) { t[1] = now; first = true; }
    t[2] = now;
    t[6] = ++n;
  }

  __device__ void consume() {
    bool tl_first = false;
    unsigned long long tl_n = 0;
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
      if (d.kind >= 0) stamp_chunk(tl_first, tl_n);
      if (d.kind < 0) {
        // tell the control warp that the work is over
        const int buf = rr % kRowBufs;
        if (!warp_wait(&C.row_free[buf], ((rr / kRowBufs) & 1) ^ 1)) return;
        if (warp == 0 && lane == 0) C.rows[buf].d = d;
        __syncwarp();
        if (lane == 0) mbar_arrive(&C.row_ready[buf]);
        return;
      }

      if (d.kind == 2) {
        // ---- a chunk of a pair's re-read: per-segment draw weights --------
        const int dp = dr & 1;
        if (d.chunk == 0 && !warp_wait(&C.draw_free[dp], ((dr >> 1) & 1) ^ 1)) return;
        const unsigned char* data = ring + static_cast<size_t>(slot) * kChunkBytes;
        const int rem = slice_bytes - d.chunk * kHalfBytes;
        const int nvec = (min(max(rem, 0), kHalfBytes) + 15) / 16;
        uint4 rt[kDrawVecsPerLane], rd[kDrawVecsPerLane];
#pragma unroll
        for (int j = 0; j < kDrawVecsPerLane; ++j) {
          const int v = warp * kDrawVecsPerWarp + j * 32 + lane;
          const bool in = v < nvec;
          rt[j] = in ? *reinterpret_cast<const uint4*>(data + static_cast<size_t>(v) * 16) : V::neg_inf();
          rd[j] = in ? *reinterpret_cast<const uint4*>(data + kHalfBytes + static_cast<size_t>(v) * 16)
                     : V::neg_inf();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&C.empty[slot]);
        const f2 cc = pack2(c2, c2), nkt = pack2(-d.K0, -d.K0), nlt = pack2(-d.L0, -d.L0);
        const f2 gh = pack2(d.G0, d.G0), gl = pack2(d.G1, d.G1);
        f2 accr[NV / 2], accp[NV / 2];
#pragma unroll
        for (int i = 0; i < NV / 2; ++i) { accr[i] = 0ull; accp[i] = 0ull; }
#pragma unroll
        for (int j = 0; j < kDrawVecsPerLane; ++j) {
          f2 zt[NV / 2], zd[NV / 2];
          V::pairs(rt[j], zt);
          V::pairs(rd[j], zd);
#pragma unroll
          for (int i = 0; i < NV / 2; ++i) {
            // max(0, p - q) as p (1 - 2^delta): no cancellation where p ~ q;
            // the same roundings as the scalar resid_weight of the walk
            f2 p;
            float w0, w1;
            resid_weight2(zt[i], zd[i], cc, nkt, nlt, gh, gl, p, w0, w1);
            accr[i] = add2(accr[i], pack2(w0, w1));
            accp[i] = add2(accp[i], p);
          }
        }
        float a0, a1, sr = 0.f, sp = 0.f;
#pragma unroll
        for (int i = 0; i < NV / 2; ++i) {
          unpack2(accr[i], a0, a1); sr += a0 + a1;
          unpack2(accp[i], a0, a1); sp += a0 + a1;
        }
        const float wr = warp_sum(sr), wp = warp_sum(sp);
        if (lane == 0) {
          C.rmass[dp][d.chunk * kConsumerWarps + warp] = wr;
          C.pmass[dp][d.chunk * kConsumerWarps + warp] = wp;
          if (timed_out) atomicOr(&C.draw_err[dp], 1);
          if (warp == 0 && d.chunk == d.nchunks - 1) C.draw_rec[dp] = d.rec;
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
      const int rem = d.kind == 3 ? 0 : slice_bytes - d.chunk * kChunkBytes;   // an end marker is empty
      const int nvec = (min(max(rem, 0), kChunkBytes) + 15) / 16;
      uint4 raw[kVecsPerLane];
#pragma unroll
      for (int j = 0; j < kVecsPerLane; ++j) {
        const int v = warp * kVecsPerWarp + j * 32 + lane;
        raw[j] = v < nvec ? *reinterpret_cast<const uint4*>(data + static_cast<size_t>(v) * 16) : V::neg_inf();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&C.empty[slot]);   // the slot is free again

      const int seg = d.chunk * kConsumerWarps + warp;
      const int seg_base = slice_lo + seg * kSegElems;
      if (timed_out) rBad |= 2;
      // the drafted token's logit
      if (d.x >= 0 && d.x < P.V && !GREEDY) {
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
      // Each lane keeps its own running state over the row (rM, rArg / rK,
      // rS relative to its own maximum); the warp combines once, at the row
      // end, and per chunk only for the bonus row, whose per-segment sums the
      // draw needs.
      if (GREEDY) {
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
        if (lm > rM) { rM = lm; rArg = li; }   // chunks come in index order: ties keep the first
        rBad |= bad;
      } else {
        const float lm = V::vmax(raw);
        float ks = -INFINITY, ls = 0.f;
        if (lm > -INFINITY) {
          ks = __fmul_rn(lm, c2);      // fl(m c), used identically wherever rescaled
          const f2 cc = pack2(c2, c2), nk = pack2(-ks, -ks);
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
          float a0, a1;
#pragma unroll
          for (int i = 0; i < NV / 2; ++i) { unpack2(acc[i], a0, a1); ls += a0 + a1; }
          // NaN logits make ls NaN: caught at the row end
          if (ks > rK) { rS = rS * fast_exp2(__fsub_rn(rK, ks)) + ls; rK = ks; }
          else         { rS += ls * fast_exp2(__fsub_rn(ks, rK)); }
        } else {
          // no finite logit in this lane's part: only NaN can still hide here
          int nan_seen = 0;
#pragma unroll
          for (int j = 0; j < kVecsPerLane; ++j) {
            float z[NV];
            V::unpack(raw[j], z);
#pragma unroll
            for (int e = 0; e < NV; ++e) nan_seen |= (z[e] != z[e]);
          }
          rBad |= nan_seen;
        }
        rM = fmaxf(rM, lm);
        if (d.kind == 0 && d.pos == d.kb && seg < kMaxChunks * kConsumerWarps) {
          // bonus row: the segment's (fl(m c), sum) for the draw
          const float wm = from_ordered_key(__reduce_max_sync(0xffffffffu, ordered_key(lm)));
          const float Ks = wm > -INFINITY ? __fmul_rn(wm, c2) : -INFINITY;
          const float ss = warp_sum(ks > -INFINITY ? ls * fast_exp2(__fsub_rn(ks, Ks)) : 0.f);
          if (lane == 0) {
            RB.segK[seg] = Ks;
            RB.segS[seg] = ss;
          }
        }
      }

      if (d.chunk == d.nchunks - 1) {
        // publish the row: this warp's state, the descriptor (warp 0)
        float wM, wK = -INFINITY, wS = 0.f;
        int wArg = 0x7fffffff;
        if (GREEDY) {
          wM = rM;
          wArg = rArg;
          warp_argmax(wM, wArg);
        } else {
          wM = from_ordered_key(__reduce_max_sync(0xffffffffu, ordered_key(rM)));
          wK = wM > -INFINITY ? __fmul_rn(wM, c2) : -INFINITY;   // = the largest lane rK
          wS = warp_sum(rK > -INFINITY ? rS * fast_exp2(__fsub_rn(rK, wK)) : 0.f);
        }
        const int wBad = static_cast<int>(__reduce_or_sync(0xffffffffu, static_cast<unsigned>(rBad)));
        if (lane == 0) {
          RB.wK[warp] = wK; RB.wS[warp] = wS; RB.wM[warp] = wM; RB.wArg[warp] = wArg; RB.wBad[warp] = wBad;
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

  // The segment holding the target weight `tgt` among `nseg` masses (index
  // order); seg_t is what is left of tgt at the segment's start.  Past the
  // end (rounding) it is the last segment with positive mass.
  template <typename T>
  __device__ void locate(const T* mass, int nseg, double tgt, int& seg, double& seg_t) const {
    const int per = (nseg + 31) / 32;
    const int g0 = min(nseg, lane * per), g1 = min(nseg, g0 + per);
    double gs = 0.0;
    for (int i = g0; i < g1; ++i) gs += static_cast<double>(mass[i]);
    const double incl = warp_incl_scan(gs, lane);
    const double excl = incl - gs;
    const unsigned hit = __ballot_sync(0xffffffffu, gs > 0.0 && tgt < incl);
    const unsigned posg = __ballot_sync(0xffffffffu, gs > 0.0);
    const int owner = hit ? (__ffs(hit) - 1) : (posg ? 31 - __clz(posg) : -1);
    seg = -1;
    seg_t = 0.0;
    if (owner >= 0 && lane == owner) {
      double run = excl, last_run = excl;
      int last = -1;
      for (int i = g0; i < g1; ++i) {
        const double m = static_cast<double>(mass[i]);
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

  // Which CTA's slice holds the target: each lane < cs holds slice weight w
  // (the same values, in the same lanes, in every CTA, so every CTA agrees).
  // Returns the rank (-1 if no slice has weight) and, in that lane's terms,
  // what is left of the target at the slice's start.
  __device__ int slice_owner(double w, double s, double& tot, double& t_loc) const {
    const double incl = warp_incl_scan(w, lane);
    tot = __shfl_sync(0xffffffffu, incl, 31);
    const double tgt = s * tot;
    const unsigned hit = __ballot_sync(0xffffffffu, w > 0.0 && tgt < incl);
    const unsigned any = __ballot_sync(0xffffffffu, w > 0.0);
    const int owner = hit ? (__ffs(hit) - 1) : (any ? 31 - __clz(any) : -1);
    t_loc = __shfl_sync(0xffffffffu, tgt - (incl - w), owner >= 0 ? owner : 0);
    return owner;
  }

  // Walk NSTEPS x 32 vectors starting at vector v0, a warp inclusive scan
  // per step, to the token where the running weight passes t.
  // RESID: weights max(0, p - q); else p.
  template <int NSTEPS, bool RESID>
  __device__ int walk(int v0, double t, const unsigned char* rowT, const unsigned char* rowD,
                      float Kt, float Lt, float Gh, float Gl) const {
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
        float p;
        if (RESID) w[e] = resid_weight(zt[e], zd[e], P.c2, Kt, Lt, Gh, Gl, p);
        else w[e] = fast_exp2(__fsub_rn(__fmaf_rn(zt[e], P.c2, -Kt), Lt));
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

  // Outputs of a settled sequence (written by one CTA of the cluster).
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
      if (ok) v = j < a ? R.tok[j] : (j == a ? y : -1);
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
    }
    __syncwarp();
  }

  // Hand a walk to the walker warps, in turn (lane 0 of the control warp):
  // walks of sequences that finish together then overlap.  Waits, bounded,
  // while the chosen ring is full: the walkers always make progress.
  int wsel_ = 0;
  __device__ void push_walk(const WalkReq& r) {
    if (lane == 0) {
      const int w = wsel_;
      wsel_ = (wsel_ + 1) % kWalkers;
      const unsigned long long t0 = global_ns();
      while (C.wreq_tail[w] - C.wreq_head[w] >= kWalkReqs) {
        if (static_cast<long long>(global_ns() - t0) > kDrainLimitNs) {
          atomicOr(P.ws.err_word, 1u << 5 /* SV_ERR_TIMEOUT */);
          break;
        }
        __nanosleep(64);
      }
      const int tail = C.wreq_tail[w];
      C.wreq[w][tail % kWalkReqs] = r;
      __threadfence_block();
      C.wreq_tail[w] = tail + 1;
    }
    __syncwarp();
  }

  // ======================= walker warps ======================================
  // The only warps of the CTA that wait on logits read from global memory
  // outside the staging ring: the walk inside the drawn segment, then the
  // sequence's outputs.  Nothing waits for them but the reuse of a record.

  __device__ void walker(int w) {
    int head = 0;
    unsigned long long idle_since = 0;
    while (true) {
      int tail = 0, done = 0;
      if (lane == 0) { done = C.ctl_done; tail = C.wreq_tail[w]; }
      tail = __shfl_sync(0xffffffffu, tail, 0);
      done = __shfl_sync(0xffffffffu, done, 0);
      if (head == tail) {
        if (done) {
          // the control warp has left: take what it pushed before leaving
          if (lane == 0) tail = C.wreq_tail[w];
          tail = __shfl_sync(0xffffffffu, tail, 0);
          if (head == tail) {
            if (P.timeline && lane == 0)
              atomicMax(P.timeline + static_cast<size_t>(blockIdx.x) * kTimelineSlots + 4, global_ns());
            return;
          }
        } else {
          if (!idle_since) idle_since = global_ns();
          if (static_cast<long long>(global_ns() - idle_since) > 8 * kDrainLimitNs) {
            if (lane == 0) atomicOr(P.ws.err_word, 1u << 5 /* SV_ERR_TIMEOUT */);
            return;
          }
          __nanosleep(128);
          continue;
        }
      }
      idle_since = 0;
      __threadfence_block();
      const WalkReq r = C.wreq[w][head % kWalkReqs];
      int y = -1;
      if (r.v0 >= 0) {
        if (r.mode == 0)
          y = walk<kVecsPerLane, false>(r.v0, r.t, row_ptr(r.b, r.pos, 0), nullptr, r.K0, r.L0, 0.f, 0.f);
        else if (r.mode == 1)
          y = walk<kDrawVecsPerLane, true>(r.v0, r.t, row_ptr(r.b, r.pos, 0), row_ptr(r.b, r.pos, 1),
                                           r.K0, r.L0, r.Gh, r.Gl);
        else
          y = walk<kDrawVecsPerLane, false>(r.v0, r.t, row_ptr(r.b, r.pos, 0), nullptr, r.K0, r.L0, 0.f, 0.f);
      }
      if (lane == 0) C.rec[r.rec].y = y;
      __syncwarp();
      finish_sequence(r.rec);
      if (lane == 0) {
        C.rec[r.rec].open = 0;
        C.wreq_head[w] = head + 1;
      }
      __syncwarp();
      ++head;
    }
  }

  // This CTA's part of a finished row: its consumer warps combined.  Each
  // warp's K is fl(M_w c) of its own maximum, so the part's K is fl(M c).
  __device__ void local_part(const RowBuf& RB, RowPart& out) const {
    const bool in = lane < kConsumerWarps;
    const float m = in ? RB.wM[lane] : -INFINITY;
    const float M = from_ordered_key(__reduce_max_sync(0xffffffffu, ordered_key(m)));
    out.M = M;
    out.arg = GREEDY ? __reduce_min_sync(0xffffffffu, (in && m == M) ? RB.wArg[lane] : 0x7fffffff) : 0;
    out.bad = static_cast<int>(__reduce_or_sync(0xffffffffu, in ? static_cast<unsigned>(RB.wBad[lane]) : 0u));
    const float K = M > -INFINITY ? __fmul_rn(M, P.c2) : -INFINITY;
    out.K = K;
    const float wk = in ? RB.wK[lane] : -INFINITY;
    float v = (!GREEDY && wk > -INFINITY) ? RB.wS[lane] * fast_exp2(__fsub_rn(wk, K)) : 0.f;
#pragma unroll
    for (int o = kConsumerWarps / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    out.S = v;
    const int x = RB.d.x;
    out.has_zx = (!GREEDY && x >= slice_lo && x < slice_lo + slice_n) ? 1 : 0;
    out.zx = out.has_zx ? RB.zx : 0.f;
    out.pad = 0;
  }

  __device__ void send_row_part(int xs, const RowPart& pt) const {
    if (lane < cs) {
      const uint32_t dst = peer(&C.xrow[xs][rank], lane);
      const uint32_t bar = peer(&C.xrow_ready[xs], lane);
      st_async(dst, make_uint4(__float_as_uint(pt.M), __float_as_uint(pt.K), __float_as_uint(pt.S),
                               __float_as_uint(pt.zx)), bar);
      st_async(dst + 16, make_uint4(static_cast<unsigned>(pt.arg), static_cast<unsigned>(pt.bad),
                                    static_cast<unsigned>(pt.has_zx), 0u), bar);
    }
    __syncwarp();
  }

  // Every CTA's part of the row has arrived: combine, decide, and settle
  // the sequence if this was its last row and no re-read follows.
  __device__ void finish_row(int buf, int xs) {
    const float c2 = P.c2;
    const RowBuf& RB = C.rows[buf];
    const Desc d = RB.d;
    const bool in = lane < cs;
    RowPart pt{};
    if (in) pt = C.xrow[xs][lane];
    const float pm = in ? pt.M : -INFINITY;
    const float M = from_ordered_key(__reduce_max_sync(0xffffffffu, ordered_key(pm)));
    const int arg = GREEDY ? __reduce_min_sync(0xffffffffu, (in && pm == M) ? pt.arg : 0x7fffffff) : 0;
    const int bad = static_cast<int>(__reduce_or_sync(0xffffffffu, in ? static_cast<unsigned>(pt.bad) : 0u));
    const float pk = in ? pt.K : -INFINITY;
    const float K = M > -INFINITY ? __fmul_rn(M, c2) : -INFINITY;   // = the largest part K
    float sv = (!GREEDY && pk > -INFINITY) ? pt.S * fast_exp2(__fsub_rn(pk, K)) : 0.f;
    for (int o = cs >> 1; o > 0; o >>= 1) sv += __shfl_xor_sync(0xffffffffu, sv, o);
    const float Ssum = __shfl_sync(0xffffffffu, sv, 0);
    const unsigned hz = __ballot_sync(0xffffffffu, in && pt.has_zx);
    const float zx = __shfl_sync(0xffffffffu, in ? pt.zx : 0.f, hz ? __ffs(hz) - 1 : 0);
    // every part is in registers: arm the slot for its next row and let the
    // senders reuse it
    if (cs > 1) {
      if (lane == 0) mbar_expect_tx(&C.xrow_ready[xs], static_cast<uint32_t>(cs * sizeof(RowPart)));
      if (in) mbar_arrive_peer(peer(&C.xrow_free[xs], lane));
    }
    const float L = log2f(Ssum);
    SeqRec& R = C.rec[d.rec];
    const size_t b = static_cast<size_t>(d.b);
    const bool diag = P.diag && rank == 0;   // one CTA of the cluster writes the diagnostics
    const bool marker = (d.kind == 3);      // the sequence was cut short after a rejection
    const bool last = (d.kind == 0 && d.pos == d.kb) || marker;
    int bonus = 0, settle = 0;
    if (lane == 0 && !marker) {
      if (d.pos == 0 && d.kind == 0) {
        // first row of the sequence: open its record
        R.b = d.b; R.kb = d.kb; R.a = -1; R.err = 0; R.y = -1; R.zero_resid = 0;
        R.open = 1; R.draw = 0; R.s = d.s;
        R.decided = 0; R.stop = 0;
        __threadfence_block();
        R.seq_tag = d.seq;
      }
      if (bad & 2) R.err |= kErrTimeout;
      if (d.pos < d.kb) R.tok[d.pos] = d.x;
      if (d.pos < d.kb && (d.x < 0 || d.x >= P.V)) R.err |= kErrBadToken;
      if (GREEDY) {
        if ((bad & 1) || !(M > -INFINITY)) R.err |= kErrNonfinite;
        if (diag) P.ws.m_t[b * (P.k + 1) + d.pos] = M;
        if (d.pos < d.kb) {
          const bool acc = (d.x == arg);
          if (diag) P.ws.alpha[b * P.k + d.pos] = acc ? 1.f : 0.f;
          if (!acc && R.a < 0) { R.a = d.pos; R.y = arg; }
        } else if (R.a < 0) {
          R.y = arg;
        }
      } else {
        if ((bad & 1) || !(isfinite(M) && isfinite(Ssum) && Ssum > 0.f)) R.err |= kErrNonfinite;
        if (d.kind == 0) {
          if (diag) {
            P.ws.m_t[b * (P.k + 1) + d.pos] = M;
            P.ws.L_t[b * (P.k + 1) + d.pos] = log2f(Ssum);
          }
          C.pairK = K; C.pairL = L; C.pairZx = zx; C.pairS = Ssum;
        } else if (diag) {
          P.ws.m_d[b * P.k + d.pos] = M;
          P.ws.L_d[b * P.k + d.pos] = log2f(Ssum);
        }
        if (d.kind == 1 && !R.err) {
          // the pair is complete: acceptance test of draft d.pos.  With
          // G = Gh + Gl the log2 ratio of the target's to the draft's
          // normaliser, log2 (q(x) / p(x)) = delta = (z_d(x) - z_t(x)) c + G
          // (the residual weights' delta) and alpha = min(1, 2^-delta)
          const float zt = C.pairZx, zd = zx;
          float Gh, Gl;
          log2_ratio(C.pairK, C.pairS, K, Ssum, Gh, Gl);
          float alpha;
          if (zt == -INFINITY) alpha = 0.f;               // p(x) = 0
          else if (zd == -INFINITY) alpha = 1.f;          // q(x) = 0 < p(x)
          else {
            const float delta = __fadd_rn(__fmaf_rn(__fsub_rn(zd, zt), c2, Gh), Gl);
            alpha = delta <= 0.f ? 1.f : exp2f(-delta);
          }
          if (diag) P.ws.alpha[b * P.k + d.pos] = alpha;
          if (!(d.u < alpha) && R.a < 0) {
            // first rejection: the pair is read again for the residual draw
            R.a = d.pos;
            R.Kt = C.pairK; R.Lt = C.pairL;   // the target row's log2 S, taken only here
            R.Gh = Gh; R.Gl = Gl;
          }
        } else if (last && R.a < 0 && !R.err) {
          bonus = 1;   // every draft accepted: the bonus draw
        }
      }
      if ((GREEDY && d.pos < d.kb) || (!GREEDY && d.kind == 1)) {
        // pair d.pos is decided: the producer may stop streaming this sequence
        R.stop = (R.a >= 0 || R.err) ? 1 : 0;
        __threadfence_block();
        R.decided = d.pos + 1;
      }
    }
    if (lane == 0) {
      if (last) {
        // the outcome is known: tell the producer whether a re-read follows
        R.draw = (!GREEDY && R.a >= 0 && !R.err) ? 1 : 0;
        __threadfence_block();
        R.resolved = d.seq + 1;
        settle = R.draw ? 0 : 1;
      }
    }
    bonus = __shfl_sync(0xffffffffu, bonus, 0);
    settle = __shfl_sync(0xffffffffu, settle, 0);
    __syncwarp();
    int fin_rank = 0;
    if (bonus) {
      // the slice holding s * S from every CTA's (K, S); inside it, the
      // segment from the sums kept while streaming, then one segment of the
      // bonus row is read again
      const double w = (in && pk > -INFINITY)
                           ? static_cast<double>(pt.S) * static_cast<double>(fast_exp2(__fsub_rn(pk, K) - L))
                           : 0.0;
      double tot, t_loc;
      const int owner = slice_owner(w, static_cast<double>(d.s), tot, t_loc);
      fin_rank = owner >= 0 ? owner : 0;
      if (owner == rank) {
        const int nseg = nchunks * kConsumerWarps;
        for (int sg = lane; sg < nseg; sg += 32) {
          const float ks = RB.segK[sg];
          C.bmass[sg] = ks == -INFINITY ? 0.0
                        : static_cast<double>(RB.segS[sg]) * static_cast<double>(fast_exp2(__fsub_rn(ks, K) - L));
        }
        __syncwarp();
        int seg;
        double seg_t;
        locate(C.bmass, nseg, t_loc, seg, seg_t);
        if (lane == 0 && P.diag) P.ws.mass[b * (P.k + 1) + d.kb] = static_cast<float>(tot);
        WalkReq wr;
        wr.rec = d.rec; wr.mode = 0; wr.v0 = seg >= 0 ? v_lo + seg * kVecsPerWarp : -1;
        wr.b = d.b; wr.pos = d.kb; wr.pad = 0; wr.t = seg_t;
        wr.K0 = K; wr.L0 = L; wr.Gh = 0.f; wr.Gl = 0.f;
        push_walk(wr);       // the walker writes the outputs and frees the record
        settle = 0;
      }
      __syncwarp();
    }
    if (settle) {
      if (rank == fin_rank) finish_sequence(d.rec);
      if (lane == 0) R.open = 0;
      __syncwarp();
    }
  }

  // Every CTA's masses of a re-read have arrived: the slice, then the
  // segment, then the token; the CTA whose slice holds it settles the sequence.
  __device__ void finish_draw(int dp, int xs) {
    int rc = 0;
    if (lane == 0) rc = C.draw_rec[dp];
    rc = __shfl_sync(0xffffffffu, rc, 0);
    SeqRec& R = C.rec[rc];
    const bool in = lane < cs;
    double r = 0.0, p = 0.0;
    int err = 0;
    if (in) {
      const DrawPart& dpt = C.xdraw[xs][lane];
      r = dpt.r; p = dpt.p; err = dpt.err;
    }
    err = warp_or(err);
    const double rtot = warp_sum(r);
    if (lane == 0) mbar_expect_tx(&C.xdraw_ready[xs], static_cast<uint32_t>(cs * sizeof(DrawPart)));
    if (in) mbar_arrive_peer(peer(&C.xdraw_free[xs], lane));
    // exact arithmetic rules a zero residual out (a rejection implies p > q
    // somewhere); if rounding leaves none, the draw is from p_a (counted)
    const bool resid = rtot > 0.0;
    double tot, t_loc;
    const int owner = slice_owner(resid ? r : p, static_cast<double>(R.s), tot, t_loc);
    const int fin_rank = owner >= 0 ? owner : 0;
    if (lane == 0) {
      if (err) R.err |= kErrTimeout;
      R.zero_resid = resid ? 0 : 1;
    }
    __syncwarp();
    if (owner == rank) {
      const int nseg = ndraw * kConsumerWarps;
      int seg;
      double seg_t;
      locate(resid ? C.rmass[dp] : C.pmass[dp], nseg, t_loc, seg, seg_t);
      if (lane == 0 && P.diag) P.ws.mass[static_cast<size_t>(R.b) * (P.k + 1) + R.a] = static_cast<float>(tot);
      WalkReq wr;
      wr.rec = rc; wr.mode = resid ? 1 : 2; wr.v0 = seg >= 0 ? v_lo + seg * kDrawVecsPerWarp : -1;
      wr.b = R.b; wr.pos = R.a; wr.pad = 0; wr.t = seg_t;
      wr.K0 = R.Kt; wr.L0 = R.Lt; wr.Gh = R.Gh; wr.Gl = R.Gl;
      push_walk(wr);       // the walker writes the outputs and frees the record
    } else {
      if (rank == fin_rank) finish_sequence(rc);
      if (lane == 0) R.open = 0;
      __syncwarp();
    }
  }

  __device__ void control() {
    control_loop();
    if (P.timeline && lane == 0) P.timeline[static_cast<size_t>(blockIdx.x) * kTimelineSlots + 3] = global_ns();
    __syncwarp();
    if (lane == 0) { __threadfence_block(); C.ctl_done = 1; }
  }

  __device__ void control_loop() {
    // rows: parts are sent as soon as a row is local, up to kXRing ahead of
    // the oldest row whose exchange is not complete; rows finish in order
    int rs = 0, rf = 0, end_row = -1;
    int di = 0, dphase = 0;       // draws: 0 wait local, 1 send, 2 wait every part
    double dR = 0.0, dP = 0.0;
    int dErr = 0;
    int end_draws = -1;           // re-reads in all, known at the end of the work
    unsigned long long idle_since = 0;
    while (true) {
      bool progressed = false;
      while (end_row < 0 && rs - rf < kXRing) {
        const int buf = rs % kRowBufs;
        const int xs = rs % kXRing;
        if (!probe(&C.row_ready[buf], static_cast<uint32_t>(rs / kRowBufs) & 1u)) break;
        if (C.rows[buf].d.kind < 0) {
          end_row = rs;
          progressed = true;
          break;
        }
        if (cs > 1 && !probe(&C.xrow_free[xs], (static_cast<uint32_t>(rs / kXRing) & 1u) ^ 1u)) break;
        RowPart mine;
        local_part(C.rows[buf], mine);
        if (cs > 1) {
          send_row_part(xs, mine);
        } else {
          // a cluster of one: the part is the row
          if (lane == 0) C.xrow[xs][0] = mine;
          __syncwarp();
        }
        ++rs;
        progressed = true;
      }
      if (rf < rs) {
        const int buf = rf % kRowBufs;
        const int xs = rf % kXRing;
        if (cs == 1 || probe(&C.xrow_ready[xs], static_cast<uint32_t>(rf / kXRing) & 1u)) {
          // a sequence's first row waits until its record is free again
          int free_rec = 1;
          if (lane == 0) {
            const Desc& d = C.rows[buf].d;
            if (d.pos == 0 && d.kind == 0 && C.rec[d.rec].open) free_rec = 0;
          }
          free_rec = __shfl_sync(0xffffffffu, free_rec, 0);
          if (free_rec) {
            finish_row(buf, xs);
            __syncwarp();
            if (lane == 0) mbar_arrive(&C.row_free[buf]);
            ++rf;
            progressed = true;
          }
        }
      }
      if (end_row >= 0 && rf == end_row && end_draws < 0) end_draws = C.rows[end_row % kRowBufs].d.x;
      {
        const int dp = di & 1;
        const int xs = di % kXRing;
        if (dphase == 0 && (end_draws < 0 || di < end_draws) &&
            probe(&C.draw_ready[dp], static_cast<uint32_t>(di >> 1) & 1u)) {
          const int nseg = ndraw * kConsumerWarps;
          double r = 0.0, p = 0.0;
          for (int sg = lane; sg < nseg; sg += 32) {
            r += static_cast<double>(C.rmass[dp][sg]);
            p += static_cast<double>(C.pmass[dp][sg]);
          }
          dR = warp_sum(r);
          dP = warp_sum(p);
          if (lane == 0) { dErr = C.draw_err[dp]; C.draw_err[dp] = 0; }
          dErr = __shfl_sync(0xffffffffu, dErr, 0);
          dphase = 1;
          progressed = true;
        }
        if (dphase == 1 && probe(&C.xdraw_free[xs], (static_cast<uint32_t>(di / kXRing) & 1u) ^ 1u)) {
          if (lane < cs) {
            const uint32_t dst = peer(&C.xdraw[xs][rank], lane);
            const uint32_t bar = peer(&C.xdraw_ready[xs], lane);
            const unsigned long long rb = static_cast<unsigned long long>(__double_as_longlong(dR));
            const unsigned long long pb = static_cast<unsigned long long>(__double_as_longlong(dP));
            st_async(dst, make_uint4(static_cast<unsigned>(rb), static_cast<unsigned>(rb >> 32),
                                     static_cast<unsigned>(pb), static_cast<unsigned>(pb >> 32)), bar);
            st_async(dst + 16, make_uint4(static_cast<unsigned>(dErr), 0u, 0u, 0u), bar);
          }
          __syncwarp();
          dphase = 2;
          progressed = true;
        }
        if (dphase == 2 && probe(&C.xdraw_ready[xs], static_cast<uint32_t>(di / kXRing) & 1u)) {
          finish_draw(dp, xs);
          __syncwarp();
          if (lane == 0) mbar_arrive(&C.draw_free[dp]);
          ++di;
          dphase = 0;
          progressed = true;
        }
      }
      if (end_draws >= 0 && di >= end_draws) return;
      if (progressed) {
        idle_since = 0;
      } else {
        if (!idle_since) idle_since = global_ns();
        if (static_cast<long long>(global_ns() - idle_since) > 4 * kDrainLimitNs) {
          if (lane == 0) atomicOr(P.ws.err_word, 1u << 5 /* SV_ERR_TIMEOUT */);
          return;
        }
        // wait in hardware, briefly, for what the rows need next
        if (end_row >= 0) __nanosleep(64);
        else if (rf < rs && cs > 1) mbar_park(&C.xrow_ready[rf % kXRing], static_cast<uint32_t>(rf / kXRing) & 1u, 300u);
        else mbar_park(&C.row_ready[rs % kRowBufs], static_cast<uint32_t>(rs / kRowBufs) & 1u, 300u);
      }
    }
  }
};

template <int ELT, bool GREEDY>
__global__ void __launch_bounds__(kThreads, 1)
verify_kernel(const VerifyParams P) {
  extern __shared__ __align__(1024) unsigned char smem[];
  Ctrl& C = *reinterpret_cast<Ctrl*>(smem);
  unsigned char* ring = smem + kCtrlBytes;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cs = cluster_ctas();
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
      mbar_init(&C.tk_full[r], 1);
      mbar_init(&C.tk_empty[r], cs);
      C.draw_err[r] = 0;
    }
    // the data barriers complete on one local arrival (made when a slot is
    // armed) plus the bytes of the asynchronous stores of every sender
    for (int x = 0; x < kXRing; ++x) {
      mbar_init(&C.xrow_ready[x], 1);
      mbar_init(&C.xrow_free[x], cs);
      mbar_init(&C.xdraw_ready[x], 1);
      mbar_init(&C.xdraw_free[x], cs);
    }
    for (int r = 0; r < kRecs; ++r) {
      C.rec[r].open = 0; C.rec[r].resolved = 0;
      C.rec[r].seq_tag = -1; C.rec[r].decided = 0; C.rec[r].stop = 0;
    }
    for (int w = 0; w < kWalkers; ++w) { C.wreq_head[w] = 0; C.wreq_tail[w] = 0; }
    C.ctl_done = 0;
    fence_mbar_init();
    for (int r = 0; r < 2; ++r) mbar_expect_tx(&C.tk_full[r], 4u);
    for (int x = 0; x < kXRing; ++x) {
      mbar_expect_tx(&C.xrow_ready[x], static_cast<uint32_t>(cs * sizeof(RowPart)));
      mbar_expect_tx(&C.xdraw_ready[x], static_cast<uint32_t>(cs * sizeof(DrawPart)));
    }
  }
  unsigned long long* tl = P.timeline ? P.timeline + static_cast<size_t>(blockIdx.x) * kTimelineSlots : nullptr;
  if (tl && tid == 0) tl[7] = global_ns();
  cluster_sync();                   // every CTA's barriers exist before anyone arrives on them
  grid_dependency_wait();           // the work list of plan_kernel is ready
  if (tl && tid == 0) tl[0] = global_ns();
  {
    Verifier<ELT, GREEDY> v(P, C, ring, lane, warp, cs, cluster_rank());
    if (warp < kConsumerWarps) v.consume();
    else if (warp == kConsumerWarps) v.produce();
    else if (warp == kConsumerWarps + 1) v.control();
    else v.walker(warp - kConsumerWarps - 2);
  }
  cluster_sync();                   // nobody leaves while a peer may still reach its shared memory
  if (tl && tid == 0) tl[5] = global_ns();
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
  const void* fns[4] = {reinterpret_cast<const void*>(&verify_kernel<2, false>),
                        reinterpret_cast<const void*>(&verify_kernel<4, false>),
                        reinterpret_cast<const void*>(&verify_kernel<2, true>),
                        reinterpret_cast<const void*>(&verify_kernel<4, true>)};
  for (const void* f : fns) {
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t query_ctas_per_sm(int smem_bytes, int* out) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, verify_kernel<2, false>, kThreads,
                                                       static_cast<size_t>(smem_bytes));
}

namespace {
void verify_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute (&attr)[2], int cluster, int ctas,
                   int smem_bytes, cudaStream_t s) {
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg = cudaLaunchConfig_t{};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
}
}  // namespace

cudaError_t query_max_clusters(int cluster, int smem_bytes, int* out) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  verify_config(cfg, attr, cluster, cluster, smem_bytes, nullptr);
  cfg.numAttrs = 1;
  cfg.attrs = attr + 1;   // the cluster shape alone
  return cudaOccupancyMaxActiveClusters(out, reinterpret_cast<const void*>(&verify_kernel<2, false>), &cfg);
}

cudaError_t launch_verify(const VerifyParams& params, int ctas, int smem_bytes, cudaStream_t s) {
  NvtxRange range("spec_verify");
  if (params.pieces) return launch_pieces(params, s);   // its own plan, in batch order
  VerifyParams p = params;
  p.ctas = ctas;   // the work-list kernel starts the ticket counter after every cluster's first
  plan_kernel<<<1, kPlanThreads, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  verify_config(cfg, attr, p.cluster, ctas, smem_bytes, s);
  if (p.greedy) {
    if (p.elt == 2) return cudaLaunchKernelEx(&cfg, verify_kernel<2, true>, p);
    return cudaLaunchKernelEx(&cfg, verify_kernel<4, true>, p);
  }
  if (p.elt == 2) return cudaLaunchKernelEx(&cfg, verify_kernel<2, false>, p);
  return cudaLaunchKernelEx(&cfg, verify_kernel<4, false>, p);
}

cudaError_t launch_compact(int B, int k, const int* out_tokens, const int* out_len,
                           int* packed, int* offsets, cudaStream_t s) {
  NvtxRange range("spec_verify_compact");
  compact_kernel<<<1, kCompactThreads, 0, s>>>(B, k, out_tokens, out_len, packed, offsets);
  return cudaGetLastError();
}

cudaError_t launch_debug(const Workspace& ws, int B, int k, int greedy, float inv_T, double* lse_t,
                         double* lse_d, double* accept_prob, double* mass, cudaStream_t s) {
  NvtxRange range("spec_verify_debug");
  const int n = B * (k + 1);
  debug_kernel<<<(n + 255) / 256, 256, 0, s>>>(ws, B, k, greedy, inv_T, lse_t, lse_d, accept_prob, mass);
  return cudaGetLastError();
}

cudaError_t launch_init_workspace(const Workspace& ws, cudaStream_t s) {
  init_workspace_kernel<<<1, 32, 0, s>>>(ws);
  return cudaGetLastError();
}

}  // namespace sv
