// Piece-streaming verification: the same rule as verify_kernel, scheduled for
// small batches.
//
// verify_kernel gives a whole sequence to one CTA cluster, so at a few
// hundred sequences the last ones to finish leave most SMs idle.  Here the
// unit of work is a piece of a row: every needed row (target rows 0..k_b,
// draft rows 0..k_b-1 of each sequence) is cut into np pieces of at most one
// 64 KB staging slot, and the units are dealt round-robin to persistent CTAs
// (one per SM) in the order of plan_kernel's work list (longest sequences
// first, each sequence's pieces together), so every CTA streams the same
// number of bytes and none waits for a ticket.  Nothing waits for another
// CTA on the data path: the sequence is decided by whichever CTA reduces its
// last piece (an acq_rel counter per sequence):
//
//   piece     consumer warps: per warp (M, fl(M c), sum 2^(z c - K)) of its
//             segment (greedy: maximum and first argmax), and the logit of
//             the drafted token if it falls there;  control warps: the
//             piece's part written out, the sequence's counter;
//   sequence  a decider warp of the CTA completing it: every row's
//             (M, K, S, L) from its pieces in piece order, every acceptance
//             test alpha = min(1, p(x)/q(x)), u < alpha, the first rejection
//             a; if every draft was accepted, the bonus token by inverse CDF
//             over the bonus row's segment sums (kept while streaming) and a
//             walk of one segment; else the rejected pair is read again;
//   re-read   the pair in nr pieces (target and draft halves of one slot),
//             handed round-robin to the CTAs' mailboxes and taken before new
//             rows: per-segment masses of max(0, p - q) = p (1 - 2^delta);
//             the CTA completing the last piece finds the segment holding
//             s S and walks it.
// A sequence's outputs are written once every row is reduced, so an invalid
// row anywhere in 0..k_b fails it, as in verify_kernel.  Every reduction runs
// in a fixed order, so the outputs are deterministic and equal to
// verify_kernel's up to the summation order of the row sums.
//
// The rule is the standard speculative-sampling rule read into "Accelerating
// RL Post-Training Rollouts via System-Integrated Speculative Decoding", §2
// core mechanism: accept with min(1, p/q), stop at the first rejection,
// resample from max(0, p - q) or draw the bonus token from the last target
// row.

#include <cuda_runtime.h>
#include <cstdint>
#include <cmath>

#include "sv_internal.h"
#include "sv_device.cuh"

namespace sv {
namespace {

constexpr int kCtlWarps = 2;     // control warps (alternate units), each with its decider warp
constexpr int kPThreads = (kConsumerWarps + 1 + 2 * kCtlWarps) * 32;   // + producer
constexpr int kWarpProducer = kConsumerWarps;
constexpr int kWarpCtl0 = kConsumerWarps + 1;
constexpr int kWarpDec0 = kConsumerWarps + 1 + kCtlWarps;
constexpr int kCtrSettled = 32;  // sequences settled (a 128-byte line of its own)
constexpr int kUBufs = 8;        // unit results in flight between consumers and control warps
constexpr int kJobs = 64;        // decider jobs (ring)
constexpr int kSegs = kConsumerWarps;                     // segments per piece (one per consumer warp)
constexpr int kHalf = kChunkBytes / 2;                    // one row's half of a re-read slot
constexpr int kHalfVecsPerWarp = kHalf / 16 / kConsumerWarps;   // 128
constexpr int kHalfVecsPerLane = kHalfVecsPerWarp / 32;         // 4
constexpr int kMaxResid = 2 * kMaxChunks;                 // re-read pieces of a pair (rows up to 1 MiB)

enum : int { kErrBadTok = 1 << 3, kErrNonfin = 1 << 4, kErrTime = 1 << 5 };
enum : int { kJobSeq = 0, kJobResid = 1, kJobEnd = 2 };
constexpr int kMaxRows = 64;     // rows of a sequence: 2 k + 1 <= 63
constexpr int kScratch = 256;    // decider scratch: float4 piece parts, or doubles of segment weights x 2

// What a staging slot holds.
struct PDesc {
  int b, kb, pos, kind;        // kind 0 target, 1 draft, 2 re-read of a rejected pair, -1 end
  int piece, nbytes, r, x;     // r: row index (kinds 0/1); x: unused (-1)
  float K0, L0, G0, G1;        // re-read: target normaliser, log2 normaliser ratio (Gh + Gl)
};

// A unit's results: the descriptor and one float4 per consumer warp.
struct UBuf {
  PDesc d;
  float4 w[kConsumerWarps];
};

struct Job {
  int kind, r, b, pos;
  int rowkind, pad0, pad1, pad2;
};

struct PCtrl {
  uint64_t full[kPiecesStages], empty[kPiecesStages];
  uint64_t ufull[kUBufs], ufree[kUBufs];
  PDesc desc[kPiecesStages];
  UBuf ub[kUBufs];
  Job jobs[kCtlWarps][kJobs];   // control warp i -> decider warp i
  volatile int job_ready[kCtlWarps][kJobs];
  volatile int job_head[kCtlWarps];
  int job_tail[kCtlWarps];
  int gstart[33], gunits[33], gcount[33];   // per draft length L: first sequence, first unit, sequences
  int n_valid, total_units;
  struct Dec {                  // a decider's scratch
    union {
      float4 part[kScratch];    // piece parts of a sequence's rows
      double segw[2 * kScratch];  // segment weights of a draw
    };
    float4 row[kMaxRows];       // each row's (M, K, S, L) (greedy: M, arg, 0, 0)
    float zx[kMaxRows];         // each pair row's logit of the drafted token
    int bad[kMaxRows];
  } dec[kCtlWarps];
  int seq_b[kPiecesMaxB];       // the work list (batch index), longest first
};

constexpr int kPCtrlBytes = ((static_cast<int>(sizeof(PCtrl)) + 1023) / 1024) * 1024;
static_assert(kMaxResid * kSegs <= 2 * kScratch && kMaxChunks * kSegs <= 2 * kScratch,
              "a draw's segment weights fit in a decider's scratch");
static_assert(kPCtrlBytes + kPiecesStages * kChunkBytes <= 227 * 1024, "control block and ring must fit in one CTA");

// ---------------------------------------------------------------------------
// Memory-model helpers: counters and flags shared between CTAs.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int atom_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ float4 ld_relaxed_f4(const float4* p) {
  float4 v;
  asm volatile("ld.relaxed.gpu.global.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ float2 ld_relaxed_f2(const float2* p) {
  float2 v;
  asm volatile("ld.relaxed.gpu.global.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ float ld_relaxed_f(const float* p) {
  float v;
  asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ int ld_relaxed_i(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// ---------------------------------------------------------------------------

template <int ELT, bool GREEDY>
struct Pieces {
  using V = Vec<ELT>;
  static constexpr int NV = V::N;

  const VerifyParams& P;
  PCtrl& C;
  unsigned char* ring;
  const int lane, warp;
  const long long row_bytes;

  __device__ Pieces(const VerifyParams& p, PCtrl& c, unsigned char* r, int ln, int wp)
      : P(p), C(c), ring(r), lane(ln), warp(wp), row_bytes(static_cast<long long>(p.V) * ELT) {}

  __device__ const unsigned char* trow(int b, int pos) const {
    return static_cast<const unsigned char*>(P.target) +
           (static_cast<size_t>(b) * (P.k + 1) + pos) * static_cast<size_t>(row_bytes);
  }
  __device__ const unsigned char* drow(int b, int pos) const {
    return static_cast<const unsigned char*>(P.draft) +
           (static_cast<size_t>(b) * P.k + pos) * static_cast<size_t>(row_bytes);
  }
  __device__ int row_index(int b, int pos, int kind) const {
    return kind == 0 ? b * (P.k + 1) + pos : P.B * (P.k + 1) + b * P.k + pos;
  }

  __device__ bool warp_wait(uint64_t* bar, uint32_t parity) const {
    int ok = 1;
    if (lane == 0) ok = mbar_wait_bounded(bar, parity, kDrainLimitNs) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok && lane == 0) atomicOr(P.ws.err_word, 1u << 5 /* SV_ERR_TIMEOUT */);
    __syncwarp();
    return ok != 0;
  }

  // ======================= producer ==========================================

  // Stream unit t of the work list: (b, k_b, pos, kind, piece).
  __device__ void map_unit(int t, int& b, int& kb, int& pos, int& kind, int& piece) const {
    int L = P.k;
    while (L > 0 && t >= C.gunits[L] + C.gcount[L] * (GREEDY ? L + 1 : 2 * L + 1) * P.np) --L;
    const int per = (GREEDY ? L + 1 : 2 * L + 1) * P.np;
    const int off = t - C.gunits[L];
    const int n = C.gstart[L] + off / per;
    const int local = off - (off / per) * per;
    const int row = local / P.np;
    piece = local - row * P.np;
    b = C.seq_b[n];
    kb = L;
    if (GREEDY) { pos = row; kind = 0; }
    else if (row < 2 * L) { pos = row >> 1; kind = row & 1; }
    else { pos = L; kind = 0; }
  }

  __device__ bool acquire_slot(int q) {
    return warp_wait(&C.empty[q % kPiecesStages], ((q / kPiecesStages) & 1) ^ 1);
  }

  // Stream unit t into slot q.
  __device__ void issue_stream(int q, int t) {
    int b, kb, pos, kind, piece;
    map_unit(t, b, kb, pos, kind, piece);
    const int slot = q % kPiecesStages;
    const int e0 = piece * P.pe;
    const int n = min(P.pe, P.V - e0);
    const int nbytes = n * ELT;
    if (lane == 0) {
      PDesc& d = C.desc[slot];
      d.b = b; d.kb = kb; d.pos = pos; d.kind = kind;
      d.piece = piece; d.nbytes = nbytes; d.r = row_index(b, pos, kind); d.x = -1;
      const unsigned char* src = (kind == 0 ? trow(b, pos) : drow(b, pos)) + static_cast<size_t>(e0) * ELT;
      mbar_expect_tx(&C.full[slot], static_cast<uint32_t>(nbytes));
      bulk_load(ring + static_cast<size_t>(slot) * kChunkBytes, src, static_cast<uint32_t>(nbytes), &C.full[slot]);
    }
    __syncwarp();
  }

  // Re-read piece j of sequence b's rejected pair (lane 0; its message was
  // acquired, so the pair's record is visible).
  __device__ void issue_resid(int q, int b, int j) {
    const int slot = q % kPiecesStages;
    if (lane == 0) {
      int4 ent;
      asm volatile("ld.relaxed.gpu.global.v4.s32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(ent.x), "=r"(ent.y), "=r"(ent.z), "=r"(ent.w) : "l"(P.pw.rq + b) : "memory");
      const float4 nrm = ld_relaxed_f4(P.pw.rqn + b);
      const int a = ent.x;
      const int e0 = j * P.he;
      const int n = min(P.he, P.V - e0);
      const int nbytes = n * ELT;
      PDesc& d = C.desc[slot];
      d.b = b; d.kb = ent.y; d.pos = a; d.kind = 2;
      d.piece = j; d.nbytes = nbytes; d.r = b; d.x = -1;
      d.K0 = nrm.x; d.L0 = nrm.y; d.G0 = nrm.z; d.G1 = nrm.w;
      unsigned char* dst = ring + static_cast<size_t>(slot) * kChunkBytes;
      mbar_expect_tx(&C.full[slot], static_cast<uint32_t>(2 * nbytes));
      bulk_load(dst, trow(b, a) + static_cast<size_t>(e0) * ELT, static_cast<uint32_t>(nbytes), &C.full[slot]);
      bulk_load(dst + kHalf, drow(b, a) + static_cast<size_t>(e0) * ELT, static_cast<uint32_t>(nbytes),
                &C.full[slot]);
    }
    __syncwarp();
  }

  // The producer fills one slot at a time: with a re-read piece if one was
  // handed to this CTA (the draws of decided sequences come first), else
  // with its next stream unit (blockIdx.x, then every gridDim.x-th).  It
  // reads its mailbox's count every fourth slot, using the value requested
  // four slots earlier, so that no global load stalls it while the ring has
  // room.
  __device__ void produce() {
    int q = 0;
    int t = blockIdx.x;
    const int G = gridDim.x;
    int mt = 0, mt_req = 0, mhead = 0;  // lane 0: mailbox count known, requested; messages taken
    int* mtail = P.pw.mtail + blockIdx.x * 32;
    const int* mbox = P.pw.mbox + static_cast<size_t>(blockIdx.x) * P.pw.mcap;
    bool stream_open = true;
    unsigned long long idle_since = 0;
    while (true) {
      if (!acquire_slot(q)) break;
      int msg = 0;
      if (lane == 0 && mhead < mt) {
        // the slot was counted before the message was written: wait for it
        const unsigned long long t0 = global_ns();
        while ((msg = ld_acquire(mbox + mhead)) == 0) {
          if (static_cast<long long>(global_ns() - t0) > kDrainLimitNs) {
            atomicOr(P.ws.err_word, 1u << 5 /* SV_ERR_TIMEOUT */);
            msg = -1;
            break;
          }
          __nanosleep(32);
        }
        ++mhead;
      }
      msg = __shfl_sync(0xffffffffu, msg, 0);
      bool issued = false;
      if (msg > 0) {
        const int m = msg - 1;
        issue_resid(q, m / P.nr, m - (m / P.nr) * P.nr);
        issued = true;
      } else if (stream_open && t < C.total_units) {
        issue_stream(q, t);
        t += G;
        issued = true;
      }
      if (issued) {
        if (lane == 0 && (q & 3) == 3) { mt = max(mt, mt_req); mt_req = ld_relaxed_i(mtail); }
        ++q;
        idle_since = 0;
        continue;
      }
      stream_open = false;
      // nothing for this slot yet: done once every sequence is settled
      int settled = 0;
      if (lane == 0) {
        mt = max(mt, ld_relaxed_i(mtail));
        settled = ld_relaxed_i(P.pw.ctr + kCtrSettled);
      }
      settled = __shfl_sync(0xffffffffu, settled, 0);
      if (settled >= C.n_valid) break;
      if (!idle_since) idle_since = global_ns();
      if (static_cast<long long>(global_ns() - idle_since) > kDrainLimitNs) {
        if (lane == 0) atomicOr(P.ws.err_word, 1u << 5 /* SV_ERR_TIMEOUT */);
        break;
      }
      __nanosleep(200);
    }
    // one end marker per control warp (also after an error, so that every
    // warp stops)
    for (int i = 0; i < kCtlWarps; ++i) {
      if (!acquire_slot(q)) break;
      if (lane == 0) {
        C.desc[q % kPiecesStages].kind = -1;
        mbar_arrive(&C.full[q % kPiecesStages]);
      }
      __syncwarp();
      ++q;
    }
  }

  // ======================= consumers =========================================

  __device__ void consume() {
    const float c2 = P.c2;
    int q = 0, ends = 0;
    while (true) {
      const int slot = q % kPiecesStages;
      const uint32_t par = static_cast<uint32_t>(q / kPiecesStages) & 1u;
      int timed_out = 0;
      if (!mbar_wait_bounded(&C.full[slot], par, P.wait_limit_ns)) {
        timed_out = 1;
        if (!mbar_wait_bounded(&C.full[slot], par, kDrainLimitNs)) {
          if (lane == 0) atomicOr(P.ws.err_word, 1u << 5 /* SV_ERR_TIMEOUT */);
          return;   // the producer is gone
        }
      }
      const PDesc d = C.desc[slot];
      const int ubi = q % kUBufs;
      if (!warp_wait(&C.ufree[ubi], ((q / kUBufs) & 1) ^ 1)) return;
      UBuf& U = C.ub[ubi];
      const unsigned char* data = ring + static_cast<size_t>(slot) * kChunkBytes;
      if (d.kind < 0) {
        __syncwarp();
        if (lane == 0) {
          if (warp == 0) U.d = d;
          mbar_arrive(&C.empty[slot]);
          mbar_arrive(&C.ufull[ubi]);
        }
        ++q;
        // one end marker per control warp: stop after the last
        if (++ends == kCtlWarps) return;
        continue;
      }
      float4 out;
      if (d.kind == 2) {
        const int nvec = (d.nbytes + 15) / 16;
        uint4 rt[kHalfVecsPerLane], rd[kHalfVecsPerLane];
#pragma unroll
        for (int j = 0; j < kHalfVecsPerLane; ++j) {
          const int v = warp * kHalfVecsPerWarp + j * 32 + lane;
          const bool in = v < nvec;
          rt[j] = in ? *reinterpret_cast<const uint4*>(data + static_cast<size_t>(v) * 16) : V::neg_inf();
          rd[j] = in ? *reinterpret_cast<const uint4*>(data + kHalf + static_cast<size_t>(v) * 16) : V::neg_inf();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&C.empty[slot]);
        const f2 cc = pack2(c2, c2), nkt = pack2(-d.K0, -d.K0), nlt = pack2(-d.L0, -d.L0);
        const f2 gh = pack2(d.G0, d.G0), gl = pack2(d.G1, d.G1);
        f2 accr[NV / 2], accp[NV / 2];
#pragma unroll
        for (int i = 0; i < NV / 2; ++i) { accr[i] = 0ull; accp[i] = 0ull; }
#pragma unroll
        for (int j = 0; j < kHalfVecsPerLane; ++j) {
          f2 zt[NV / 2], zd[NV / 2];
          V::pairs(rt[j], zt);
          V::pairs(rd[j], zd);
#pragma unroll
          for (int i = 0; i < NV / 2; ++i) {
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
        out = make_float4(warp_sum(sr), warp_sum(sp), 0.f, __int_as_float(timed_out ? 2 : 0));
      } else {
        const int nvec = (d.nbytes + 15) / 16;
        uint4 raw[kVecsPerLane];
#pragma unroll
        for (int j = 0; j < kVecsPerLane; ++j) {
          const int v = warp * kVecsPerWarp + j * 32 + lane;
          raw[j] = v < nvec ? *reinterpret_cast<const uint4*>(data + static_cast<size_t>(v) * 16) : V::neg_inf();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&C.empty[slot]);
        int bad = 0;
        if (GREEDY) {
          const int base = d.piece * P.pe + warp * kVecsPerWarp * NV;
          float lm = -INFINITY;
          int li = 0x7fffffff;
#pragma unroll
          for (int j = 0; j < kVecsPerLane; ++j) {
            float z[NV];
            V::unpack(raw[j], z);
#pragma unroll
            for (int e = 0; e < NV; ++e) {
              bad |= (z[e] != z[e]) || (z[e] == INFINITY);
              if (z[e] > lm) { lm = z[e]; li = base + (j * 32 + lane) * NV + e; }
            }
          }
          warp_argmax(lm, li);
          bad = warp_or(bad);
          out = make_float4(lm, __int_as_float(li), 0.f, __int_as_float(bad | (timed_out ? 2 : 0)));
        } else {
          // the lane's (fl(m c), sum 2^(z c - K)), then the warp's
          const float lm = V::vmax(raw);
          float ks = -INFINITY, ls = 0.f;
          if (lm > -INFINITY) {
            ks = __fmul_rn(lm, c2);
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
          } else {
            // no finite logit in this lane's part: only NaN can still hide here
#pragma unroll
            for (int j = 0; j < kVecsPerLane; ++j) {
              float z[NV];
              V::unpack(raw[j], z);
#pragma unroll
              for (int e = 0; e < NV; ++e) bad |= (z[e] != z[e]);
            }
          }
          // NaN logits make ls NaN, +inf makes lm (and ks) +inf: both caught here
          bad |= !(ls == ls) || lm == INFINITY;
          const float wm = from_ordered_key(__reduce_max_sync(0xffffffffu, ordered_key(lm == lm ? lm : -INFINITY)));
          const float wk = wm > -INFINITY ? __fmul_rn(wm, c2) : -INFINITY;
          const float ws = warp_sum(ks > -INFINITY && ls == ls ? ls * fast_exp2(__fsub_rn(ks, wk)) : 0.f);
          bad = warp_or(bad);
          out = make_float4(wm, wk, ws, __int_as_float(bad | (timed_out ? 2 : 0)));
        }
      }
      if (lane == 0) {
        U.w[warp] = out;
        if (warp == 0) U.d = d;
        mbar_arrive(&C.ufull[ubi]);
      }
      __syncwarp();
      ++q;
    }
  }

  // ======================= control warps =====================================

  // Push a job for this control warp's decider (bounded wait while its ring
  // is full).
  __device__ void push_job(int cw, const Job& jb) {
    if (lane == 0) {
      const int slot = C.job_tail[cw]++;
      const unsigned long long t0 = global_ns();
      while (slot - C.job_head[cw] >= kJobs) {
        if (static_cast<long long>(global_ns() - t0) > kDrainLimitNs) {
          atomicOr(P.ws.err_word, 1u << 5 /* SV_ERR_TIMEOUT */);
          break;
        }
        __nanosleep(64);
      }
      C.jobs[cw][slot % kJobs] = jb;
      __threadfence_block();
      C.job_ready[cw][slot % kJobs] = slot + 1;
    }
    __syncwarp();
  }

  __device__ void control(int cw) {
    const float c2 = P.c2;
    for (int u = cw;; u += kCtlWarps) {
      const int ubi = u % kUBufs;
      if (!warp_wait(&C.ufull[ubi], static_cast<uint32_t>(u / kUBufs) & 1u)) {
        Job jb{};
        jb.kind = kJobEnd;
        push_job(cw, jb);
        return;
      }
      const UBuf& U = C.ub[ubi];
      const PDesc d = U.d;
      const float4 w = lane < kConsumerWarps ? U.w[lane] : make_float4(-INFINITY, -INFINITY, 0.f, 0.f);
      __syncwarp();
      if (lane == 0) mbar_arrive(&C.ufree[ubi]);
      if (d.kind < 0) {
        Job jb{};
        jb.kind = kJobEnd;
        push_job(cw, jb);
        return;
      }
      const bool in = lane < kConsumerWarps;
      const int wbad = in ? __float_as_int(w.w) : 0;
      const int bad = static_cast<int>(__reduce_or_sync(0xffffffffu, static_cast<unsigned>(wbad)));
      if (d.kind == 2) {
        // a re-read piece: the per-segment masses, then the pair's counter
        float* rm = P.pw.rmass + (static_cast<size_t>(d.b) * P.nr + d.piece) * kSegs;
        float* pm = P.pw.pmass + (static_cast<size_t>(d.b) * P.nr + d.piece) * kSegs;
        if (in) { rm[lane] = w.x; pm[lane] = w.y; }
        __threadfence();       // every lane's stores before lane 0's release below
        __syncwarp();
        int old = 0;
        if (lane == 0) {
          if (bad) atomicOr(P.pw.rflag + d.b, bad);
          old = atom_add_acq_rel(P.pw.rcnt + d.b, 1);
        }
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old == P.nr - 1) {
          Job jb{};
          jb.kind = kJobResid; jb.b = d.b; jb.pos = d.pos; jb.r = d.r; jb.pad0 = d.kb;
          push_job(cw, jb);
        }
        continue;
      }
      float4 part;
      if (GREEDY) {
        const float M = from_ordered_key(__reduce_max_sync(0xffffffffu, ordered_key(in ? w.x : -INFINITY)));
        const int arg = __reduce_min_sync(0xffffffffu, (in && w.x == M) ? __float_as_int(w.y) : 0x7fffffff);
        part = make_float4(M, __int_as_float(arg), 0.f, __int_as_float(bad));
      } else {
        const float M = from_ordered_key(__reduce_max_sync(0xffffffffu, ordered_key(in ? w.x : -INFINITY)));
        const float K = M > -INFINITY ? __fmul_rn(M, c2) : -INFINITY;
        float v = (in && w.y > -INFINITY) ? w.z * fast_exp2(__fsub_rn(w.y, K)) : 0.f;
#pragma unroll
        for (int o = kConsumerWarps / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        part = make_float4(M, K, __shfl_sync(0xffffffffu, v, 0), __int_as_float(bad));
        if (d.kind == 0 && d.pos == d.kb && in) {
          // bonus row: each consumer warp's segment (K, S), for the draw
          P.pw.bseg[(static_cast<size_t>(d.b) * P.np + d.piece) * kSegs + lane] = make_float2(w.y, w.z);
          __threadfence();     // before lane 0's release below
        }
      }
      __syncwarp();
      // the piece's part, then the sequence's counter: the last piece
      // decides the sequence
      int old = 0;
      if (lane == 0) {
        P.pw.rowpart[static_cast<size_t>(d.r) * P.np + d.piece] = part;
        old = atom_add_acq_rel(P.pw.seqcnt + d.b, 1);
      }
      old = __shfl_sync(0xffffffffu, old, 0);
      if (old == (GREEDY ? d.kb + 1 : 2 * d.kb + 1) * P.np - 1) {
        Job jb{};
        jb.kind = kJobSeq; jb.b = d.b; jb.pad0 = d.kb;
        push_job(cw, jb);
      }
    }
  }

  // ======================= decider warp ======================================

  __device__ void finish_outputs(int b, int kb, int a, int y, int err, int zero_resid) {
    const int k = P.k;
    int* ot = P.out_tokens + static_cast<size_t>(b) * (k + 1);
    const bool ok = !err && y >= 0;
    for (int j = lane; j <= k; j += 32) {
      int v = -1;
      if (ok) v = j < a ? P.tokens[static_cast<size_t>(b) * k + j] : (j == a ? y : -1);
      ot[j] = v;
    }
    if (lane == 0) {
      P.out_len[b] = ok ? a + 1 : 0;
      if (ok) {
        atomicAdd(P.ws.stats + kStatSequences, 1ull);
        atomicAdd(P.ws.stats + kStatProposed, static_cast<unsigned long long>(kb));
        atomicAdd(P.ws.stats + kStatAccepted, static_cast<unsigned long long>(a));
        atomicAdd(P.ws.stats + kStatEmitted, static_cast<unsigned long long>(a + 1));
        if (kb == 0) atomicAdd(P.ws.stats + kStatSpecOff, 1ull);
        if (zero_resid) atomicAdd(P.ws.stats + kStatZeroResidual, 1ull);
      } else {
        atomicAdd(P.ws.stats + kStatErrorSeqs, 1ull);
        unsigned bits = static_cast<unsigned>(err & (kErrBadTok | kErrNonfin | kErrTime));
        if (!bits) bits = kErrNonfin;    // no token could be drawn
        atomicOr(P.ws.err_word, bits);
      }
      __threadfence();
      atomicAdd(P.pw.ctr + kCtrSettled, 1);
    }
    __syncwarp();
  }

  // The segment holding target weight t among n weights (index order),
  // fp64 running sums; past the end (rounding): the last positive one.
  // Returns the segment and what is left of t at its start.
  __device__ int locate(const double* wts, int n, double t, double& seg_t) const {
    const int per = (n + 31) / 32;
    const int g0 = min(n, lane * per), g1 = min(n, g0 + per);
    double gs = 0.0;
    for (int i = g0; i < g1; ++i) gs += wts[i];
    const double incl = warp_incl_scan(gs, lane);
    const double excl = incl - gs;
    const unsigned hit = __ballot_sync(0xffffffffu, gs > 0.0 && t < incl);
    const unsigned posg = __ballot_sync(0xffffffffu, gs > 0.0);
    const int owner = hit ? (__ffs(hit) - 1) : (posg ? 31 - __clz(posg) : -1);
    int seg = -1;
    double st = 0.0;
    if (owner >= 0 && lane == owner) {
      double run = excl, last_run = excl;
      int last = -1;
      for (int i = g0; i < g1; ++i) {
        const double m = wts[i];
        if (m > 0.0) { last = i; last_run = run; }
        if (seg < 0 && m > 0.0 && t < run + m) { seg = i; st = t - run; }
        run += m;
      }
      if (seg < 0) { seg = last; st = t - last_run; }
    }
    if (owner >= 0) {
      seg = __shfl_sync(0xffffffffu, seg, owner);
      st = __shfl_sync(0xffffffffu, st, owner);
    }
    seg_t = st;
    return seg;
  }

  // Vector v of a row, -inf past the row.
  __device__ uint4 load_vec(const unsigned char* row, int v, int v_end) const {
    if (v >= v_end || v < 0) return V::neg_inf();
    return __ldg(reinterpret_cast<const uint4*>(row) + v);
  }

  // Walk NSTEPS x 32 vectors from vector v0, none at or past v_end (the end
  // of the piece the segment belongs to), a warp inclusive scan per step, to
  // the token where the running weight passes t.  RESID: weights
  // max(0, p - q); else p.  Same arithmetic as the consumers' weights.
  template <int NSTEPS, bool RESID>
  __device__ int walk(int v0, int v_end, double t, const unsigned char* rowT, const unsigned char* rowD,
                                   float Kt, float Lt, float Gh, float Gl) const {
    uint4 rt[NSTEPS], rd[RESID ? NSTEPS : 1];
#pragma unroll
    for (int j = 0; j < NSTEPS; ++j) {
      rt[j] = load_vec(rowT, v0 + j * 32 + lane, v_end);
      if (RESID) rd[RESID ? j : 0] = load_vec(rowD, v0 + j * 32 + lane, v_end);
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

  // Every piece of sequence b is reduced: its rows, tests, first rejection,
  // and the bonus draw or the re-read of the rejected pair.
  __device__ void seq_done(int b, int kb) {
    const float c2 = P.c2;
    const int np = P.np, k1 = P.k + 1;
    const int nrows = GREEDY ? kb + 1 : 2 * kb + 1;
    typename PCtrl::Dec& S = C.dec[dw];
    fence_acq_rel_gpu();
    // row ri of the sequence (in streaming order): target row i = ri / 2
    // (ri even) or draft row ri / 2 (ri odd); the bonus row is ri = 2 k_b
    // (greedy: target row ri)
    auto row_of = [&](int ri) {
      if (GREEDY) return row_index(b, ri, 0);
      return row_index(b, ri >> 1, ri & 1);
    };
    // what the tests and the bonus draw need, requested with the parts
    int x = -1;
    float u = 0.f;
    if (lane < kb) {
      x = __ldg(P.tokens + static_cast<size_t>(b) * P.k + lane);
      if (!GREEDY) u = __ldg(P.uniforms + static_cast<size_t>(b) * k1 + lane);
    }
    const float s = GREEDY ? 0.f : __ldg(P.uniforms + static_cast<size_t>(b) * k1 + P.k);
    const int nseg = np * kSegs;
    float2 bs[kMaxChunks * kSegs / 32];
#pragma unroll
    for (int i = 0; i < kMaxChunks * kSegs / 32; ++i) {
      const int sg = lane + 32 * i;
      bs[i] = (!GREEDY && sg < nseg) ? ld_relaxed_f2(P.pw.bseg + static_cast<size_t>(b) * nseg + sg)
                                     : make_float2(-INFINITY, 0.f);
    }
    // every row's (M, K, S, L) from its pieces in piece order, rows taken
    // kScratch / np at a time through shared memory
    const int per = kScratch / np;
    float zt_x = 0.f, zd_x = 0.f;    // the drafted tokens' logits (lane i: draft i)
    for (int r0 = 0; r0 < nrows; r0 += per) {
      const int r1 = min(nrows, r0 + per);
      __syncwarp();
      for (int i = lane; i < (r1 - r0) * np; i += 32)
        S.part[i] = ld_relaxed_f4(P.pw.rowpart + static_cast<size_t>(row_of(r0 + i / np)) * np + i % np);
      __syncwarp();
      if (r0 == 0 && !GREEDY && lane < kb && x >= 0 && x < P.V) {
        // requested here, used after the combines below
        zt_x = V::scalar(trow(b, lane), x);
        zd_x = V::scalar(drow(b, lane), x);
      }
      for (int ri = r0 + lane; ri < r1; ri += 32) {
        const float4* pp = S.part + (ri - r0) * np;
        int bad = 0;
        float4 st;
        if (GREEDY) {
          float M = -INFINITY;
          int arg = 0x7fffffff;
          for (int j = 0; j < np; ++j) {
            bad |= __float_as_int(pp[j].w);
            if (pp[j].x > M) { M = pp[j].x; arg = __float_as_int(pp[j].y); }   // pieces in order: ties keep the first
          }
          st = make_float4(M, __int_as_float(arg), 0.f, 0.f);
          bad = ((bad & 1) || !(M > -INFINITY) ? kErrNonfin : 0) | ((bad & 2) ? kErrTime : 0);
        } else {
          float M = -INFINITY;
          for (int j = 0; j < np; ++j) { bad |= __float_as_int(pp[j].w); M = fmaxf(M, pp[j].x); }
          const float K = M > -INFINITY ? __fmul_rn(M, c2) : -INFINITY;
          float v = 0.f;
          for (int j = 0; j < np; ++j) v += pp[j].y > -INFINITY ? pp[j].z * fast_exp2(__fsub_rn(pp[j].y, K)) : 0.f;
          st = make_float4(M, K, v, log2f(v));
          bad = ((bad & 1) || !(isfinite(M) && isfinite(v) && v > 0.f) ? kErrNonfin : 0) | ((bad & 2) ? kErrTime : 0);
        }
        S.row[ri] = st;
        S.bad[ri] = bad;
        // diagnostics
        if (!P.diag) {
        } else if (GREEDY) {
          P.ws.m_t[static_cast<size_t>(b) * k1 + ri] = st.x;
        } else if (ri & 1) {
          P.ws.m_d[static_cast<size_t>(b) * P.k + (ri >> 1)] = st.x;
          P.ws.L_d[static_cast<size_t>(b) * P.k + (ri >> 1)] = st.w;
        } else {
          P.ws.m_t[static_cast<size_t>(b) * k1 + (ri >> 1)] = st.x;
          P.ws.L_t[static_cast<size_t>(b) * k1 + (ri >> 1)] = st.w;
        }
      }
    }
    if (!GREEDY && lane < kb) { S.zx[2 * lane] = zt_x; S.zx[2 * lane + 1] = zd_x; }
    __syncwarp();
    // the tests, lane i for draft i: alpha = min(1, 2^-delta) with
    // delta = log2 (q(x) / p(x)) = (z_d(x) - z_t(x)) c + G, G the log2 ratio
    // of the target's to the draft's normaliser
    int err = 0;
    for (int ri = lane; ri < nrows; ri += 32) err |= S.bad[ri];
    bool reject = false;
    float Gh = 0.f, Gl = 0.f;
    if (lane < kb) {
      if (x < 0 || x >= P.V) {
        err |= kErrBadTok;
      } else if (GREEDY) {
        reject = x != __float_as_int(S.row[lane].y);
        if (P.diag) P.ws.alpha[static_cast<size_t>(b) * P.k + lane] = reject ? 0.f : 1.f;
      } else {
        const float4 T = S.row[2 * lane], D = S.row[2 * lane + 1];
        const float zt = S.zx[2 * lane], zd = S.zx[2 * lane + 1];
        log2_ratio(T.y, T.z, D.y, D.z, Gh, Gl);
        float alpha;
        if (zt == -INFINITY) alpha = 0.f;               // p(x) = 0
        else if (zd == -INFINITY) alpha = 1.f;          // q(x) = 0 < p(x)
        else {
          const float delta = __fadd_rn(__fmaf_rn(__fsub_rn(zd, zt), c2, Gh), Gl);
          alpha = delta <= 0.f ? 1.f : exp2f(-delta);
        }
        if (P.diag) P.ws.alpha[static_cast<size_t>(b) * P.k + lane] = alpha;
        reject = !(u < alpha);
      }
    }
    err = warp_or(err);
    const unsigned rej = __ballot_sync(0xffffffffu, reject);
    const int a = rej ? __ffs(rej) - 1 : kb;
    if (err) { finish_outputs(b, kb, a, -1, err, 0); return; }
    if (GREEDY) {
      finish_outputs(b, kb, a, __float_as_int(S.row[a].y), 0, 0);
      return;
    }
    if (a < kb) {
      // the rejected pair is read again in nr pieces, handed round-robin to
      // the CTAs' mailboxes (piece j to CTA (b nr + j) mod ctas): the pair's
      // record first, then one message per piece
      Gh = __shfl_sync(0xffffffffu, Gh, a);
      Gl = __shfl_sync(0xffffffffu, Gl, a);
      if (lane == 0) {
        const float4 T = S.row[2 * a];
        P.pw.rq[b] = make_int4(a, kb, 0, 0);
        P.pw.rqn[b] = make_float4(T.y, T.w, Gh, Gl);
        __threadfence();
      }
      __syncwarp();
      for (int j = lane; j < P.nr; j += 32) {
        const int m = b * P.nr + j;
        const int cta = m % P.ctas;
        const int slot = atomicAdd(P.pw.mtail + cta * 32, 1);
        st_release(P.pw.mbox + static_cast<size_t>(cta) * P.pw.mcap + slot, m + 1);
      }
      __syncwarp();
      return;
    }
    // every draft accepted: the bonus token from p_{k_b}: the segment from
    // the segment sums kept while streaming, then a walk of that segment
    const float4 T = S.row[2 * kb];
    double* seg_w = S.segw;
#pragma unroll
    for (int i = 0; i < kMaxChunks * kSegs / 32; ++i) {
      const int sg = lane + 32 * i;
      if (sg < nseg)
        seg_w[sg] = bs[i].x == -INFINITY ? 0.0
                    : static_cast<double>(bs[i].y) * static_cast<double>(fast_exp2(__fsub_rn(bs[i].x, T.y) - T.w));
    }
    __syncwarp();
    double tot = 0.0;
    for (int i = lane; i < nseg; i += 32) tot += seg_w[i];
    tot = warp_sum(tot);
    double seg_t;
    const int seg = locate(seg_w, nseg, static_cast<double>(s) * tot, seg_t);
    int y = -1;
    if (seg >= 0) {
      const int piece = seg / kSegs, sw = seg - piece * kSegs;
      const int v0 = (piece * P.pe) / NV + sw * kVecsPerWarp;
      const int v_end = min(P.V, (piece + 1) * P.pe) / NV;
      y = walk<kVecsPerLane, false>(v0, v_end, seg_t, trow(b, kb), nullptr, T.y, T.w, 0.f, 0.f);
    }
    if (lane == 0 && P.diag) P.ws.mass[static_cast<size_t>(b) * k1 + kb] = static_cast<float>(tot);
    finish_outputs(b, kb, kb, y, 0, 0);
  }

  // Every re-read piece of sequence b's rejected pair is reduced: the draw.
  __device__ void resid_done(const Job& jb) {
    const int b = jb.b, a = jb.pos;
    const int k1 = P.k + 1;
    fence_acq_rel_gpu();
    double* rseg_w = C.dec[dw].segw;
    const int nseg = P.nr * kSegs;
    double r = 0.0;
    for (int i = lane; i < nseg; i += 32) r += static_cast<double>(ld_relaxed_f(P.pw.rmass + static_cast<size_t>(b) * nseg + i));
    const double rtot = warp_sum(r);
    // exact arithmetic rules a zero residual out (a rejection implies p > q
    // somewhere); if rounding leaves none, the draw is from p_a (counted)
    const bool resid = rtot > 0.0;
    const float* src = resid ? P.pw.rmass : P.pw.pmass;
    for (int i = lane; i < nseg; i += 32) rseg_w[i] = static_cast<double>(ld_relaxed_f(src + static_cast<size_t>(b) * nseg + i));
    __syncwarp();
    double tot = 0.0;
    for (int i = lane; i < nseg; i += 32) tot += rseg_w[i];
    tot = warp_sum(tot);
    const float s = P.uniforms[static_cast<size_t>(b) * k1 + P.k];
    const float4 nrm = ld_relaxed_f4(P.pw.rqn + b);
    int flag = 0;
    if (lane == 0) flag = ld_relaxed_i(P.pw.rflag + b);
    flag = __shfl_sync(0xffffffffu, flag, 0);
    double seg_t;
    const int seg = locate(rseg_w, nseg, static_cast<double>(s) * tot, seg_t);
    int y = -1;
    if (seg >= 0) {
      const int piece = seg / kSegs, sw = seg - piece * kSegs;
      const int v0 = (piece * P.he) / NV + sw * kHalfVecsPerWarp;
      const int v_end = min(P.V, (piece + 1) * P.he) / NV;
      if (resid)
        y = walk<kHalfVecsPerLane, true>(v0, v_end, seg_t, trow(b, a), drow(b, a), nrm.x, nrm.y, nrm.z, nrm.w);
      else
        y = walk<kHalfVecsPerLane, false>(v0, v_end, seg_t, trow(b, a), nullptr, nrm.x, nrm.y, 0.f, 0.f);
    }
    if (lane == 0 && P.diag) P.ws.mass[static_cast<size_t>(b) * k1 + a] = static_cast<float>(tot);
    finish_outputs(b, jb.pad0, a, y, (flag & 2) ? kErrTime : 0, resid ? 0 : 1);
  }

  int dw = 0;   // decider warp index (its job ring and scratch)

  __device__ void decider(int d) {
    dw = d;
    int head = 0;
    unsigned long long idle_since = 0;
    while (true) {
      int ready = 0;
      if (lane == 0) ready = C.job_ready[dw][head % kJobs] == head + 1;
      ready = __shfl_sync(0xffffffffu, ready, 0);
      if (!ready) {
        if (!idle_since) idle_since = global_ns();
        if (static_cast<long long>(global_ns() - idle_since) > 8 * kDrainLimitNs) {
          if (lane == 0) atomicOr(P.ws.err_word, 1u << 5 /* SV_ERR_TIMEOUT */);
          return;
        }
        __nanosleep(64);
        continue;
      }
      idle_since = 0;
      __threadfence_block();
      const Job jb = C.jobs[dw][head % kJobs];
      __syncwarp();
      if (lane == 0) C.job_head[dw] = head + 1;
      ++head;
      if (jb.kind == kJobEnd) {
        return;                  // its control warp has stopped
      } else if (jb.kind == kJobSeq) {
        seq_done(jb.b, jb.pad0);
      } else {
        resid_done(jb);
      }
      __syncwarp();
    }
  }
};

template <int ELT, bool GREEDY>
__global__ void __launch_bounds__(kPThreads, 1) verify_pieces_kernel(const VerifyParams P) {
  extern __shared__ __align__(1024) unsigned char smem[];
  PCtrl& C = *reinterpret_cast<PCtrl*>(smem);
  unsigned char* ring = smem + kPCtrlBytes;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < kPiecesStages; ++s) {
      mbar_init(&C.full[s], 1);
      mbar_init(&C.empty[s], kConsumerWarps);
    }
    for (int u = 0; u < kUBufs; ++u) {
      mbar_init(&C.ufull[u], kConsumerWarps);
      mbar_init(&C.ufree[u], 1);
    }
    for (int i = 0; i < kCtlWarps; ++i) { C.job_tail[i] = 0; C.job_head[i] = 0; }
    fence_mbar_init();
  }
  for (int j = tid; j < kCtlWarps * kJobs; j += kPThreads) C.job_ready[j / kJobs][j % kJobs] = 0;
  grid_dependency_wait();             // plan_kernel: the work list, the counters
  // the work list and its groups (draft length L, longest first)
  const int n = __ldcg(P.ws.n_seqs);
  for (int i = tid; i < n; i += kPThreads) C.seq_b[i] = __ldcg(&P.ws.seqs[i].x);
  if (tid == 0) {
    int start = 0, units = 0;
    for (int L = P.k; L >= 0; --L) {
      const int upto = __ldcg(P.pw.grp + L);          // sequences with k_b >= L
      C.gstart[L] = start;
      C.gunits[L] = units;
      C.gcount[L] = upto - start;
      units += (upto - start) * (GREEDY ? L + 1 : 2 * L + 1) * P.np;
      start = upto;
    }
    C.n_valid = n;
    C.total_units = units;
  }
  __syncthreads();
  {
    Pieces<ELT, GREEDY> v(P, C, ring, lane, warp);
    if (warp < kConsumerWarps) v.consume();
    else if (warp == kWarpProducer) v.produce();
    else if (warp < kWarpDec0) v.control(warp - kWarpCtl0);
    else v.decider(warp - kWarpDec0);
  }
}

}  // namespace

int pieces_smem_bytes() { return kPCtrlBytes + kPiecesStages * kChunkBytes; }

cudaError_t prepare_pieces_kernel() {
  const void* fns[4] = {reinterpret_cast<const void*>(&verify_pieces_kernel<2, false>),
                        reinterpret_cast<const void*>(&verify_pieces_kernel<4, false>),
                        reinterpret_cast<const void*>(&verify_pieces_kernel<2, true>),
                        reinterpret_cast<const void*>(&verify_pieces_kernel<4, true>)};
  for (const void* f : fns) {
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, pieces_smem_bytes());
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_pieces(const VerifyParams& p, cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(p.ctas), 1, 1);
  cfg.blockDim = dim3(kPThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(pieces_smem_bytes());
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.greedy) {
    if (p.elt == 2) return cudaLaunchKernelEx(&cfg, verify_pieces_kernel<2, true>, p);
    return cudaLaunchKernelEx(&cfg, verify_pieces_kernel<4, true>, p);
  }
  if (p.elt == 2) return cudaLaunchKernelEx(&cfg, verify_pieces_kernel<2, false>, p);
  return cudaLaunchKernelEx(&cfg, verify_pieces_kernel<4, false>, p);
}

}  // namespace sv
