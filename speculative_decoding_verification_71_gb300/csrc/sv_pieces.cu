// Row-streaming schedule of speculative-sampling verification
// (SV_KERNEL_PIECES), for sm_103a.
//
// The same rule as verify_kernel (accept draft i with min(1, p_i/q_i) up to
// the first rejection, then the residual max(0, p - q) or the bonus row),
// the same arithmetic, another schedule: the rows of the batch are streamed
// as independent 64 KB pieces spread evenly over one CTA per SM, with no
// exchange between CTAs, and the per-sequence decisions come after.  Four
// launches per call, each waiting for its predecessor's results with
// programmatic dependent launch:
//   rows_stats_kernel   the plan in every CTA (rows of the sequences before
//                       each, in batch order: 2 k_b + 1), then every needed
//                       row, piece by piece: a producer warp
//                       streams the pieces through three shared-memory slots
//                       with cp.async.bulk, 16 consumer warps reduce them; the
//                       last warp to finish a piece combines the warps' parts
//                       into its record (max, sum of 2^(z c - fl(max c)), the
//                       drafted token's logit), at a fixed place per
//                       (sequence, row, piece); bonus rows also keep each
//                       warp segment's sum for the draw;
//   rows_decide_kernel  one warp per sequence: the rows from their pieces, the
//                       tests, the first rejection, the accepted prefix; a
//                       job for the residual, or the bonus row's numbers for
//                       its draw; an invalid k_b answered;
//   rows_resid_kernel   every job's rejected pair read again in 16 KB
//                       half-pieces dealt round robin over two CTAs per SM: each
//                       warp segment's sums of max(0, p - q) and of p;
//   rows_draw_kernel    one warp per job and one per fully accepted
//                       sequence: the segment holding s * S, the token.
// Rows must be 16-byte aligned (bulk copies); other calls run the cluster
// kernel.

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "sv_internal.h"
#include "sv_device.cuh"

namespace sv {
namespace {

constexpr int kRWarps = kConsumerWarps;              // consumer warps (16)
constexpr int kRProducer = kRWarps;                  // the producer warp's index
constexpr int kRThreads = (kRWarps + 1) * 32;
constexpr int kRStages = 3;                          // 64 KB staging slots
constexpr int kRHalf = kRowsHalfBytes;               // a re-read slot: 16 KB of each row of the pair
constexpr int kQSlot = 2 * kRHalf;                   // re-read staging slot (both rows)
constexpr int kRStatVecs = kChunkBytes / 16 / kRWarps / 32;   // 8 vectors per lane and piece
constexpr int kRDrawVecs = kRHalf / 16 / kRWarps / 32;        // 2 vectors per lane and half-piece
constexpr int kRBufs = kRStages + 1;                 // per-piece part buffers (warps run at most a ring apart)
constexpr int kRSmallThreads = 64;                   // decide / draw kernels: 2 warps, one sequence each

// flags of a part or record
enum : int { kFBad = 1, kFHasZx = 2, kFTimeout = 4 };
enum : int { kErrBadTok = 1 << 3, kErrNonfin = 1 << 4, kErrTime = 1 << 5 };

struct alignas(16) WPart {     // one warp's share of a piece
  float m, s, zx;              // max, sum of 2^(z c - fl(m c)) (greedy: argmax as int bits), token logit
  int flags;
};

// What a staging slot holds (written by the producer, read by the consumers).
struct RDesc {
  int u;                       // unit (piece or half-piece) index of this CTA's range, counted from 0
  int rec;                     // stats: the record index (row * np + piece); re-read: the job
  int part;                    // stats: the piece; re-read: the half-piece
  int bytes;                   // bytes of each row in the slot
  int b, kb, pos, kind;        // the row (stats) or the pair (re-read)
  int x;                       // drafted token at pos (pairs' rows), else -1
  int pad[3];
  float4 num;                  // re-read: the pair's (K_t, L_t, Gh, Gl)
};

struct RCtrl {
  uint64_t full[kRStages];     // slot filled (producer -> consumers)
  uint64_t empty[kRStages];    // slot released (one arrival per consumer warp)
  RDesc desc[kRStages];
  WPart part[kRBufs][kRWarps];
  int cnt[kRBufs];             // warps done with the piece in this buffer
  int rowoff[kPiecesMaxB + 1]; // statistics kernel: rows of the sequences before b (its own copy)
  int warp_tot[32];
};
constexpr int kRCtrlBytes = ((static_cast<int>(sizeof(RCtrl)) + 1023) / 1024) * 1024;

// The re-read kernel's control block: two CTAs share an SM (34 warps), each
// with three 32 KB slots.
struct QCtrl {
  uint64_t full[kRStages];
  uint64_t empty[kRStages];
  RDesc desc[kRStages];
};
constexpr int kQCtrlBytes = ((static_cast<int>(sizeof(QCtrl)) + 1023) / 1024) * 1024;
constexpr int kQSmem = kQCtrlBytes + kRStages * kQSlot;
static_assert(2 * kQSmem <= 227 * 1024, "two re-read CTAs must fit in one SM");
static_assert(kRCtrlBytes + kRStages * kChunkBytes <= 227 * 1024, "three slots must fit in one CTA");

__device__ __forceinline__ const unsigned char* row_ptr(const VerifyParams& P, int b, int pos, int kind) {
  const size_t rb = static_cast<size_t>(P.V) * P.elt;
  if (kind == 0) return static_cast<const unsigned char*>(P.target) + (static_cast<size_t>(b) * (P.k + 1) + pos) * rb;
  return static_cast<const unsigned char*>(P.draft) + (static_cast<size_t>(b) * P.k + pos) * rb;
}

// Vector v of a row (16-byte aligned rows), -inf past its end.
template <int ELT>
__device__ __forceinline__ uint4 row_vec(const unsigned char* row, int v, int nvec_row) {
  return v < nvec_row ? __ldg(reinterpret_cast<const uint4*>(row) + v) : Vec<ELT>::neg_inf();
}

// The segment holding the target weight `tgt` among `nseg` masses (index
// order, lanes taking contiguous runs); seg_t is what is left of tgt at the
// segment's start.  Past the end (rounding) it is the last segment with
// positive mass.  Warp-wide, in fp32: GB300's fp64 pipe is narrow, and the
// sums' rounding (under 1e-6 of the mass) stays inside the 1e-5 band within
// which a draw counts as a near-tie.
__device__ void locate_seg(const float* mass, int nseg, float tgt, int lane, int& seg, float& seg_t) {
  const int per = (nseg + 31) / 32;
  const int g0 = min(nseg, lane * per), g1 = min(nseg, g0 + per);
  float gs = 0.f;
  for (int i = g0; i < g1; ++i) gs += mass[i];
  const float incl = warp_incl_scan(gs, lane);
  const float excl = incl - gs;
  const unsigned hit = __ballot_sync(0xffffffffu, gs > 0.f && tgt < incl);
  const unsigned posg = __ballot_sync(0xffffffffu, gs > 0.f);
  const int owner = hit ? (__ffs(hit) - 1) : (posg ? 31 - __clz(posg) : -1);
  seg = -1;
  seg_t = 0.f;
  if (owner >= 0 && lane == owner) {
    float run = excl, last_run = excl;
    int last = -1;
    for (int i = g0; i < g1; ++i) {
      const float m = mass[i];
      if (m > 0.f) { last = i; last_run = run; }
      if (seg < 0 && m > 0.f && tgt < run + m) { seg = i; seg_t = tgt - run; }
      run += m;
    }
    if (seg < 0) { seg = last; seg_t = tgt - last_run; }
  }
  if (owner >= 0) {
    seg = __shfl_sync(0xffffffffu, seg, owner);
    seg_t = __shfl_sync(0xffffffffu, seg_t, owner);
  }
}

// Walk NSTEPS x 32 vectors from vector v0 of a row, a warp inclusive scan per
// step, to the token where the running weight passes t.  RESID: weights
// max(0, p - q); else p.  Warp-wide.
template <int ELT, int NSTEPS, bool RESID>
__device__ int walk_seg(const unsigned char* rowT, const unsigned char* rowD, int v0, int nvec_row, float t,
                        float c2, float Kt, float Lt, float Gh, float Gl, int lane) {
  using VV = Vec<ELT>;
  constexpr int NV = VV::N;
  uint4 rt[NSTEPS], rd[RESID ? NSTEPS : 1];
#pragma unroll
  for (int j = 0; j < NSTEPS; ++j) {
    rt[j] = row_vec<ELT>(rowT, v0 + j * 32 + lane, nvec_row);
    if (RESID) rd[RESID ? j : 0] = row_vec<ELT>(rowD, v0 + j * 32 + lane, nvec_row);
  }
  float base = 0.f;
  int found = -1, last_positive = -1;
#pragma unroll
  for (int j = 0; j < NSTEPS; ++j) {
    float w[NV], zt[NV], zd[NV];
    VV::unpack(rt[j], zt);
    if (RESID) VV::unpack(rd[RESID ? j : 0], zd);
    float ls = 0.f;
#pragma unroll
    for (int e = 0; e < NV; ++e) {
      float p;
      if (RESID) w[e] = resid_weight(zt[e], zd[e], c2, Kt, Lt, Gh, Gl, p);
      else w[e] = fast_exp2(__fsub_rn(__fmaf_rn(zt[e], c2, -Kt), Lt));
      ls += w[e];
    }
    const float incl = warp_incl_scan(ls, lane);
    float excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) excl = 0.f;
    const float step_total = __shfl_sync(0xffffffffu, incl, 31);
    const int x0 = (v0 + j * 32 + lane) * NV;
    const bool mine = found < 0 && ls > 0.f && t < base + incl && !(t < base + excl);
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
        float c = base + excl;
        int lastp = -1;
#pragma unroll
        for (int e = 0; e < NV; ++e) {
          if (w[e] > 0.f) lastp = x0 + e;
          c += w[e];
          if (pick < 0 && w[e] > 0.f && t < c) pick = x0 + e;
        }
        if (pick < 0) pick = lastp;
      }
      found = __shfl_sync(0xffffffffu, pick, hl);
    }
    base += step_total;
  }
  return found >= 0 ? found : last_positive;
}

// Outputs and counters of a finished sequence (lane 0 writes the scalars).
// xl: lane j holds drafted token j (k <= 31).  prefix_done: the accepted
// prefix and the empty tail are written already (a residual draw's sequence):
// only the drawn token remains, unless the draw failed.
__device__ void write_outputs(const VerifyParams& P, int b, int kb, int a, int y, int err, int zero_resid,
                              int xl, int lane, bool prefix_done = false) {
  const int k = P.k;
  const bool ok = !err && y >= 0;
  const int acc = a < 0 ? kb : a;
  int* ot = P.out_tokens + static_cast<size_t>(b) * (k + 1);
  if (ok && prefix_done) {
    if (lane == acc) ot[acc] = y;
  } else if (lane <= k) {
    ot[lane] = !ok ? -1 : (lane < acc ? xl : (lane == acc ? y : -1));
  }
  if (lane == 0) {
    P.out_len[b] = ok ? acc + 1 : 0;
    if (ok) {
      atomicAdd(P.ws.stats + kStatSequences, 1ull);
      atomicAdd(P.ws.stats + kStatProposed, static_cast<unsigned long long>(kb));
      atomicAdd(P.ws.stats + kStatAccepted, static_cast<unsigned long long>(acc));
      atomicAdd(P.ws.stats + kStatEmitted, static_cast<unsigned long long>(acc + 1));
      if (kb == 0) atomicAdd(P.ws.stats + kStatSpecOff, 1ull);
      if (zero_resid) atomicAdd(P.ws.stats + kStatZeroResidual, 1ull);
    } else {
      atomicAdd(P.ws.stats + kStatErrorSeqs, 1ull);
      unsigned bits = static_cast<unsigned>(err & (kErrBadTok | kErrNonfin | kErrTime));
      if (!bits) bits = kErrNonfin;   // no token could be drawn
      atomicOr(P.ws.err_word, bits);
    }
  }
}

// ---------------------------------------------------------------------------
// rows_stats_kernel: every needed row, 64 KB piece by piece
// ---------------------------------------------------------------------------

template <int ELT, bool GREEDY>
struct RowStats {
  using V = Vec<ELT>;
  static constexpr int NV = V::N;
  static constexpr int kPieceElems = kChunkBytes / ELT;
  static constexpr int kSegElems = kRStatVecs * 32 * NV;      // logits per warp segment

  const VerifyParams& P;
  RCtrl& C;
  unsigned char* ring;
  const int lane, warp;
  const long long row_bytes;
  int u0, u1;                  // this CTA's pieces [u0, u1) of rows * np, in row order

  __device__ RowStats(const VerifyParams& p, RCtrl& c, unsigned char* r, int ln, int wp)
      : P(p), C(c), ring(r), lane(ln), warp(wp), row_bytes(static_cast<long long>(p.V) * p.elt) {
    const long long units = static_cast<long long>(c.rowoff[p.B]) * p.np;
    u0 = static_cast<int>(units * blockIdx.x / gridDim.x);
    u1 = static_cast<int>(units * (blockIdx.x + 1) / gridDim.x);
  }

  __device__ void produce() {
    const uint64_t first_out = evict_first_policy();
    if (u0 >= u1) return;
    // the sequence holding this CTA's first row (rows in batch order)
    int lo = 0, hi = P.B;            // rowoff[lo] <= r < rowoff[hi]
    const int r_first = u0 / P.np;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (C.rowoff[mid] <= r_first) lo = mid; else hi = mid;
    }
    int b = lo, kb = 0, nrows_b = 0, r_base = 0, r_cur = -1, pos = 0, kind = 0, x = -1, ri = 0;
    const int stride = 2 * P.k + 1;   // record rows per sequence (the most a sequence has)
    for (int u = u0, q = 0; u < u1; ++u, ++q) {
      const int r = u / P.np, j = u - r * P.np;
      if (r != r_cur) {   // the next row: its sequence, position and drafted token
        r_cur = r;
        while (r >= C.rowoff[b + 1]) ++b;   // (sequences with no rows are passed over)
        if (r_base != C.rowoff[b] || nrows_b == 0) {
          r_base = C.rowoff[b];
          nrows_b = C.rowoff[b + 1] - r_base;
          kb = P.greedy ? nrows_b - 1 : (nrows_b - 1) >> 1;
        }
        ri = r - r_base;
        if (P.greedy) { pos = ri; kind = 0; }
        else if (ri < 2 * kb) { pos = ri >> 1; kind = ri & 1; }
        else { pos = kb; kind = 0; }
        x = pos < kb ? __ldg(P.tokens + static_cast<size_t>(b) * P.k + pos) : -1;
      }
      const int s = q % kRStages;
      int ok = 1;
      if (lane == 0) ok = mbar_wait_bounded(&C.empty[s], ((q / kRStages) & 1) ^ 1, kDrainLimitNs) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, ok, 0)) {
        if (lane == 0) atomicOr(P.ws.err_word, 1u << 5 /* SV_ERR_TIMEOUT */);
        return;   // the consumers time out on the slots left and flag their pieces
      }
      if (lane == 0) {
        const long long off = static_cast<long long>(j) * kChunkBytes;
        const int bytes = static_cast<int>(min(static_cast<long long>(kChunkBytes), row_bytes - off));
        RDesc& d = C.desc[s];
        d.u = u - u0; d.rec = (b * stride + ri) * P.np + j; d.part = j; d.bytes = bytes;
        d.b = b; d.kb = kb; d.pos = pos; d.kind = kind; d.x = x;
        mbar_expect_tx(&C.full[s], static_cast<uint32_t>(bytes));
        bulk_load_hint(ring + static_cast<size_t>(s) * kChunkBytes, row_ptr(P, b, pos, kind) + off,
                       static_cast<uint32_t>(bytes), &C.full[s], first_out);
      }
      __syncwarp();
    }
  }

  __device__ void consume() {
    const float c2 = P.c2;
    for (int u = u0, q = 0; u < u1; ++u, ++q) {
      const int s = q % kRStages;
      int flags = 0;
      if (!mbar_wait_bounded(&C.full[s], static_cast<uint32_t>(q / kRStages) & 1u, P.wait_limit_ns)) {
        flags |= kFTimeout;
        if (!mbar_wait_bounded(&C.full[s], static_cast<uint32_t>(q / kRStages) & 1u, kDrainLimitNs)) {
          if (lane == 0) atomicOr(P.ws.err_word, 1u << 5 /* SV_ERR_TIMEOUT */);
          return;   // the producer is gone
        }
      }
      const RDesc d = C.desc[s];
      const unsigned char* data = ring + static_cast<size_t>(s) * kChunkBytes;
      const int nvec = (d.bytes + 15) / 16;
      uint4 raw[kRStatVecs];
#pragma unroll
      for (int jj = 0; jj < kRStatVecs; ++jj) {
        const int v = warp * (kRStatVecs * 32) + jj * 32 + lane;
        raw[jj] = v < nvec ? *reinterpret_cast<const uint4*>(data + static_cast<size_t>(v) * 16) : V::neg_inf();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&C.empty[s]);

      const int seg_base = d.part * kPieceElems + warp * kSegElems;
      WPart wp;
      if (GREEDY) {
        float lm = -INFINITY;
        int li = 0x7fffffff, bad = 0;
#pragma unroll
        for (int jj = 0; jj < kRStatVecs; ++jj) {
          float z[NV];
          V::unpack(raw[jj], z);
#pragma unroll
          for (int e = 0; e < NV; ++e) {
            bad |= (z[e] != z[e]) || (z[e] == INFINITY);
            if (z[e] > lm) { lm = z[e]; li = seg_base + (jj * 32 + lane) * NV + e; }
          }
        }
        warp_argmax(lm, li);
        flags |= __reduce_or_sync(0xffffffffu, static_cast<unsigned>(bad)) ? kFBad : 0;
        wp.m = lm; wp.s = __int_as_float(li); wp.zx = 0.f; wp.flags = flags;
      } else {
        // the drafted token's logit, if it lies in this warp's segment
        float zx = 0.f;
        int has = 0;
        if (d.x >= 0 && d.x < P.V) {
          const int rel = d.x - seg_base;
          if (rel >= 0 && rel < kSegElems) {
            const int vv = rel / NV, jj = vv >> 5, e = rel - vv * NV;
            float zz = 0.f;
            if ((vv & 31) == lane) {
#pragma unroll
              for (int j2 = 0; j2 < kRStatVecs; ++j2) {
                if (j2 == jj) {
                  float z[NV];
                  V::unpack(raw[j2], z);
#pragma unroll
                  for (int e2 = 0; e2 < NV; ++e2) if (e2 == e) zz = z[e2];
                }
              }
            }
            zx = __shfl_sync(0xffffffffu, zz, vv & 31);
            has = 1;
          }
        }
        const float lm = V::vmax(raw);
        float ks = -INFINITY, ls = 0.f;
        int bad = 0;
        if (lm > -INFINITY) {
          ks = __fmul_rn(lm, c2);      // fl(m c), used identically wherever rescaled
          const f2 cc = pack2(c2, c2), nk = pack2(-ks, -ks);
          f2 acc[NV / 2];
#pragma unroll
          for (int i = 0; i < NV / 2; ++i) acc[i] = 0ull;
#pragma unroll
          for (int jj = 0; jj < kRStatVecs; ++jj) {
            f2 z[NV / 2];
            V::pairs(raw[jj], z);
#pragma unroll
            for (int i = 0; i < NV / 2; ++i) acc[i] = add2(acc[i], exp2_2(fma2(z[i], cc, nk)));
          }
          float a0, a1;
#pragma unroll
          for (int i = 0; i < NV / 2; ++i) { unpack2(acc[i], a0, a1); ls += a0 + a1; }
        } else {
          // no finite logit in this lane's part: only NaN can still hide here
#pragma unroll
          for (int jj = 0; jj < kRStatVecs; ++jj) {
            float z[NV];
            V::unpack(raw[jj], z);
#pragma unroll
            for (int e = 0; e < NV; ++e) bad |= (z[e] != z[e]);
          }
        }
        const float wM = from_ordered_key(__reduce_max_sync(0xffffffffu, ordered_key(lm)));
        const float wK = wM > -INFINITY ? __fmul_rn(wM, c2) : -INFINITY;
        const float wS = warp_sum(ks > -INFINITY ? ls * fast_exp2(__fsub_rn(ks, wK)) : 0.f);
        flags |= (__reduce_or_sync(0xffffffffu, static_cast<unsigned>(bad)) ? kFBad : 0) | (has ? kFHasZx : 0);
        wp.m = wM; wp.s = wS; wp.zx = zx; wp.flags = flags;
        if (d.kind == 0 && d.pos == d.kb && lane == 0)   // a bonus row: each segment's (fl(m c), sum) for its draw
          P.pw.bseg[(static_cast<size_t>(d.b) * P.np + d.part) * kRWarps + warp] = make_float2(wK, wS);
      }
      // the last warp to finish the piece combines the warps' parts, in
      // warp order, into the piece's record
      const int buf = q % kRBufs;
      int last = 0;
      if (lane == 0) {
        C.part[buf][warp] = wp;
        __threadfence_block();
        last = atomicAdd(&C.cnt[buf], 1) == kRWarps - 1 ? 1 : 0;
      }
      if (__shfl_sync(0xffffffffu, last, 0)) {
        __threadfence_block();
        const bool in = lane < kRWarps;
        const WPart pt = C.part[buf][in ? lane : 0];
        const int fl = static_cast<int>(__reduce_or_sync(0xffffffffu, in ? static_cast<unsigned>(pt.flags) : 0u));
        float4 rec;
        if (GREEDY) {
          float bv = in ? pt.m : -INFINITY;
          int bi = in ? __float_as_int(pt.s) : 0x7fffffff;
          warp_argmax(bv, bi);
          rec = make_float4(bv, __int_as_float(bi), 0.f, __int_as_float(fl));
        } else {
          const float pm = in ? pt.m : -INFINITY;
          const float M = from_ordered_key(__reduce_max_sync(0xffffffffu, ordered_key(pm)));
          const float K = M > -INFINITY ? __fmul_rn(M, c2) : -INFINITY;
          const float pk = pm > -INFINITY ? __fmul_rn(pm, c2) : -INFINITY;
          float sv = (in && pk > -INFINITY) ? pt.s * fast_exp2(__fsub_rn(pk, K)) : 0.f;
#pragma unroll
          for (int o = kRWarps / 2; o > 0; o >>= 1) sv += __shfl_xor_sync(0xffffffffu, sv, o);
          const unsigned hz = __ballot_sync(0xffffffffu, in && (pt.flags & kFHasZx));
          const float zx = __shfl_sync(0xffffffffu, pt.zx, hz ? __ffs(hz) - 1 : 0);
          rec = make_float4(M, __shfl_sync(0xffffffffu, sv, 0), zx, __int_as_float(fl));
        }
        if (lane == 0) {
          P.pw.rec[d.rec] = rec;
          C.cnt[buf] = 0;
        }
        __syncwarp();
      }
    }
  }
};

template <int ELT, bool GREEDY>
__global__ void __launch_bounds__(kRThreads, 1) rows_stats_kernel(const VerifyParams P) {
  extern __shared__ __align__(1024) unsigned char smem[];
  RCtrl& C = *reinterpret_cast<RCtrl*>(smem);
  unsigned char* ring = smem + kRCtrlBytes;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < kRStages; ++s) {
      mbar_init(&C.full[s], 1);
      mbar_init(&C.empty[s], kRWarps);
    }
    for (int i = 0; i < kRBufs; ++i) C.cnt[i] = 0;
    fence_mbar_init();
  }
  grid_dependents_launch();
  // The plan and the producer's copies read only the call's inputs, so they
  // start before the dependency wait, overlapping the previous call's last
  // kernel (the inputs are complete when the call is enqueued); everything
  // that writes the workspace waits first (the consumers, below).
  // The call's plan, in every CTA: rows of the sequences before b, in batch
  // order (2 k_b + 1 each, k_b + 1 for T = 0; none for an invalid k_b)
  const int B = P.B, nw = kRThreads / 32;
  if (tid == 0) C.rowoff[0] = 0;
  int carry = 0;
  for (int base = 0; base < B; base += kRThreads) {
    const int bb = base + tid;
    const int kb = bb < B ? __ldg(P.draft_len + bb) : -1;
    const int cnt = (bb < B && kb >= 0 && kb <= P.k) ? (GREEDY ? kb + 1 : 2 * kb + 1) : 0;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int up = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += up;
    }
    if (lane == 31) C.warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int wt = lane < nw ? C.warp_tot[lane] : 0;
      int wi = wt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int up = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += up;
      }
      if (lane < nw) C.warp_tot[lane] = wi - wt;
    }
    __syncthreads();
    if (bb < B) C.rowoff[bb + 1] = carry + C.warp_tot[warp] + incl;
    __syncthreads();
    carry = C.rowoff[min(B, base + kRThreads)];
  }
  RowStats<ELT, GREEDY> k(P, C, ring, lane, warp);
  if (warp == kRProducer) {
    k.produce();
  } else {
    grid_dependency_wait();      // the previous call no longer reads the records, sums or counters
    if (blockIdx.x == 0 && tid == 0) {
      *P.pw.njobs = 0;
      *P.pw.epoch += 1;
    }
    k.consume();
  }
}

// ---------------------------------------------------------------------------
// rows_decide_kernel: one warp per work-list entry
// ---------------------------------------------------------------------------

// A row's numbers from its pieces' records (lane j holds piece j; np <= 32):
// M the maximum, K = fl(M c), S = sum of the pieces' sums rescaled onto K (a
// fixed butterfly), the drafted token's logit, the flags; greedy: M and the
// first argmax.
template <bool GREEDY>
__device__ void merge_row(const VerifyParams& P, float4 rc, int lane, float& M, float& K, float& S, float& zx,
                          int& flags, int& arg) {
  const bool in = lane < P.np;
  if (!in) rc = make_float4(-INFINITY, 0.f, 0.f, 0.f);
  flags = static_cast<int>(__reduce_or_sync(0xffffffffu, in ? static_cast<unsigned>(__float_as_int(rc.w)) : 0u));
  if (GREEDY) {
    float bv = rc.x;
    int bi = in ? __float_as_int(rc.y) : 0x7fffffff;
    warp_argmax(bv, bi);
    M = bv; arg = bi; K = 0.f; S = 0.f; zx = 0.f;
    return;
  }
  // a NaN part is carried by the flags: the record's sum is NaN
  const float pm = rc.x;
  M = from_ordered_key(__reduce_max_sync(0xffffffffu, ordered_key(pm)));
  K = M > -INFINITY ? __fmul_rn(M, P.c2) : -INFINITY;
  const float pk = pm > -INFINITY ? __fmul_rn(pm, P.c2) : -INFINITY;
  float sv = (in && pk > -INFINITY) ? rc.y * fast_exp2(__fsub_rn(pk, K)) : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sv += __shfl_xor_sync(0xffffffffu, sv, o);
  S = __shfl_sync(0xffffffffu, sv, 0);
  const unsigned hz = __ballot_sync(0xffffffffu, in && (__float_as_int(rc.w) & kFHasZx));
  zx = __shfl_sync(0xffffffffu, rc.z, hz ? __ffs(hz) - 1 : 0);
  arg = 0;
}

template <int ELT, bool GREEDY>
__global__ void __launch_bounds__(kRSmallThreads) rows_decide_kernel(const VerifyParams P) {
  grid_dependency_wait();      // the pieces' records
  grid_dependents_launch();
  const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
  const int b = blockIdx.x * (kRSmallThreads / 32) + wi;
  if (b >= P.B) return;
  const int k = P.k;
  // everything that depends on b alone, in one round trip (the records sit at
  // a fixed stride of 2k + 1 rows per sequence; the first 32 are loaded
  // before the length is known, the unused ones ignored)
  const int kb_in = __ldg(P.draft_len + b);
  const float4 held0 = lane < (GREEDY ? k + 1 : 2 * k + 1) * P.np
                           ? __ldcg(P.pw.rec + static_cast<size_t>(b) * (2 * k + 1) * P.np + lane)
                           : make_float4(-INFINITY, 0.f, 0.f, 0.f);
  const int x_all = lane < k ? __ldg(P.tokens + static_cast<size_t>(b) * k + lane) : -1;
  const float ul = (!GREEDY && lane <= k) ? __ldg(P.uniforms + static_cast<size_t>(b) * (k + 1) + lane) : 0.f;
  if (P.diag) {   // every diagnostic of the sequence NaN first: only the rows read get values
    for (int j = lane; j <= k; j += 32) {
      const size_t i = static_cast<size_t>(b) * (k + 1) + j;
      P.ws.m_t[i] = NAN; P.ws.L_t[i] = NAN; P.ws.mass[i] = NAN;
    }
    for (int j = lane; j < k; j += 32) {
      const size_t i = static_cast<size_t>(b) * k + j;
      P.ws.m_d[i] = NAN; P.ws.L_d[i] = NAN; P.ws.alpha[i] = NAN;
    }
    __syncwarp();
  }
  if (kb_in < 0 || kb_in > k) {
    // an invalid k_b: no rows were read; the sequence emits nothing
    int* ot = P.out_tokens + static_cast<size_t>(b) * (k + 1);
    for (int j = lane; j <= k; j += 32) ot[j] = -1;
    if (lane == 0) {
      P.out_len[b] = 0;
      atomicOr(P.ws.err_word, 1u << 2 /* SV_ERR_BAD_DRAFT_LEN */);
      atomicAdd(P.ws.stats + kStatErrorSeqs, 1ull);
    }
    return;
  }
  const int kb = kb_in;
  const float c2 = P.c2;
  const bool diag = P.diag != 0;
  const int xl = lane < kb ? x_all : -1;
  const float s_samp = __shfl_sync(0xffffffffu, ul, k);
  int a = -1, err = 0, y = -1;
  float pK = 0.f, pS = 0.f, pzx = 0.f;                  // target row of the current pair
  float aKt = 0.f, aLt = 0.f, aGh = 0.f, aGl = 0.f;     // the rejected pair's numbers
  float bK = 0.f, bS = 0.f;                             // the bonus row
  const int nrows = GREEDY ? kb + 1 : 2 * kb + 1;
  const int np = P.np, nrec = nrows * np;
  const float4* recs = P.pw.rec + static_cast<size_t>(b) * (2 * k + 1) * np;
  // the sequence's piece records, 32 at a time (one load per lane, all in
  // flight together); row ri's records are lanes ri np - batch, ...
  int batch = 0;
  float4 held = lane < nrec ? held0 : make_float4(-INFINITY, 0.f, 0.f, 0.f);
  for (int ri = 0; ri < nrows; ++ri) {
    int pos, kind;
    if (GREEDY) { pos = ri; kind = 0; }
    else if (ri < 2 * kb) { pos = ri >> 1; kind = ri & 1; }
    else { pos = kb; kind = 0; }
    if (ri * np + np > batch + 32) {
      batch = ri * np;
      held = batch + lane < nrec ? __ldcg(recs + batch + lane) : make_float4(-INFINITY, 0.f, 0.f, 0.f);
    }
    const int src = min(31, ri * np - batch + lane);
    float4 rc;
    rc.x = __shfl_sync(0xffffffffu, held.x, src);
    rc.y = __shfl_sync(0xffffffffu, held.y, src);
    rc.z = __shfl_sync(0xffffffffu, held.z, src);
    rc.w = __shfl_sync(0xffffffffu, held.w, src);
    float M, K, S, zx;
    int fl, arg;
    merge_row<GREEDY>(P, rc, lane, M, K, S, zx, fl, arg);
    const int x = __shfl_sync(0xffffffffu, xl, pos < kb ? pos : 0);
    if (fl & kFTimeout) err |= kErrTime;
    if (pos < kb && (x < 0 || x >= P.V)) err |= kErrBadTok;
    const size_t bt = static_cast<size_t>(b) * (k + 1) + pos, bd = static_cast<size_t>(b) * k + pos;
    if (GREEDY) {
      if ((fl & kFBad) || !(M > -INFINITY)) err |= kErrNonfin;
      if (diag && lane == 0) P.ws.m_t[bt] = M;
      if (pos < kb) {
        const bool acc = (x == arg);
        if (diag && lane == 0) P.ws.alpha[bd] = acc ? 1.f : 0.f;
        if (!acc && a < 0) { a = pos; y = arg; }
      } else if (a < 0) {
        y = arg;
      }
      continue;
    }
    if ((fl & kFBad) || !(isfinite(M) && isfinite(S) && S > 0.f)) err |= kErrNonfin;
    if (kind == 0) {
      if (diag && lane == 0) { P.ws.m_t[bt] = M; P.ws.L_t[bt] = log2f(S); }
      if (pos < kb) { pK = K; pS = S; pzx = zx; }
      else { bK = K; bS = S; }
    } else {
      if (diag && lane == 0) { P.ws.m_d[bd] = M; P.ws.L_d[bd] = log2f(S); }
      if (!err) {
        // the acceptance test of draft pos (the cluster kernel's arithmetic):
        // delta = (z_d(x) - z_t(x)) c + G, alpha = min(1, 2^-delta)
        float Gh, Gl;
        log2_ratio(pK, pS, K, S, Gh, Gl);
        float alpha;
        if (pzx == -INFINITY) alpha = 0.f;              // p(x) = 0
        else if (zx == -INFINITY) alpha = 1.f;          // q(x) = 0 < p(x)
        else {
          const float delta = __fadd_rn(__fmaf_rn(__fsub_rn(zx, pzx), c2, Gh), Gl);
          alpha = delta <= 0.f ? 1.f : exp2f(-delta);
        }
        if (diag && lane == 0) P.ws.alpha[bd] = alpha;
        const float u = __shfl_sync(0xffffffffu, ul, pos);
        if (!(u < alpha) && a < 0) {
          a = pos;
          aKt = pK; aLt = log2f(pS); aGh = Gh; aGl = Gl;
        }
      }
    }
  }
  if (err || GREEDY) {
    write_outputs(P, b, kb, a, err ? -1 : y, err, 0, xl, lane);
    return;
  }
  if (a >= 0) {
    // the residual draw needs the pair read again: a job for the next kernels
    int j = 0;
    if (lane == 0) j = atomicAdd(P.pw.njobs, 1);
    j = __shfl_sync(0xffffffffu, j, 0);
    if (lane == 0) {
      P.pw.job[j] = make_int4(__float_as_int(s_samp), b, a, kb);
      P.pw.jobn[j] = make_float4(aKt, aLt, aGh, aGl);
    }
    // the accepted prefix and the empty tail now; the draw writes token a
    int* ot = P.out_tokens + static_cast<size_t>(b) * (k + 1);
    if (lane <= k) ot[lane] = lane < a ? xl : -1;
    return;
  }
  // every draft accepted: the bonus token is drawn by the draw kernel, from
  // the bonus row's segment sums; here the accepted prefix and the row's
  // numbers, tagged with the call
  int* ot = P.out_tokens + static_cast<size_t>(b) * (k + 1);
  if (lane <= k) ot[lane] = lane < kb ? xl : -1;
  if (lane == 0)
    P.pw.bonus[b] = make_float4(__int_as_float(__ldcg(P.pw.epoch)), bK, log2f(bS), s_samp);
}

// ---------------------------------------------------------------------------
// rows_resid_kernel: the rejected pairs read again, 16 KB of each row per slot
// ---------------------------------------------------------------------------

template <int ELT>
struct RowResid {
  using V = Vec<ELT>;
  static constexpr int NV = V::N;

  const VerifyParams& P;
  QCtrl& C;
  unsigned char* ring;
  const int lane, warp;
  const long long row_bytes;
  // half-pieces are dealt round robin (this CTA's: blockIdx.x + i * grid), so
  // that the first one's job is known before the job count arrives

  __device__ RowResid(const VerifyParams& p, QCtrl& c, unsigned char* r, int ln, int wp)
      : P(p), C(c), ring(r), lane(ln), warp(wp), row_bytes(static_cast<long long>(p.V) * p.elt) {}

  __device__ void produce() {
    const uint64_t first_out = evict_first_policy();
    const int nr = P.nr, G = gridDim.x;
    // the count and the first job in one round trip; each later job one
    // half-piece ahead
    const int units = __ldcg(P.pw.njobs) * nr;
    int u = blockIdx.x, j = u / nr;
    int4 jb = make_int4(0, 0, 0, 0);
    float4 jn = make_float4(0.f, 0.f, 0.f, 0.f);
    if (j < P.B) { jb = __ldcg(P.pw.job + j); jn = __ldcg(P.pw.jobn + j); }
    for (int q = 0; u < units; u += G, ++q) {
      const int h = u - j * nr;
      const int s = q % kRStages;
      int ok = 1;
      if (lane == 0) ok = mbar_wait_bounded(&C.empty[s], ((q / kRStages) & 1) ^ 1, kDrainLimitNs) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, ok, 0)) {
        if (lane == 0) atomicOr(P.ws.err_word, 1u << 5 /* SV_ERR_TIMEOUT */);
        return;
      }
      if (lane == 0) {
        const long long off = static_cast<long long>(h) * kRHalf;
        const int bytes = static_cast<int>(min(static_cast<long long>(kRHalf), row_bytes - off));
        RDesc& d = C.desc[s];
        d.u = q; d.rec = j; d.part = h; d.bytes = bytes;
        d.b = jb.y; d.kb = jb.w; d.pos = jb.z; d.kind = 2; d.x = -1;
        d.num = jn;
        unsigned char* dst = ring + static_cast<size_t>(s) * kQSlot;
        mbar_expect_tx(&C.full[s], static_cast<uint32_t>(2 * bytes));
        bulk_load_hint(dst, row_ptr(P, jb.y, jb.z, 0) + off, static_cast<uint32_t>(bytes), &C.full[s], first_out);
        bulk_load_hint(dst + kRHalf, row_ptr(P, jb.y, jb.z, 1) + off, static_cast<uint32_t>(bytes), &C.full[s],
                       first_out);
      }
      __syncwarp();
      j = (u + G) / nr;   // the next half-piece's job
      if (u + G < units) { jb = __ldcg(P.pw.job + j); jn = __ldcg(P.pw.jobn + j); }
    }
  }

  // Each warp's segment sums of max(0, p - q) and of p, the residual weights
  // of the cluster kernel (no cancellation where p ~ q).
  __device__ void consume() {
    const float c2 = P.c2;
    const int units = __ldcg(P.pw.njobs) * P.nr;
    for (int u = blockIdx.x, q = 0; u < units; u += gridDim.x, ++q) {
      const int s = q % kRStages;
      bool timed_out = false;
      if (!mbar_wait_bounded(&C.full[s], static_cast<uint32_t>(q / kRStages) & 1u, P.wait_limit_ns)) {
        timed_out = true;
        if (!mbar_wait_bounded(&C.full[s], static_cast<uint32_t>(q / kRStages) & 1u, kDrainLimitNs)) {
          if (lane == 0) atomicOr(P.ws.err_word, 1u << 5 /* SV_ERR_TIMEOUT */);
          return;
        }
      }
      const RDesc d = C.desc[s];
      const unsigned char* data = ring + static_cast<size_t>(s) * kQSlot;
      const int nvec = (d.bytes + 15) / 16;
      uint4 rt[kRDrawVecs], rd[kRDrawVecs];
#pragma unroll
      for (int jj = 0; jj < kRDrawVecs; ++jj) {
        const int v = warp * (kRDrawVecs * 32) + jj * 32 + lane;
        const bool in = v < nvec;
        rt[jj] = in ? *reinterpret_cast<const uint4*>(data + static_cast<size_t>(v) * 16) : V::neg_inf();
        rd[jj] = in ? *reinterpret_cast<const uint4*>(data + kRHalf + static_cast<size_t>(v) * 16) : V::neg_inf();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&C.empty[s]);
      const f2 cc = pack2(c2, c2), nkt = pack2(-d.num.x, -d.num.x), nlt = pack2(-d.num.y, -d.num.y);
      const f2 gh = pack2(d.num.z, d.num.z), gl = pack2(d.num.w, d.num.w);
      f2 accr[NV / 2], accp[NV / 2];
#pragma unroll
      for (int i = 0; i < NV / 2; ++i) { accr[i] = 0ull; accp[i] = 0ull; }
#pragma unroll
      for (int jj = 0; jj < kRDrawVecs; ++jj) {
        f2 zt[NV / 2], zd[NV / 2];
        V::pairs(rt[jj], zt);
        V::pairs(rd[jj], zd);
#pragma unroll
        for (int i = 0; i < NV / 2; ++i) {
          // the residual weights of resid_weight2, with the series taken two
          // lanes per f32x2 instruction (bit-identical, lane by lane)
          const f2 p = exp2_2(add2(fma2(zt[i], cc, nkt), nlt));
          const f2 delta = add2(fma2(sub2(zd[i], zt[i]), cc, gh), gl);
          float w0, w1;
          unpack2(mul2(p, one_minus_exp2_2r(delta)), w0, w1);
          accr[i] = add2(accr[i], pack2(fmaxf(w0, 0.f), fmaxf(w1, 0.f)));
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
        const size_t g = (static_cast<size_t>(d.rec) * P.nr + d.part) * kRWarps + warp;
        P.pw.rmass[g] = timed_out ? NAN : wr;
        P.pw.pmass[g] = timed_out ? NAN : wp;
      }
    }
  }
};

template <int ELT>
__global__ void __launch_bounds__(kRThreads, 2) rows_resid_kernel(const VerifyParams P) {
  extern __shared__ __align__(1024) unsigned char smem[];
  QCtrl& C = *reinterpret_cast<QCtrl*>(smem);
  unsigned char* ring = smem + kQCtrlBytes;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < kRStages; ++s) {
      mbar_init(&C.full[s], 1);
      mbar_init(&C.empty[s], kRWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  grid_dependency_wait();      // the jobs
  grid_dependents_launch();
  RowResid<ELT> k(P, C, ring, lane, warp);
  if (warp == kRProducer) k.produce();
  else k.consume();
}

// ---------------------------------------------------------------------------
// rows_draw_kernel: one warp per job, the residual draw
// ---------------------------------------------------------------------------
// The bonus draw of sequence b, if every draft of it was accepted in this
// call (one warp; wm: kMaxChunks * kRWarps floats of shared scratch): the
// segment holding s * S among the bonus row's segment sums, kept while it
// streamed, then that segment read again.
template <int ELT>
__device__ void bonus_draw(const VerifyParams& P, int b, int lane, float* wm) {
  const int k = P.k;
  // the row's numbers, the call number, the length and the segment sums in one round trip
  const float4 bo = __ldcg(P.pw.bonus + b);
  const int ep = __ldcg(P.pw.epoch);
  const int kb = __ldg(P.draft_len + b);
  const int nseg = P.np * kRWarps;
  float2 bsg[kMaxChunks * kRWarps / 32];
#pragma unroll
  for (int i = 0; i < kMaxChunks * kRWarps / 32; ++i) {
    const int g = lane + 32 * i;
    bsg[i] = g < nseg ? __ldcg(P.pw.bseg + static_cast<size_t>(b) * nseg + g) : make_float2(-INFINITY, 0.f);
  }
  if (__float_as_int(bo.x) != ep) return;   // not a fully accepted sequence of this call
  const float bK = bo.y, L = bo.z, s_samp = bo.w;
#pragma unroll
  for (int i = 0; i < kMaxChunks * kRWarps / 32; ++i) {
    const int g = lane + 32 * i;
    if (g < nseg) wm[g] = bsg[i].x == -INFINITY ? 0.f : bsg[i].y * fast_exp2(__fsub_rn(bsg[i].x, bK) - L);
  }
  __syncwarp();
  float part = 0.f;
  {
    const int per = (nseg + 31) / 32;
    const int g0 = min(nseg, lane * per), g1 = min(nseg, g0 + per);
    for (int g = g0; g < g1; ++g) part += wm[g];
  }
  const float tot = warp_sum(part);
  int seg;
  float seg_t;
  locate_seg(wm, nseg, s_samp * tot, lane, seg, seg_t);
  if (P.diag && lane == 0) P.ws.mass[static_cast<size_t>(b) * (k + 1) + kb] = tot;
  const int nvec_row = static_cast<int>((static_cast<long long>(P.V) * ELT) / 16);
  int y = -1;
  if (seg >= 0) {
    const int v0 = (seg / kRWarps) * (kChunkBytes / 16) + (seg % kRWarps) * (kRStatVecs * 32);
    y = walk_seg<ELT, kRStatVecs, false>(row_ptr(P, b, kb, 0), nullptr, v0, nvec_row, seg_t, P.c2, bK, L, 0.f, 0.f,
                                        lane);
  }
  write_outputs(P, b, kb, -1, y, 0, 0, -1, lane, true);
}

// Warps [0, B): the residual draw of job w; warps [B, 2B): the bonus draw of
// sequence w - B.
template <int ELT>
__global__ void __launch_bounds__(kRSmallThreads) rows_draw_kernel(const VerifyParams P) {
  __shared__ float bmass[kRSmallThreads / 32][kMaxChunks * kRWarps];
  grid_dependency_wait();      // the re-read masses
  grid_dependents_launch();    // the next call's statistics kernel may start reading its inputs
  const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
  const int w = blockIdx.x * (kRSmallThreads / 32) + wi;
  if (w >= 2 * P.B) return;
  if (w >= P.B) {
    bonus_draw<ELT>(P, w - P.B, lane, bmass[wi]);
    return;
  }
  const int j = w;
  // the job, its numbers and masses with the job count, in one round trip
  // (j < B: in bounds whether or not it is a job of this call)
  const int njobs = __ldcg(P.pw.njobs);
  const int4 jb = __ldcg(P.pw.job + j);
  const float4 jn = __ldcg(P.pw.jobn + j);
  const int nseg = P.nr * kRWarps;
  const float* rm = P.pw.rmass + static_cast<size_t>(j) * nseg;
  const float* pm = P.pw.pmass + static_cast<size_t>(j) * nseg;
  const int per = (nseg + 31) / 32;
  const int g0 = min(nseg, lane * per), g1 = min(nseg, g0 + per);
  float r = 0.f, pp = 0.f;
  for (int g = g0; g < g1; ++g) {   // (issued with the job's load: they depend on j alone)
    r += __ldcg(rm + g);
    pp += __ldcg(pm + g);
  }
  if (j >= njobs) return;
  const int b = jb.y, a = jb.z, kb = jb.w, k = P.k;
  const float rtot = warp_sum(r);
  // exact arithmetic rules a zero residual out (a rejection implies p > q
  // somewhere); if rounding leaves none, the draw is from p_a (counted)
  const bool resid = rtot > 0.f;
  const float tot = resid ? rtot : warp_sum(pp);
  int err = (rtot != rtot || tot != tot) ? kErrTime : 0;   // a timed-out re-read left NaN
  const float s = __int_as_float(jb.x);   // the sampling uniform, carried by the job
  int seg;
  float seg_t;
  locate_seg(resid ? rm : pm, nseg, s * tot, lane, seg, seg_t);
  if (P.diag && lane == 0) P.ws.mass[static_cast<size_t>(b) * (k + 1) + a] = tot;
  int y = -1;
  if (!err && seg >= 0) {
    const int nvec_row = static_cast<int>((static_cast<long long>(P.V) * ELT) / 16);
    const int v0 = (seg / kRWarps) * (kRHalf / 16) + (seg % kRWarps) * (kRDrawVecs * 32);
    const unsigned char* rowT = row_ptr(P, b, a, 0);
    if (resid)
      y = walk_seg<ELT, kRDrawVecs, true>(rowT, row_ptr(P, b, a, 1), v0, nvec_row, seg_t, P.c2, jn.x, jn.y, jn.z,
                                          jn.w, lane);
    else
      y = walk_seg<ELT, kRDrawVecs, false>(rowT, nullptr, v0, nvec_row, seg_t, P.c2, jn.x, jn.y, 0.f, 0.f, lane);
  }
  write_outputs(P, b, kb, a, y, err, resid ? 0 : 1, -1, lane, true);
}

cudaError_t launch_dep(void (*fn)(const VerifyParams), int grid, int threads, int smem, cudaStream_t s,
                       const VerifyParams& p) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, p);
}

template <int ELT, bool GREEDY>
cudaError_t launch_rows(const VerifyParams& p, cudaStream_t s) {
  const int smem = kRCtrlBytes + kRStages * kChunkBytes;
  const int small = (p.B + kRSmallThreads / 32 - 1) / (kRSmallThreads / 32);
  // grids no larger than the most work a batch of this shape can hold
  const long long most_pieces = static_cast<long long>(p.B) * (GREEDY ? p.k + 1 : 2 * p.k + 1) * p.np;
  const long long most_halves = static_cast<long long>(p.B) * p.nr;
  const int stats_ctas = static_cast<int>(min(static_cast<long long>(p.ctas), most_pieces));
  const int resid_ctas = static_cast<int>(min(2LL * p.ctas, most_halves));
  cudaError_t e = launch_dep(rows_stats_kernel<ELT, GREEDY>, stats_ctas, kRThreads, smem, s, p);
  if (e == cudaSuccess) e = launch_dep(rows_decide_kernel<ELT, GREEDY>, small, kRSmallThreads, 0, s, p);
  if (!GREEDY) {
    if (e == cudaSuccess) e = launch_dep(rows_resid_kernel<ELT>, resid_ctas, kRThreads, kQSmem, s, p);
    if (e == cudaSuccess) e = launch_dep(rows_draw_kernel<ELT>, 2 * small, kRSmallThreads, 0, s, p);
  }
  return e;
}

}  // namespace

int pieces_smem_bytes() { return kRCtrlBytes + kRStages * kChunkBytes; }
int pieces_threads() { return kRThreads; }

cudaError_t prepare_pieces_kernel() {
  const void* fns[4] = {reinterpret_cast<const void*>(&rows_stats_kernel<2, false>),
                        reinterpret_cast<const void*>(&rows_stats_kernel<4, false>),
                        reinterpret_cast<const void*>(&rows_stats_kernel<2, true>),
                        reinterpret_cast<const void*>(&rows_stats_kernel<4, true>)};
  for (const void* f : fns) {
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, pieces_smem_bytes());
    if (e != cudaSuccess) return e;
  }
  const void* resid[2] = {reinterpret_cast<const void*>(&rows_resid_kernel<2>),
                          reinterpret_cast<const void*>(&rows_resid_kernel<4>)};
  for (const void* f : resid) {
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_pieces(const VerifyParams& p, cudaStream_t s) {
  NvtxRange range("spec_verify_rows");
  if (p.greedy) return p.elt == 2 ? launch_rows<2, true>(p, s) : launch_rows<4, true>(p, s);
  return p.elt == 2 ? launch_rows<2, false>(p, s) : launch_rows<4, false>(p, s);
}

}  // namespace sv
