// Tree verification: recursive rejection sampling over a draft tree.
//
// "ReSpec: Towards Optimizing Speculative Decoding in Reinforcement Learning
// Systems" (GAP 1) configures speculation by rounds, a branching factor and a
// draft length; the page gives no rule for verifying branching drafts.  The
// reading implemented here takes the children of a node as independent draws
// from the drafter's distribution q at that node and tests them in index
// order against a residual r that starts at the target distribution p:
//
//   child c with token x is accepted iff u_c < min(1, r(x) / q(x));
//   after a rejection r <- max(0, r - q) / S, S its mass (S = 0: r is kept);
//   an accepted child emits its token and the walk continues at it;
//   if every child is rejected, y is drawn from the last residual, and at a
//   node without children y is the bonus token drawn from p;
//   the draw is the inverse CDF in token order with the sampling uniform
//   s = u[b, 0]; T == 0 accepts the first child equal to the first argmax of
//   the node's target row and emits that argmax.
//
// A cluster of cs CTAs walks one sequence: each CTA owns a contiguous slice
// of every row (whole 256-logit chunks), and the slices' partial sums are
// exchanged through distributed shared memory and combined in rank order, so
// every CTA takes the same decisions.  cs is the largest of 8, 4, 2, 1 that
// keeps one CTA per SM for the whole batch.  Within a CTA a producer warp
// streams the slice of the rows a pass needs (the node's target row and, with
// children, its draft row) through three 32 KB shared-memory slots with
// cp.async.bulk, 16 KB of each row per slot, and 8 consumer warps reduce
// each slot, two logits per f32x2 instruction.  Two such CTAs fit on an SM
// (about 103 KB of shared memory and at most 112 registers a thread), so the
// walks of back-to-back calls share the SMs.  Each visited node costs one
// pass for the row maximum and log-sum of 2^(z c) of both rows, one more pass
// per rejected child (the residual mass, with the sum of each warp's
// 128-vector segment kept for the draw) and one pass for a bonus draw; the
// later passes find the rows in L2.  Only the rows the walk visits are read.
// Every reduction runs in a fixed order, so the result is deterministic.

#include <cuda_runtime.h>

#include <cmath>
#include <cstddef>
#include <cstdint>

#include "../../include/specverify.h"
#include "sv_device.cuh"

namespace sv {
namespace {

constexpr int kTreeWarps = 8;                           // consumer warps
constexpr int kTreeThreads = (kTreeWarps + 1) * 32;     // + the producer warp
constexpr int kTreeProducer = kTreeWarps;               // its warp index
constexpr int kTreeStages = 3;                          // 32 KB staging slots
constexpr int kTreeHalf = 16 * 1024;                    // bytes of one row per slot
constexpr int kTreeVecsPerWarp = kTreeHalf / 16 / kTreeWarps;   // 128: one segment
constexpr int kTreeVecsPerLane = kTreeVecsPerWarp / 32;         // 4
constexpr int kChunkElems = 256;                        // slice boundaries: whole 256-logit chunks
constexpr int kTreeMaxV = 524288;
constexpr int kTreeMaxSegs = (kTreeMaxV * 4 / kTreeHalf) * kTreeWarps;   // 1024
constexpr int kTreeMaxNodes = SV_TREE_MAX_NODES;
constexpr int kTreeMaxCluster = 8;
constexpr int kTreeRingBytes = kTreeStages * 2 * kTreeHalf;

struct TreeParams {
  const unsigned char* target;   // [B, M, V]
  const unsigned char* draft;    // [B, M, V]
  const int32_t* parents;        // [B, M]
  const int32_t* tokens;         // [B, M]
  const int32_t* n_nodes;        // [B]
  const float* uniforms;         // [B, M]
  int32_t* out_tokens;           // [B, M]
  int32_t* out_nodes;            // [B, M]
  int32_t* out_len;              // [B]
  int32_t* status;               // [B] or null
  float* alpha;                  // [B, M] or null
  int B, M, V;
  int vec;                       // rows 16-byte aligned: bulk copies and vector loads
  float c2;                      // log2(e) / T
  int cs;                        // CTAs per sequence (the cluster): each streams a slice of every row
};

// Sixteen bytes of logits from element e0 of a row, straight from global
// memory (the draw's re-read): -inf past V; element loads for unaligned rows.
template <int ELT>
__device__ __forceinline__ uint4 load_vec(const unsigned char* row, int e0, int V, int vec) {
  using VV = Vec<ELT>;
  if (vec && e0 + VV::N <= V) return __ldg(reinterpret_cast<const uint4*>(row + static_cast<size_t>(e0) * ELT));
  unsigned char buf[16];
#pragma unroll
  for (int e = 0; e < VV::N; ++e) VV::store_scalar(buf, e, e0 + e < V ? VV::scalar(row, e0 + e) : -INFINITY);
  return *reinterpret_cast<const uint4*>(buf);
}

// What a CTA contributes to one exchange of its cluster (three 16-byte
// words, read by a peer with three vector loads).
struct __align__(16) XSlot {
  float Kt, St, Kd, Sd;     // row statistics of its slice (greedy: Kt = best logit, St = draft maximum)
  int bad, idx, y, failed;  // a bad logit seen; greedy argmax; the drawn token; a bounded wait gave up
  double total, pad2;       // its slice's weight
};

// Per-CTA scratch for the walk.
struct TreeShared {
  uint64_t full[kTreeStages];        // slot filled (producer -> consumer warps)
  uint64_t empty[kTreeStages];       // slot released (one arrival per consumer warp)
  int par[kTreeMaxNodes], tok[kTreeMaxNodes];
  float u[kTreeMaxNodes];
  int kids[kTreeMaxNodes];
  int nkids, n, cur, len, st, next, y, owner;
  int pass_both;                     // the pass streams the draft row too
  int failed;                        // a bounded wait of the streaming gave up
  int lastq[kTreeStages];            // producer: the last slot count copied into each stage (-1: none)
  float csum[kTreeMaxSegs];          // segment sums of the last weight pass (this CTA's segments)
  double cc, PP, invPP;              // residual after the rejections so far: max(0, p - cc q) / PP
  double l2ratio;                    // log2(S^t / S^d) of the current node
  float wA, wGh, wGl;                // weights of the last pass: max(0, A 2^(z^t c - K^t) - B 2^(z^d c - K^d)),
                                     // as A 2^(z^t c - K^t) (1 - 2^delta), delta = (z^d - z^t) c + Gh + Gl
  float wm[kTreeWarps], ws[kTreeWarps], wmd[kTreeWarps], wsd[kTreeWarps];
  int wbad[kTreeWarps], widx[kTreeWarps];
  float Kt, St, Kd, Sd;              // row statistics of the current node (whole row)
  float myKt, mySt, myKd, mySd;      // the same for this CTA's slice
  double total;                      // weight of the last pass (whole row)
  double mytotal;                    // ... of this CTA's slice
  double base[kTreeMaxCluster];      // weight of the slices before each CTA's
  double slice[kTreeMaxCluster];     // weight of each CTA's slice
  XSlot xs[2];                       // exchange slots (double-buffered)
  XSlot got[kTreeMaxCluster];        // the slots of the last exchange, rank order
  // the outputs, written to global memory only at the end (after the
  // dependency wait: the previous call on the stream may still write them)
  int otok[kTreeMaxNodes], onode[kTreeMaxNodes];
  float oal[kTreeMaxNodes];
};

__device__ __forceinline__ uint4 ld_peer_v4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a) : "memory");
  return v;
}

// One exchange: thread 0 has filled sh.xs[xp].  After the cluster barrier
// every CTA's slot is visible; thread r < cs copies rank r's slot into
// sh.got[r] (three 16-byte loads), so that thread 0 then merges them in rank
// order from local shared memory.  The slots are double-buffered: a CTA
// writes a slot again only after the next barrier, which every peer reaches
// only after reading it.  Each slot also carries whether a bounded wait of
// its CTA gave up, and every CTA takes the OR: the walk ends at the same
// step in all of them (a CTA that stopped alone would leave its peers at a
// cluster barrier that it never reaches).
__device__ __forceinline__ void exchange(TreeShared& sh, int& xp, int cs) {
  if (threadIdx.x == 0) sh.xs[xp].failed = *reinterpret_cast<volatile int*>(&sh.failed);
  cluster_sync();
  const int t = threadIdx.x;
  if (t < cs) {
    const uint32_t a = peer(&sh.xs[xp], t);
    uint4* dst = reinterpret_cast<uint4*>(&sh.got[t]);
    dst[0] = ld_peer_v4(a);
    dst[1] = ld_peer_v4(a + 16);
    dst[2] = ld_peer_v4(a + 32);
  }
  __syncthreads();
  if (t == 0) {
    int f = 0;
    for (int r = 0; r < cs; ++r) f |= sh.got[r].failed;
    if (f) *reinterpret_cast<volatile int*>(&sh.failed) = 1;
  }
  xp ^= 1;
}

// Merge of (K, S) pairs, S = sum 2^(z c - K), K = fl(max z * c): the larger
// K wins and the other sum is rescaled.  (-inf, 0) is the empty pair.
__device__ __forceinline__ void merge_ks(float& K, float& S, float K2, float S2) {
  if (!(S2 > 0.f)) return;
  if (!(S > 0.f)) {
    K = K2;
    S = S2;
    return;
  }
  if (K2 > K) {
    S = S * fast_exp2(K - K2) + S2;
    K = K2;
  } else {
    S += S2 * fast_exp2(K2 - K);
  }
}

// CTA-wide (K, S) of the consumer lanes' running (max, K, sum) triples, in
// warp order (thread 0).  Every thread of the CTA calls it.
__device__ void combine_stats(float m, float K, float s, float& Kout, float& Sout, float* wm, float* ws, float c2) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float M = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float KM = M * c2;
  float v = (m == -INFINITY) ? 0.f : s * fast_exp2(K - KM);
  v = warp_sum(v);
  if (lane == 0 && warp < kTreeWarps) {
    wm[warp] = M;
    ws[warp] = v;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float Mall = -INFINITY;
    for (int w = 0; w < kTreeWarps; ++w) Mall = fmaxf(Mall, wm[w]);
    const float Kall = Mall * c2;
    float S = 0.f;
    for (int w = 0; w < kTreeWarps; ++w)
      if (wm[w] != -INFINITY) S += ws[w] * fast_exp2(wm[w] * c2 - Kall);
    Kout = (Mall == -INFINITY) ? -INFINITY : Kall;
    Sout = (Mall == -INFINITY) ? 0.f : S;
  }
}

// Residual after h rejections at a node, in closed form: with r_1 = p and
// r_{h+1} = max(0, r_h - q) / S_h (or r_h / S_h when S_h was zero and r was
// kept), r_{h+1} = max(0, p - c_h q) / P_h where c_0 = 0, P_0 = 1,
// c_h = c_{h-1} + P_{h-1} (c unchanged when r was kept), P_h = P_{h-1} S_h.
// A weight pass therefore needs, per logit pair, only
//   w = max(0, A e^t - B e^d),  e = 2^(z c - K) (unnormalised p and q),
// with A, B fixed for the pass: the bonus weights are A = 1, B = 0; the
// residual after one more rejection A = 1 / (S^t P), B = (c + P) / (S^d P);
// r itself (zero-residual fallback) A = 1 / (S^t P), B = c / (S^d P).
// The difference is taken without cancellation where A e^t ~ B e^d:
//   w = A e^t (1 - 2^delta),  delta = (z^d - z^t) c + G,
//   G = log2(B / A) + K^t - K^d  (in double, held as Gh + Gl; B = 0 gives
//   Gh = -inf, Gl = 0, so w = A e^t).
__device__ __forceinline__ float pair_weight(float zt, float zd, float c2, float Kt, float A, float Gh, float Gl) {
  const float et = fast_exp2(__fmaf_rn(zt, c2, -Kt));
  const float delta = __fadd_rn(__fmaf_rn(__fsub_rn(zd, zt), c2, Gh), Gl);
  return fmaxf(__fmul_rn(__fmul_rn(A, et), one_minus_exp2(delta)), 0.f);
}
// The same for two logit pairs at once (bit-identical, lane by lane).
__device__ __forceinline__ void pair_weight2(f2 zt, f2 zd, f2 cc, f2 nkt, f2 aa, f2 gh, f2 gl, float& w0, float& w1) {
  const f2 et = exp2_2(fma2(zt, cc, nkt));
  const f2 delta = add2(fma2(sub2(zd, zt), cc, gh), gl);
  unpack2(mul2(mul2(aa, et), one_minus_exp2_2r(delta)), w0, w1);
  w0 = fmaxf(w0, 0.f);
  w1 = fmaxf(w1, 0.f);
}
// The bonus weight: no draft row (K^d may be -inf at a node without children).
__device__ __forceinline__ float bonus_weight(float zt, float c2, float Kt) { return fast_exp2(fmaf(zt, c2, -Kt)); }

// Fixed-order fp64 total of the segment sums [0, nseg): lane l adds a
// contiguous run of segments in order, then the lanes are scanned.
__device__ __forceinline__ double seg_total(const TreeShared& sh, int nseg, int lane, double& excl, int& lo, int& hi) {
  const int per = (nseg + 31) / 32;
  lo = min(lane * per, nseg);
  hi = min(lo + per, nseg);
  double part = 0.0;
  for (int c = lo; c < hi; ++c) part += static_cast<double>(sh.csum[c]);
  const double incl = warp_incl_scan(part, lane);
  excl = incl - part;
  return __shfl_sync(0xffffffffu, incl, 31);
}

// This CTA's slice of every row, streamed through the slots.  The producer
// warp and the consumer warps run the same passes in the same order and count
// the slots alike (q), so the slots' mbarrier phases match.  Every wait is
// bounded; one that gives up sets sh.failed, after which no wait is made and
// the walk ends with SV_ERR_TIMEOUT, in every CTA of the cluster at the same
// step (the flag travels with each exchange); the producer drains its copies
// before the CTA leaves.
template <int ELT>
struct Slice {
  using VV = Vec<ELT>;
  static constexpr int NV = VV::N;
  static constexpr int kSegElems = kTreeVecsPerWarp * NV;   // logits per segment (one warp's share of a slot)
  static constexpr int kSlotElems = kTreeHalf / ELT;        // logits of one row per slot

  TreeShared& sh;
  unsigned char* ring;
  const TreeParams& P;
  int e_lo;        // first logit of the slice
  int bytes;       // bytes of one row's slice
  int nsl;         // slots per pass
  int q;           // slots streamed so far

  __device__ Slice(TreeShared& s, unsigned char* r, const TreeParams& p, int c_lo, int c_hi)
      : sh(s), ring(r), P(p), q(0) {
    e_lo = min(p.V, c_lo * kChunkElems);
    const int e_hi = min(p.V, c_hi * kChunkElems);
    bytes = (e_hi - e_lo) * ELT;
    nsl = (bytes + kTreeHalf - 1) / kTreeHalf;
  }

  __device__ int nseg() const { return nsl * kTreeWarps; }
  __device__ int slot_bytes(int k) const {
    const int left = bytes - k * kTreeHalf;
    return left < kTreeHalf ? left : kTreeHalf;
  }
  __device__ unsigned char* slot(int s) const { return ring + static_cast<size_t>(s) * 2 * kTreeHalf; }
  __device__ bool failed() const { return *reinterpret_cast<volatile int*>(&sh.failed) != 0; }
  __device__ void fail() { *reinterpret_cast<volatile int*>(&sh.failed) = 1; }
  // first logit of segment g (slot g / 16, warp g % 16)
  __device__ int seg_e0(int g) const { return e_lo + (g / kTreeWarps) * kSlotElems + (g % kTreeWarps) * kSegElems; }

  // Producer warp: the pass's rows, one slot at a time.
  __device__ void produce(const unsigned char* rt, const unsigned char* rd, bool both) {
    const int lane = threadIdx.x & 31;
    for (int k = 0; k < nsl; ++k, ++q) {
      const int s = q % kTreeStages;
      int ok = 1;
      if (lane == 0) ok = (!failed() && mbar_wait_bounded(&sh.empty[s], ((q / kTreeStages) & 1) ^ 1, kDrainLimitNs)) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, ok, 0)) {
        if (lane == 0) fail();
        continue;
      }
      const int nb = slot_bytes(k);
      const size_t off = static_cast<size_t>(e_lo) * ELT + static_cast<size_t>(k) * kTreeHalf;
      unsigned char* dst = slot(s);
      if (P.vec) {
        if (lane == 0) {
          mbar_expect_tx(&sh.full[s], static_cast<uint32_t>((both ? 2 : 1) * nb));
          bulk_load(dst, rt + off, static_cast<uint32_t>(nb), &sh.full[s]);
          if (both) bulk_load(dst + kTreeHalf, rd + off, static_cast<uint32_t>(nb), &sh.full[s]);
          sh.lastq[s] = q;
        }
      } else {
        // rows not 16-byte aligned: element loads, the last vector padded with -inf
        const int e0 = e_lo + k * kSlotElems;
        const int n = nb / ELT;
        const int npad = (n + NV - 1) / NV * NV;
        for (int e = lane; e < npad; e += 32) {
          VV::store_scalar(dst, e, e < n ? VV::scalar(rt, e0 + e) : -INFINITY);
          if (both) VV::store_scalar(dst + kTreeHalf, e, e < n ? VV::scalar(rd, e0 + e) : -INFINITY);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.full[s]);
      }
    }
  }

  // Consumer warps: f(k, tv, dv) for each slot k with this lane's vectors of
  // the target (and draft) row, -inf past the slice; a slot is released as
  // soon as its vectors are in registers.
  template <typename F>
  __device__ void consume(bool both, F&& f) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int k = 0; k < nsl; ++k, ++q) {
      const int s = q % kTreeStages;
      bool ok = !failed() && mbar_wait_bounded(&sh.full[s], static_cast<uint32_t>(q / kTreeStages) & 1u, kDrainLimitNs);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok && lane == 0) fail();
      const int nvec = (slot_bytes(k) + 15) / 16;
      const unsigned char* src = slot(s);
      uint4 tv[kTreeVecsPerLane], dv[kTreeVecsPerLane];
#pragma unroll
      for (int j = 0; j < kTreeVecsPerLane; ++j) {
        const int v = warp * kTreeVecsPerWarp + j * 32 + lane;
        const bool in = v < nvec;
        tv[j] = in ? *reinterpret_cast<const uint4*>(src + static_cast<size_t>(v) * 16) : VV::neg_inf();
        dv[j] = (in && both) ? *reinterpret_cast<const uint4*>(src + kTreeHalf + static_cast<size_t>(v) * 16)
                             : VV::neg_inf();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.empty[s]);
      f(k, tv, dv);
    }
  }

  // Producer warp, before the CTA leaves: every copy it issued has landed
  // (bounded).  On the normal path the consumers waited for each already;
  // after a wait gave up, copies still in flight must not reach shared
  // memory that a later CTA owns.
  __device__ void drain() {
    if ((threadIdx.x & 31) != 0) return;
#pragma unroll
    for (int s = 0; s < kTreeStages; ++s)
      if (sh.lastq[s] >= 0)
        mbar_wait_bounded(&sh.full[s], static_cast<uint32_t>(sh.lastq[s] / kTreeStages) & 1u, kDrainLimitNs);
  }

  // One pass: the producer warp streams, the consumer warps reduce.
  template <typename F>
  __device__ void pass(const unsigned char* rt, const unsigned char* rd, bool both, F&& f) {
    if ((threadIdx.x >> 5) == kTreeProducer) produce(rt, rd, both);
    else consume(both, f);
  }
};

// Running (max, K = fl(max c), sum 2^(z c - K)) of one lane, updated by its
// vectors of one slot (a larger maximum rescales the sum).
template <int ELT>
__device__ __forceinline__ void online_vecs(const uint4 (&v)[kTreeVecsPerLane], float c2, float& m, float& K, f2& s,
                                            int& bad) {
  using VV = Vec<ELT>;
  const float vm = VV::vmax_nan(v);                  // NaN survives the maximum
  bad |= (vm != vm) || (vm == INFINITY);
  if (vm > m) {
    const float Kn = vm * c2;
    const float f = (m == -INFINITY) ? 0.f : fast_exp2(K - Kn);
    s = mul2(s, pack2(f, f));
    m = vm;
    K = Kn;
  }
  if (m != -INFINITY) {
    const f2 cc = pack2(c2, c2), nk = pack2(-K, -K);
#pragma unroll
    for (int j = 0; j < kTreeVecsPerLane; ++j) {
      f2 z[VV::N / 2];
      VV::pairs(v[j], z);
#pragma unroll
      for (int i = 0; i < VV::N / 2; ++i) s = add2(s, exp2_2(fma2(z[i], cc, nk)));
    }
  }
}

// One pass of weights over this CTA's slice of the current node's rows:
// segment sums into sh.csum, then the slices' weights exchanged in the
// cluster (sh.slice, sh.base, sh.total, identical in every CTA).
//   mode 0: bonus weights (A = 1, B = 0; the draft row is not read);
//   mode 1: the residual after one more rejection;
//   mode 2: the current residual r itself (zero-residual fallback).
template <int ELT>
__device__ void weight_pass(TreeShared& sh, Slice<ELT>& sl, const TreeParams& P, const unsigned char* rt,
                            const unsigned char* rd, int mode, int& xp) {
  using VV = Vec<ELT>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    sh.wA = mode == 0 ? 1.f : static_cast<float>(sh.invPP * (1.0 / static_cast<double>(sh.St)));
    sh.wGh = -INFINITY;
    sh.wGl = 0.f;
    const double cB = mode == 1 ? sh.cc + sh.PP : sh.cc;
    if (mode != 0 && cB > 0.0) {
      // log2(B / A) = log2(c_B) + log2(S^t / S^d)
      const double G = log2(cB) + sh.l2ratio + (static_cast<double>(sh.Kt) - static_cast<double>(sh.Kd));
      sh.wGh = static_cast<float>(G);
      sh.wGl = static_cast<float>(G - static_cast<double>(sh.wGh));
    }
  }
  __syncthreads();
  const float c2 = P.c2;
  const f2 cc = pack2(c2, c2), nkt = pack2(-sh.Kt, -sh.Kt), aa = pack2(sh.wA, sh.wA);
  const f2 gh = pack2(sh.wGh, sh.wGh), gl = pack2(sh.wGl, sh.wGl);
  sl.pass(rt, rd, mode != 0, [&](int k, const uint4 (&tv)[kTreeVecsPerLane], const uint4 (&dv)[kTreeVecsPerLane]) {
    float part = 0.f;
#pragma unroll
    for (int j = 0; j < kTreeVecsPerLane; ++j) {
      f2 zt[VV::N / 2], zd[VV::N / 2];
      VV::pairs(tv[j], zt);
      if (mode != 0) VV::pairs(dv[j], zd);
#pragma unroll
      for (int i = 0; i < VV::N / 2; ++i) {
        float w0, w1;
        if (mode == 0) unpack2(exp2_2(fma2(zt[i], cc, nkt)), w0, w1);
        else pair_weight2(zt[i], zd[i], cc, nkt, aa, gh, gl, w0, w1);
        part += w0;
        part += w1;
      }
    }
    part = warp_sum(part);
    if (lane == 0) sh.csum[k * kTreeWarps + warp] = part;
  });
  __syncthreads();
  if (warp == 0) {
    double excl;
    int lo, hi;
    const double tot = seg_total(sh, sl.nseg(), lane, excl, lo, hi);
    if (lane == 0) {
      sh.mytotal = tot;
      sh.xs[xp].total = tot;
    }
  }
  __syncthreads();
  exchange(sh, xp, P.cs);
  if (threadIdx.x == 0) {
    double acc = 0.0;
    for (int r = 0; r < P.cs; ++r) {
      const double t = sh.got[r].total;
      sh.base[r] = acc;
      sh.slice[r] = t;
      acc += t;
    }
    sh.total = acc;
  }
  __syncthreads();
}

// Inverse CDF with the sampling uniform over the weights of the last pass,
// for the CTA whose slice holds the point (warp 0): the segment from the
// segment sums, then the logit from the segment's recomputed weights, in
// index order.  `last`: the point lies past every weight (rounding); take
// the last logit with weight.
template <int ELT>
__device__ int draw(TreeShared& sh, const Slice<ELT>& sl, const TreeParams& P, const unsigned char* rt,
                    const unsigned char* rd, int mode, double t, double slice_base, bool last) {
  using VV = Vec<ELT>;
  constexpr int NV = VV::N;
  const int lane = threadIdx.x & 31;
  const int V = P.V;
  const int e_end = sl.e_lo + sl.bytes / ELT;   // end of this CTA's slice
  const int nseg = sl.nseg();
  double excl;
  int lo, hi;
  seg_total(sh, nseg, lane, excl, lo, hi);
  excl += slice_base;
  double part = 0.0;
  for (int c = lo; c < hi; ++c) part += static_cast<double>(sh.csum[c]);
  int seg = -1;
  double base = 0.0;
  const unsigned in = last ? 0u : __ballot_sync(0xffffffffu, part > 0.0 && excl <= t && t < excl + part);
  if (in) {
    const int l = __ffs(in) - 1;
    if (lane == l) {
      double acc = excl;
      for (int c = lo; c < hi; ++c) {
        const double nx = acc + static_cast<double>(sh.csum[c]);
        if (t < nx && sh.csum[c] > 0.f) {
          seg = c;
          base = acc;
          break;
        }
        acc = nx;
      }
    }
    seg = __shfl_sync(0xffffffffu, seg, l);
    base = __shfl_sync(0xffffffffu, base, l);
  }
  if (seg < 0) {
    // past the weights: the last segment with weight
    int lastc = -1;
    for (int c = lo; c < hi; ++c)
      if (sh.csum[c] > 0.f) lastc = c;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lastc = max(lastc, __shfl_xor_sync(0xffffffffu, lastc, o));
    seg = lastc;
    base = -1.0;
  }
  if (seg < 0) return -1;
  const int e0 = sl.seg_e0(seg);
  int y = -1, lastw = -1;
  double run = base;
  for (int j = 0; j < kTreeVecsPerLane && y < 0; ++j) {
    const int ev = e0 + (j * 32 + lane) * NV;
    float zt[NV], zd[NV], w[NV];
    VV::unpack(load_vec<ELT>(rt, ev, V, P.vec), zt);
    if (mode != 0) VV::unpack(load_vec<ELT>(rd, ev, V, P.vec), zd);
    float wl = 0.f;
#pragma unroll
    for (int e = 0; e < NV; ++e) {
      const bool mine = ev + e < e_end;   // logits past the slice are the next CTA's
      w[e] = !mine ? 0.f
                   : (mode == 0 ? bonus_weight(zt[e], P.c2, sh.Kt)
                                : pair_weight(zt[e], zd[e], P.c2, sh.Kt, sh.wA, sh.wGh, sh.wGl));
      wl += w[e];
      if (w[e] > 0.f) lastw = max(lastw, ev + e);
    }
    const double incl = warp_incl_scan(static_cast<double>(wl), lane);
    if (base >= 0.0) {
      const double start = run + (incl - static_cast<double>(wl));
      const unsigned hit = __ballot_sync(0xffffffffu, wl > 0.f && start <= t && t < run + incl);
      if (hit) {
        const int l = __ffs(hit) - 1;
        int pick = -1;
        if (lane == l) {
          double acc = start;
          int lastp = -1;
          for (int e = 0; e < NV; ++e) {
            if (w[e] > 0.f) lastp = ev + e;
            acc += static_cast<double>(w[e]);
            if (t < acc && w[e] > 0.f) {
              pick = ev + e;
              break;
            }
          }
          if (pick < 0) pick = lastp;
        }
        y = __shfl_sync(0xffffffffu, pick, l);
      }
    }
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (y < 0) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lastw = max(lastw, __shfl_xor_sync(0xffffffffu, lastw, o));
    y = lastw;
  }
  return y;
}

template <int ELT, bool GREEDY>
__global__ void __launch_bounds__(kTreeThreads, 2) tree_kernel(const TreeParams P) {
  __shared__ TreeShared sh;
  extern __shared__ __align__(128) unsigned char ring[];   // kTreeRingBytes
  using VV = Vec<ELT>;
  constexpr int NV = VV::N;
  const int cs = P.cs;
  const int rank = cluster_rank();
  const int b = blockIdx.x / cs;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int M = P.M, V = P.V;
  const int nch = (V + kChunkElems - 1) / kChunkElems;
  const int c_lo = static_cast<int>((static_cast<long long>(rank) * nch) / cs);
  const int c_hi = static_cast<int>((static_cast<long long>(rank + 1) * nch) / cs);
  const size_t row_bytes = static_cast<size_t>(V) * ELT;
  const float c2 = P.c2;
  const size_t rb = static_cast<size_t>(b) * M;
  const bool lead = rank == 0;        // the CTA that writes the outputs
  int xp = 0;
  Slice<ELT> sl(sh, ring, P, c_lo, c_hi);

  if (tid == 0) {
    for (int s = 0; s < kTreeStages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], kTreeWarps);
    }
    fence_mbar_init();
    sh.failed = 0;
    for (int s = 0; s < kTreeStages; ++s) sh.lastq[s] = -1;
  }
  // the next kernel on the stream may start (a next call's walk reads only
  // its inputs until it writes its outputs, after its dependency wait)
  grid_dependents_launch();
  for (int j = tid; j < M; j += kTreeThreads) {
    sh.par[j] = P.parents[rb + j];
    sh.tok[j] = P.tokens[rb + j];
    sh.u[j] = P.uniforms[rb + j];
    sh.otok[j] = -1;
    sh.onode[j] = -1;
    sh.oal[j] = NAN;
  }
  __syncthreads();
  if (tid == 0) {
    int st = 0;
    const int n = P.n_nodes[b];
    if (n < 1 || n > M) st = SV_ERR_BAD_DRAFT_LEN;
    for (int j = 1; st == 0 && j < n; ++j)
      if (sh.par[j] < 0 || sh.par[j] >= j) st = SV_ERR_BAD_DRAFT_LEN;
    for (int j = 1; st == 0 && j < n; ++j)
      if (sh.tok[j] < 0 || sh.tok[j] >= V) st = SV_ERR_BAD_TOKEN;
    sh.n = n;
    sh.st = st;
    sh.cur = 0;
    sh.len = 0;
    sh.y = -1;
  }
  __syncthreads();

  // sh.st: 0 walking, > 0 an error, -1 done.  Every decision below is taken
  // from values that are the same in every CTA of the cluster (the inputs,
  // or exchanged and combined in rank order), so the CTAs walk in lockstep
  // and meet at every cluster barrier.  The producer warp follows the walk
  // too, and streams during the passes.
  while (sh.st == 0) {
    const int cur = sh.cur;
    if (tid == 0) {
      int nk = 0;
      for (int c = cur + 1; c < sh.n; ++c)
        if (sh.par[c] == cur) sh.kids[nk++] = c;
      sh.nkids = nk;
    }
    __syncthreads();
    const int nk = sh.nkids;
    const unsigned char* rt = P.target + (rb + cur) * row_bytes;
    const unsigned char* rd = P.draft + (rb + cur) * row_bytes;

    if (GREEDY) {
      // first argmax of the target row; both rows checked
      float best = -INFINITY, dmax = -INFINITY;
      int bi = 0x7fffffff, bad = 0;
      sl.pass(rt, rd, nk > 0, [&](int k, const uint4 (&tv)[kTreeVecsPerLane], const uint4 (&dv)[kTreeVecsPerLane]) {
#pragma unroll
        for (int j = 0; j < kTreeVecsPerLane; ++j) {
          const int e0 = sl.e_lo + k * Slice<ELT>::kSlotElems + (warp * kTreeVecsPerWarp + j * 32 + lane) * NV;
          float z[NV];
          VV::unpack(tv[j], z);
#pragma unroll
          for (int e = 0; e < NV; ++e) {
            bad |= (z[e] != z[e]) || (z[e] == INFINITY);
            if (z[e] > best) {        // padding is -inf: only logits of the slice win
              best = z[e];
              bi = e0 + e;
            }
          }
          if (nk > 0) {
            VV::unpack(dv[j], z);
#pragma unroll
            for (int e = 0; e < NV; ++e) {
              bad |= (z[e] != z[e]) || (z[e] == INFINITY);
              dmax = fmaxf(dmax, z[e]);
            }
          }
        }
      });
      warp_argmax(best, bi);
      bad = warp_or(bad);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dmax = fmaxf(dmax, __shfl_xor_sync(0xffffffffu, dmax, o));
      if (lane == 0 && warp < kTreeWarps) {
        sh.wm[warp] = best;
        sh.widx[warp] = bi;
        sh.wbad[warp] = bad;
        sh.wmd[warp] = dmax;
      }
      __syncthreads();
      if (tid == 0) {
        float bv = -INFINITY, dm = -INFINITY;
        int bx = 0x7fffffff, anybad = 0;
        for (int w = 0; w < kTreeWarps; ++w) {
          anybad |= sh.wbad[w];
          dm = fmaxf(dm, sh.wmd[w]);
          if (sh.wm[w] > bv || (sh.wm[w] == bv && sh.widx[w] < bx)) {
            bv = sh.wm[w];
            bx = sh.widx[w];
          }
        }
        sh.xs[xp].Kt = bv;
        sh.xs[xp].idx = bx;
        sh.xs[xp].St = dm;
        sh.xs[xp].bad = anybad;
      }
      __syncthreads();
      exchange(sh, xp, cs);
      if (tid == 0) {
        float bv = -INFINITY, dm = -INFINITY;
        int bx = 0x7fffffff, anybad = 0;
        for (int r = 0; r < cs; ++r) {          // slices in index order: ties go to the lower rank
          const XSlot& x = sh.got[r];
          anybad |= x.bad;
          dm = fmaxf(dm, x.St);
          if (x.Kt > bv) {
            bv = x.Kt;
            bx = x.idx;
          }
        }
        if (sh.failed) {
          sh.st = SV_ERR_TIMEOUT;
        } else if (anybad || bv == -INFINITY || (nk > 0 && dm == -INFINITY)) {
          sh.st = SV_ERR_NONFINITE;
        } else {
          int next = -1;
          for (int i = 0; i < nk && next < 0; ++i) {
            const int c = sh.kids[i];
            const int ok = (sh.tok[c] == bx);
            sh.oal[c] = ok ? 1.f : 0.f;
            if (ok) next = c;
          }
          if (next >= 0) {
            sh.onode[sh.len] = next;
            sh.otok[sh.len] = sh.tok[next];
            sh.len += 1;
            sh.cur = next;
          } else {
            sh.y = bx;
            sh.st = -1;
          }
        }
      }
      __syncthreads();
      continue;
    }

    // --- row statistics: one pass over this CTA's slice of the target row
    // and, for a node with children, of the draft row; then the slices'
    // pairs are merged in rank order
    {
      float mt = -INFINITY, Kt = 0.f, md = -INFINITY, Kd = 0.f;
      f2 st2 = 0ull, sd2 = 0ull;
      int bad = 0;
      sl.pass(rt, rd, nk > 0, [&](int, const uint4 (&tv)[kTreeVecsPerLane], const uint4 (&dv)[kTreeVecsPerLane]) {
        online_vecs<ELT>(tv, c2, mt, Kt, st2, bad);
        if (nk > 0) online_vecs<ELT>(dv, c2, md, Kd, sd2, bad);
      });
      float x0, x1;
      unpack2(st2, x0, x1);
      const float st = x0 + x1;
      unpack2(sd2, x0, x1);
      const float sd = x0 + x1;
      bad = warp_or(bad);
      if (lane == 0 && warp < kTreeWarps) sh.wbad[warp] = bad;
      combine_stats(mt, Kt, st, sh.myKt, sh.mySt, sh.wm, sh.ws, c2);
      if (nk > 0) combine_stats(md, Kd, sd, sh.myKd, sh.mySd, sh.wmd, sh.wsd, c2);
      __syncthreads();
      if (tid == 0) {
        int anybad = 0;
        for (int w = 0; w < kTreeWarps; ++w) anybad |= sh.wbad[w];
        sh.xs[xp].Kt = sh.myKt;
        sh.xs[xp].St = sh.mySt;
        sh.xs[xp].Kd = nk > 0 ? sh.myKd : -INFINITY;
        sh.xs[xp].Sd = nk > 0 ? sh.mySd : 0.f;
        sh.xs[xp].bad = anybad;
      }
      __syncthreads();
      exchange(sh, xp, cs);
      if (tid == 0) {
        float K1 = -INFINITY, S1 = 0.f, K2 = -INFINITY, S2 = 0.f;
        int anybad = 0;
        for (int r = 0; r < cs; ++r) {
          const XSlot& x = sh.got[r];
          anybad |= x.bad;
          merge_ks(K1, S1, x.Kt, x.St);
          merge_ks(K2, S2, x.Kd, x.Sd);
        }
        sh.Kt = K1;
        sh.St = S1;
        sh.Kd = K2;
        sh.Sd = S2;
        if (sh.failed) sh.st = SV_ERR_TIMEOUT;
        else if (anybad || !(S1 > 0.f) || (nk > 0 && !(S2 > 0.f))) sh.st = SV_ERR_NONFINITE;
        // log2(S^t / S^d), once per node (every child's test and residual uses
        // it); in fp32, which loses nothing against the fp32 sums S
        sh.l2ratio = nk > 0 ? static_cast<double>(log2f(__fdiv_rn(S1, S2))) : 0.0;
        sh.cc = 0.0;
        sh.PP = 1.0;
        sh.invPP = 1.0;
      }
      __syncthreads();
      if (sh.st != 0) break;
    }

    // --- the children, in index order
    int accepted = -1, last_mode = 1;
    for (int i = 0; i < nk; ++i) {
      if (tid == 0) {
        const int c = sh.kids[i];
        const long long x = sh.tok[c];
        const float zt = VV::scalar(rt, x), zd = VV::scalar(rd, x);
        // r(x) / q(x) = max(0, p(x)/q(x) - c) / P, with p(x)/q(x) from its
        // logarithm in double: (z^t - z^d) c - (K^t - K^d) - log2(S^t / S^d)
        double rq;
        if (zd == -INFINITY) rq = zt == -INFINITY ? 0.0 : INFINITY;    // q(x) = 0: r > 0 iff p > 0
        else if (zt == -INFINITY) rq = 0.0;                            // p(x) = 0
        else {
          const double l2 = (static_cast<double>(zt) - static_cast<double>(zd)) * static_cast<double>(c2) -
                            (static_cast<double>(sh.Kt) - static_cast<double>(sh.Kd)) - sh.l2ratio;
          rq = fmax(exp2(l2) - sh.cc, 0.0) * sh.invPP;
        }
        const double al = fmin(1.0, rq);
        const bool acc = static_cast<double>(sh.u[c]) < al;
        sh.oal[c] = static_cast<float>(al);
        sh.next = acc ? c : -1;
      }
      __syncthreads();
      if (sh.next >= 0) {
        accepted = sh.next;
        break;
      }
      // rejected: the residual after this rejection, its mass and segment sums
      last_mode = 1;
      weight_pass<ELT>(sh, sl, P, rt, rd, 1, xp);
      if (!(sh.total > 0.0)) {
        last_mode = 2;                       // zero residual: keep r
        weight_pass<ELT>(sh, sl, P, rt, rd, 2, xp);
      }
      if (tid == 0) {
        // S = sh.total is the mass of max(0, r - q) (or of r); the new
        // residual is that weight over S
        if (last_mode == 1) sh.cc += sh.PP;
        sh.PP *= sh.total;
        sh.invPP = 1.0 / sh.PP;
      }
      __syncthreads();
    }
    if (accepted >= 0) {
      if (tid == 0) {
        sh.onode[sh.len] = accepted;
        sh.otok[sh.len] = sh.tok[accepted];
        sh.len += 1;
        sh.cur = accepted;
      }
      __syncthreads();
      continue;
    }

    // --- the draw: the bonus weights at a node without children, else the
    // last residual (whose segment sums the last pass left in sh.csum).  The
    // CTA whose slice holds s * S draws; the token is then exchanged.
    const int wmode = nk == 0 ? 0 : last_mode;
    if (nk == 0) weight_pass<ELT>(sh, sl, P, rt, rd, 0, xp);
    if (tid == 0) {
      const double t = static_cast<double>(sh.u[0]) * sh.total;
      int owner = -1, lastw = -1;
      for (int r = 0; r < cs; ++r) {
        if (sh.slice[r] > 0.0) {
          lastw = r;
          if (owner < 0 && sh.base[r] <= t && t < sh.base[r] + sh.slice[r]) owner = r;
        }
      }
      sh.owner = owner >= 0 ? owner : lastw;
      sh.next = owner >= 0 ? 0 : 1;     // 1: past every weight
    }
    __syncthreads();
    int y = -1;
    if (rank == sh.owner && warp == 0)
      y = draw<ELT>(sh, sl, P, rt, rd, wmode, static_cast<double>(sh.u[0]) * sh.total, sh.base[rank], sh.next == 1);
    if (tid == 0) sh.xs[xp].y = y;
    __syncthreads();
    exchange(sh, xp, cs);
    if (tid == 0) {
      sh.y = sh.owner >= 0 ? sh.got[sh.owner].y : -1;
      sh.st = sh.failed ? SV_ERR_TIMEOUT : -1;
    }
    __syncthreads();
  }

  if (tid == 0) {
    const int st = sh.st < 0 ? 0 : sh.st;
    if (st == 0) sh.otok[sh.len] = sh.y;
    sh.st = st;
  }
  __syncthreads();
  if (lead) {
    // the outputs, once the previous call on the stream has completed
    grid_dependency_wait();
    const int st = sh.st;
    for (int j = tid; j < M; j += kTreeThreads) {
      P.out_tokens[rb + j] = st > 0 ? -1 : sh.otok[j];
      P.out_nodes[rb + j] = st > 0 ? -1 : sh.onode[j];
      if (P.alpha) P.alpha[rb + j] = sh.oal[j];
    }
    if (tid == 0) {
      P.out_len[b] = st == 0 ? sh.len + 1 : 0;
      if (P.status) P.status[b] = st;
    }
  }
  if (warp == kTreeProducer) sl.drain();
  cluster_sync();                     // no CTA leaves while a peer may still read its slots
}

}  // namespace
}  // namespace sv

extern "C" sv_status spec_verify_tree(int B, int max_nodes, int V, sv_dtype dtype, const void* target_logits,
                                      const void* draft_logits, const int32_t* parents, const int32_t* tokens,
                                      const int32_t* n_nodes, const float* uniforms, float temperature,
                                      int32_t* out_tokens, int32_t* out_nodes, int32_t* out_len, int32_t* status,
                                      float* alpha, sv_stream_t stream) {
  if (B < 0 || max_nodes < 1 || max_nodes > sv::kTreeMaxNodes || V < 1 || V > sv::kTreeMaxV)
    return SV_ERR_INVALID_ARG;
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  if (!(temperature >= 0.f) || !std::isfinite(temperature)) return SV_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * max_nodes > (1LL << 30)) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!target_logits || !draft_logits || !parents || !tokens || !n_nodes || !uniforms || !out_tokens ||
      !out_nodes || !out_len)
    return SV_ERR_INVALID_ARG;
  const bool greedy = temperature == 0.f;
  const double c2 = greedy ? 0.0 : 1.4426950408889634 / static_cast<double>(temperature);
  if (!(c2 < 1e30)) return SV_ERR_INVALID_ARG;
  const int elt = dtype == SV_F32 ? 4 : 2;
  sv::TreeParams p{};
  p.target = static_cast<const unsigned char*>(target_logits);
  p.draft = static_cast<const unsigned char*>(draft_logits);
  p.parents = parents;
  p.tokens = tokens;
  p.n_nodes = n_nodes;
  p.uniforms = uniforms;
  p.out_tokens = out_tokens;
  p.out_nodes = out_nodes;
  p.out_len = out_len;
  p.status = status;
  p.alpha = alpha;
  p.B = B;
  p.M = max_nodes;
  p.V = V;
  p.vec = (static_cast<long long>(V) * elt) % 16 == 0 && (reinterpret_cast<uintptr_t>(target_logits) & 15u) == 0 &&
          (reinterpret_cast<uintptr_t>(draft_logits) & 15u) == 0;
  p.c2 = static_cast<float>(c2);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  void (*kern)(const sv::TreeParams) = elt == 2 ? (greedy ? sv::tree_kernel<2, true> : sv::tree_kernel<2, false>)
                                                : (greedy ? sv::tree_kernel<4, true> : sv::tree_kernel<4, false>);
  const int ring = sv::kTreeRingBytes;
  // Once per device and kernel: the slots need more than the default 48 KB
  // of dynamic shared memory, and the cluster sizes that can be resident
  // with it (clusters of 1, 2, 4, 8 CTAs) are recorded.
  struct DevInfo {
    bool ready[4];
    int sms;
    int fits[4][4];   // [kernel][log2 cluster]: clusters that fit at once
  };
  static DevInfo info[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SV_ERR_CUDA;
  const int which = (elt == 2 ? 0 : 2) + (greedy ? 1 : 0);
  DevInfo& di = info[dev];
  if (!di.ready[which]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, ring) != cudaSuccess)
      return SV_ERR_CUDA;
    if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return SV_ERR_CUDA;
    for (int l = 0; l < 4; ++l) {
      cudaLaunchConfig_t q{};
      cudaLaunchAttribute qa[1];
      qa[0].id = cudaLaunchAttributeClusterDimension;
      qa[0].val.clusterDim.x = 1u << l;
      qa[0].val.clusterDim.y = 1;
      qa[0].val.clusterDim.z = 1;
      q.gridDim = dim3(1u << l, 1, 1);
      q.blockDim = dim3(sv::kTreeThreads, 1, 1);
      q.dynamicSmemBytes = static_cast<size_t>(ring);
      q.attrs = qa;
      q.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(kern), &q) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
      }
      di.fits[which][l] = n;
    }
    di.ready[which] = true;
  }
  // CTAs per sequence: the largest cluster (up to 8) that keeps one CTA per
  // SM for the whole batch; a sequence's walk is serial, so idle SMs are
  // better spent on slices of its rows.  Two CTAs of this shape fit on an
  // SM, so the next call's walks share every SM with this call's
  int cs = 1;
  for (int l = 3; l >= 1; --l) {
    const int c = 1 << l;
    if (static_cast<long long>(B) * c <= di.sms && di.fits[which][l] > 0) {
      cs = c;
      break;
    }
  }
  if (di.fits[which][0] <= 0) return SV_ERR_UNSUPPORTED;
  p.cs = cs;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch: back-to-back calls overlap (each writes
  // its outputs after its dependency wait)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(B) * static_cast<unsigned>(cs), 1, 1);
  cfg.blockDim = dim3(sv::kTreeThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(ring);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  sv::NvtxRange range("spec_verify_tree");
  return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
