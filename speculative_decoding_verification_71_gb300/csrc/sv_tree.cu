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
// A cluster of cs CTAs walks one sequence: each CTA streams a contiguous
// slice of every row (through a cp.async ring in shared memory, see Chunks),
// and the slices' sums are exchanged through distributed shared memory and
// combined in rank order, so every CTA takes the same decisions.  cs is the
// largest of 8, 4, 2, 1 that keeps one CTA per SM for the whole batch.  Each
// visited node costs one pass over its
// target row (and draft row, if it has children) for the row maximum and
// log-sum of 2^(z c), one more pass over both rows per rejected child (the
// residual mass, with the sums of 256-logit chunks kept for the draw), and
// one pass for a bonus draw; the later passes find the rows in L2.  Only
// the rows the walk visits are read.  Every reduction runs in a fixed order,
// so the result is deterministic.

#include <cuda_runtime.h>

#include <cmath>
#include <cstddef>
#include <cstdint>

#include "../../include/specverify.h"
#include "sv_device.cuh"

namespace sv {
namespace {

constexpr int kTreeThreads = 512;
constexpr int kTreeWarps = kTreeThreads / 32;
constexpr int kChunkElems = 256;                 // logits per warp step: 8 per lane
constexpr int kTreeMaxChunks = 2048;             // V <= 524288
constexpr int kTreeMaxNodes = SV_TREE_MAX_NODES;
constexpr int kTreeMaxCluster = 8;

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
  int vec;                       // rows 16-byte aligned: vector loads
  float c2;                      // log2(e) / T
  int cs;                        // CTAs per sequence (the cluster): each streams a slice of every row
};

template <int ELT>
struct Rows {
  // Eight consecutive logits from element e0 (those past V read as -inf).
  __device__ __forceinline__ static void load8(const unsigned char* row, int e0, int V, int vec, float (&v)[8]) {
    if (vec && e0 + 8 <= V) {
      if (ELT == 2) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(row + static_cast<size_t>(e0) * 2));
        Vec<2>::unpack(w, v);
      } else {
        const uint4 w0 = __ldg(reinterpret_cast<const uint4*>(row + static_cast<size_t>(e0) * 4));
        const uint4 w1 = __ldg(reinterpret_cast<const uint4*>(row + static_cast<size_t>(e0) * 4 + 16));
        v[0] = __uint_as_float(w0.x); v[1] = __uint_as_float(w0.y);
        v[2] = __uint_as_float(w0.z); v[3] = __uint_as_float(w0.w);
        v[4] = __uint_as_float(w1.x); v[5] = __uint_as_float(w1.y);
        v[6] = __uint_as_float(w1.z); v[7] = __uint_as_float(w1.w);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        v[j] = (e0 + j < V) ? Vec<ELT>::scalar(row, e0 + j) : -INFINITY;
    }
  }
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_addr(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

// Calls f(c, e0, zt[8], zd[8]) for each chunk c in [c_lo, c_hi) of this
// warp (c = c_lo + warp, c_lo + warp + W, ...), zt / zd being the lane's eight logits of the target and
// (if `both`) draft rows from e0.  Each lane streams its own 16 (bf16) or 32
// (fp32) bytes per row and chunk through a ring of D slots in shared memory
// with cp.async, D chunks ahead of its use: every lane reads back only what
// it copied itself, so no barrier is needed, and a slot is refilled only
// after its logits were consumed.  Lanes past V or on rows that are not
// 16-byte aligned read their logits with plain loads instead.
template <int ELT>
struct Chunks {
  static constexpr int D = ELT == 2 ? 8 : 4;      // chunks in flight per warp
  static constexpr int LB = 8 * ELT;               // bytes per lane, row and chunk
  static constexpr int kRingBytes = kTreeWarps * D * 2 * 32 * LB;
  __device__ __forceinline__ static unsigned char* slot(unsigned char* ring, int warp, int s, int row, int lane) {
    return ring + ((((warp * D + s) * 2 + row) * 32 + lane) * LB);
  }
  template <typename F>
  __device__ __forceinline__ static void each(unsigned char* ring, const unsigned char* rt, const unsigned char* rd,
                                              bool both, int c_lo, int c_hi, int V, int vec, F&& f) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int mine = c_lo + warp < c_hi ? (c_hi - c_lo - warp + kTreeWarps - 1) / kTreeWarps : 0;
    auto issue = [&](int i) {
      const int c = c_lo + warp + i * kTreeWarps;
      const int e0 = c * kChunkElems + lane * 8;
      if (i < mine && vec && e0 + 8 <= V) {
        const int sl = i % D;
#pragma unroll
        for (int w = 0; w < LB / 16; ++w) {
          cp_async16(slot(ring, warp, sl, 0, lane) + 16 * w, rt + static_cast<size_t>(e0) * ELT + 16 * w);
          if (both) cp_async16(slot(ring, warp, sl, 1, lane) + 16 * w, rd + static_cast<size_t>(e0) * ELT + 16 * w);
        }
      }
      cp_async_commit();
    };
#pragma unroll
    for (int i = 0; i < D; ++i) issue(i);
    for (int i = 0; i < mine; ++i) {
      cp_async_wait<D - 1>();                      // chunk i has landed
      const int c = c_lo + warp + i * kTreeWarps;
      const int e0 = c * kChunkElems + lane * 8;
      float zt[8], zd[8];
      if (vec && e0 + 8 <= V) {
        const int sl = i % D;
        unpack(slot(ring, warp, sl, 0, lane), zt);
        if (both) unpack(slot(ring, warp, sl, 1, lane), zd);
      } else {
        Rows<ELT>::load8(rt, e0, V, 0, zt);
        if (both) Rows<ELT>::load8(rd, e0, V, 0, zd);
      }
      f(c, e0, zt, zd);
      issue(i + D);
    }
    cp_async_wait<0>();
  }
  __device__ __forceinline__ static void unpack(const unsigned char* p, float (&v)[8]) {
    if (ELT == 2) {
      Vec<2>::unpack(*reinterpret_cast<const uint4*>(p), v);
    } else {
      const uint4 a = reinterpret_cast<const uint4*>(p)[0], b = reinterpret_cast<const uint4*>(p)[1];
      v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y); v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
      v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y); v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
    }
  }
};

// What a CTA contributes to one exchange of its cluster (three 16-byte
// words, read by a peer with three vector loads).
struct __align__(16) XSlot {
  float Kt, St, Kd, Sd;     // row statistics of its slice (greedy: Kt = best logit, St = draft maximum)
  int bad, idx, y, pad;     // a bad logit seen; greedy argmax; the drawn token
  double total, pad2;       // its slice's weight
};

// Per-CTA scratch for the walk.
struct TreeShared {
  int par[kTreeMaxNodes], tok[kTreeMaxNodes];
  float u[kTreeMaxNodes];
  int kids[kTreeMaxNodes];
  int nkids, n, cur, len, st, next, y, owner;
  float csum[kTreeMaxChunks];        // chunk sums of the last weight pass (this CTA's chunks)
  double cc, PP, invPP;              // residual after the rejections so far: max(0, p - cc q) / PP
  double invSt, invSd;               // 1 / S^t, 1 / S^d of the current node
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
// only after reading it.
__device__ __forceinline__ void exchange(TreeShared& sh, int& xp, int cs) {
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
  xp ^= 1;
}

// Running (max, sum 2^(z c - fl(max c))) of one lane, updated by 8 logits.
__device__ __forceinline__ void online8(const float (&z)[8], float c2, float& m, float& K, float& s, int& bad) {
  float vm = -INFINITY;
#pragma unroll
  for (int j = 0; j < 8; ++j) vm = fmax_nan(vm, z[j]);     // NaN survives the maximum
  bad |= (vm != vm) || (vm == INFINITY);
  if (vm > m) {
    const float Kn = vm * c2;
    s = (m == -INFINITY) ? 0.f : s * fast_exp2(K - Kn);
    m = vm;
    K = Kn;
  }
  if (m != -INFINITY) {
#pragma unroll
    for (int j = 0; j < 8; ++j) s += fast_exp2(fmaf(z[j], c2, -K));
  }
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

// CTA-wide (K, S) of the lanes' running pairs, in warp order (thread 0).
__device__ void combine_stats(float m, float K, float s, float& Kout, float& Sout, float* wm, float* ws, float c2) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float M = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float KM = M * c2;
  float v = (m == -INFINITY) ? 0.f : s * fast_exp2(K - KM);
  v = warp_sum(v);
  if (lane == 0) {
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
// The bonus weight: no draft row (K^d may be -inf at a node without children).
__device__ __forceinline__ float bonus_weight(float zt, float c2, float Kt) { return fast_exp2(fmaf(zt, c2, -Kt)); }

// Fixed-order fp64 total of the chunk sums of [c_lo, c_hi): lane l adds a
// contiguous run of chunks in order, then the lanes are scanned.
__device__ __forceinline__ double chunk_total(const TreeShared& sh, int c_lo, int c_hi, int lane, double& excl,
                                             int& lo, int& hi) {
  const int n = c_hi - c_lo;
  const int per = (n + 31) / 32;
  lo = c_lo + min(lane * per, n);
  hi = min(lo + per, c_hi);
  double part = 0.0;
  for (int c = lo; c < hi; ++c) part += static_cast<double>(sh.csum[c]);
  const double incl = warp_incl_scan(part, lane);
  excl = incl - part;
  return __shfl_sync(0xffffffffu, incl, 31);
}

// One pass of weights over this CTA's slice of the current node's rows:
// chunk sums into sh.csum, then the slices' weights exchanged in the
// cluster (sh.slice, sh.base, sh.total, identical in every CTA).
//   mode 0: bonus weights (A = 1, B = 0; the draft row is not read);
//   mode 1: the residual after one more rejection;
//   mode 2: the current residual r itself (zero-residual fallback).
template <int ELT>
__device__ void weight_pass(TreeShared& sh, unsigned char* ring, const TreeParams& P, const unsigned char* rt,
                            const unsigned char* rd, int mode, int c_lo, int c_hi, int& xp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    sh.wA = mode == 0 ? 1.f : static_cast<float>(sh.invPP * sh.invSt);
    sh.wGh = -INFINITY;
    sh.wGl = 0.f;
    const double BA = (mode == 1 ? sh.cc + sh.PP : sh.cc) * (static_cast<double>(sh.St) / static_cast<double>(sh.Sd));
    if (mode != 0 && BA > 0.0) {
      const double G = log2(BA) + (static_cast<double>(sh.Kt) - static_cast<double>(sh.Kd));
      sh.wGh = static_cast<float>(G);
      sh.wGl = static_cast<float>(G - static_cast<double>(sh.wGh));
    }
  }
  __syncthreads();
  const float c2 = P.c2, Kt = sh.Kt, A = sh.wA, Gh = sh.wGh, Gl = sh.wGl;
  Chunks<ELT>::each(ring, rt, rd, mode != 0, c_lo, c_hi, P.V, P.vec,
                    [&](int c, int, const float (&zt)[8], const float (&zd)[8]) {
    float part = 0.f;
    if (mode == 0) {
#pragma unroll
      for (int j = 0; j < 8; ++j) part += bonus_weight(zt[j], c2, Kt);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) part += pair_weight(zt[j], zd[j], c2, Kt, A, Gh, Gl);
    }
    part = warp_sum(part);
    if (lane == 0) sh.csum[c] = part;
  });
  __syncthreads();
  if (warp == 0) {
    double excl;
    int lo, hi;
    const double tot = chunk_total(sh, c_lo, c_hi, lane, excl, lo, hi);
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
// for the CTA whose slice holds the point (warp 0): the chunk from the chunk
// sums, then the logit from the chunk's recomputed weights.  `last`: the
// point lies past every weight (rounding); take the last logit with weight.
template <int ELT>
__device__ int draw(TreeShared& sh, const TreeParams& P, const unsigned char* rt, const unsigned char* rd, int mode,
                    int c_lo, int c_hi, double t, double slice_base, bool last) {
  const int lane = threadIdx.x & 31;
  const int V = P.V;
  double excl;
  int lo, hi;
  chunk_total(sh, c_lo, c_hi, lane, excl, lo, hi);
  excl += slice_base;
  double part = 0.0;
  for (int c = lo; c < hi; ++c) part += static_cast<double>(sh.csum[c]);
  int chunk = -1;
  double base = 0.0;
  const unsigned in = last ? 0u : __ballot_sync(0xffffffffu, part > 0.0 && excl <= t && t < excl + part);
  if (in) {
    const int l = __ffs(in) - 1;
    if (lane == l) {
      double acc = excl;
      for (int c = lo; c < hi; ++c) {
        const double nx = acc + static_cast<double>(sh.csum[c]);
        if (t < nx && sh.csum[c] > 0.f) {
          chunk = c;
          base = acc;
          break;
        }
        acc = nx;
      }
    }
    chunk = __shfl_sync(0xffffffffu, chunk, l);
    base = __shfl_sync(0xffffffffu, base, l);
  }
  if (chunk < 0) {
    // past the weights: the last chunk with weight
    int lastc = -1;
    for (int c = lo; c < hi; ++c)
      if (sh.csum[c] > 0.f) lastc = c;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lastc = max(lastc, __shfl_xor_sync(0xffffffffu, lastc, o));
    chunk = lastc;
    base = -1.0;
  }
  if (chunk < 0) return -1;
  const int e0 = chunk * kChunkElems + lane * 8;
  float zt[8], zd[8], w[8];
  Rows<ELT>::load8(rt, e0, V, P.vec, zt);
  if (mode != 0) Rows<ELT>::load8(rd, e0, V, P.vec, zd);
  float wpart = 0.f;
  int lastw = -1;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    w[j] = mode == 0 ? bonus_weight(zt[j], P.c2, sh.Kt)
                     : pair_weight(zt[j], zd[j], P.c2, sh.Kt, sh.wA, sh.wGh, sh.wGl);
    wpart += w[j];
    if (w[j] > 0.f) lastw = e0 + j;
  }
  int y = -1;
  if (base >= 0.0) {
    const double incl = warp_incl_scan(static_cast<double>(wpart), lane);
    const double start = base + (incl - static_cast<double>(wpart));
    const unsigned hit = __ballot_sync(0xffffffffu, wpart > 0.f && start <= t && t < base + incl);
    if (hit) {
      const int l = __ffs(hit) - 1;
      if (lane == l) {
        double acc = start;
        for (int j = 0; j < 8; ++j) {
          acc += static_cast<double>(w[j]);
          if (t < acc && w[j] > 0.f) {
            y = e0 + j;
            break;
          }
        }
        if (y < 0) y = lastw;
      }
      y = __shfl_sync(0xffffffffu, y, l);
    }
  }
  if (y < 0) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lastw = max(lastw, __shfl_xor_sync(0xffffffffu, lastw, o));
    y = lastw;
  }
  return y;
}

template <int ELT, bool GREEDY>
__global__ void __launch_bounds__(kTreeThreads, 1) tree_kernel(const TreeParams P) {
  __shared__ TreeShared sh;
  extern __shared__ __align__(16) unsigned char ring[];   // Chunks<ELT>::kRingBytes
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

  for (int j = tid; j < M; j += kTreeThreads) {
    sh.par[j] = P.parents[rb + j];
    sh.tok[j] = P.tokens[rb + j];
    sh.u[j] = P.uniforms[rb + j];
    if (lead) {
      P.out_tokens[rb + j] = -1;
      P.out_nodes[rb + j] = -1;
      if (P.alpha) P.alpha[rb + j] = NAN;
    }
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
  // and meet at every cluster barrier.
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
      Chunks<ELT>::each(ring, rt, rd, nk > 0, c_lo, c_hi, V, P.vec,
                        [&](int, int e0, const float (&z)[8], const float (&zd)[8]) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          bad |= (z[j] != z[j]) || (z[j] == INFINITY);
          if (e0 + j < V && z[j] > best) {
            best = z[j];
            bi = e0 + j;
          }
        }
        if (nk > 0) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            bad |= (zd[j] != zd[j]) || (zd[j] == INFINITY);
            dmax = fmaxf(dmax, zd[j]);
          }
        }
      });
      warp_argmax(best, bi);
      bad = warp_or(bad);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dmax = fmaxf(dmax, __shfl_xor_sync(0xffffffffu, dmax, o));
      if (lane == 0) {
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
        if (anybad || bv == -INFINITY || (nk > 0 && dm == -INFINITY)) {
          sh.st = SV_ERR_NONFINITE;
        } else {
          int next = -1;
          for (int i = 0; i < nk && next < 0; ++i) {
            const int c = sh.kids[i];
            const int ok = (sh.tok[c] == bx);
            if (P.alpha && lead) P.alpha[rb + c] = ok ? 1.f : 0.f;
            if (ok) next = c;
          }
          if (next >= 0) {
            if (lead) {
              P.out_nodes[rb + sh.len] = next;
              P.out_tokens[rb + sh.len] = sh.tok[next];
            }
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
      float mt = -INFINITY, Kt = 0.f, st = 0.f, md = -INFINITY, Kd = 0.f, sd = 0.f;
      int bad = 0;
      Chunks<ELT>::each(ring, rt, rd, nk > 0, c_lo, c_hi, V, P.vec,
                        [&](int, int, const float (&z)[8], const float (&zd)[8]) {
        online8(z, c2, mt, Kt, st, bad);
        if (nk > 0) online8(zd, c2, md, Kd, sd, bad);
      });
      bad = warp_or(bad);
      if (lane == 0) sh.wbad[warp] = bad;
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
        if (anybad || !(S1 > 0.f) || (nk > 0 && !(S2 > 0.f))) sh.st = SV_ERR_NONFINITE;
        sh.invSt = 1.0 / static_cast<double>(S1);
        sh.invSd = nk > 0 ? 1.0 / static_cast<double>(S2) : 0.0;
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
        const float zt = Vec<ELT>::scalar(rt, x), zd = Vec<ELT>::scalar(rd, x);
        // r(x) / q(x) = max(0, p(x)/q(x) - c) / P, with p(x)/q(x) from its
        // logarithm in double: (z^t - z^d) c - (K^t - K^d) - log2(S^t / S^d)
        double rq;
        if (zd == -INFINITY) rq = zt == -INFINITY ? 0.0 : INFINITY;    // q(x) = 0: r > 0 iff p > 0
        else if (zt == -INFINITY) rq = 0.0;                            // p(x) = 0
        else {
          const double l2 = (static_cast<double>(zt) - static_cast<double>(zd)) * static_cast<double>(c2) -
                            (static_cast<double>(sh.Kt) - static_cast<double>(sh.Kd)) -
                            log2(static_cast<double>(sh.St) / static_cast<double>(sh.Sd));
          rq = fmax(exp2(l2) - sh.cc, 0.0) * sh.invPP;
        }
        const double al = fmin(1.0, rq);
        const bool acc = static_cast<double>(sh.u[c]) < al;
        if (P.alpha && lead) P.alpha[rb + c] = static_cast<float>(al);
        sh.next = acc ? c : -1;
      }
      __syncthreads();
      if (sh.next >= 0) {
        accepted = sh.next;
        break;
      }
      // rejected: the residual after this rejection, its mass and chunk sums
      last_mode = 1;
      weight_pass<ELT>(sh, ring, P, rt, rd, 1, c_lo, c_hi, xp);
      if (!(sh.total > 0.0)) {
        last_mode = 2;                       // zero residual: keep r
        weight_pass<ELT>(sh, ring, P, rt, rd, 2, c_lo, c_hi, xp);
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
        if (lead) {
          P.out_nodes[rb + sh.len] = accepted;
          P.out_tokens[rb + sh.len] = sh.tok[accepted];
        }
        sh.len += 1;
        sh.cur = accepted;
      }
      __syncthreads();
      continue;
    }

    // --- the draw: the bonus weights at a node without children, else the
    // last residual (whose chunk sums the last pass left in sh.csum).  The
    // CTA whose slice holds s * S draws; the token is then exchanged.
    const int wmode = nk == 0 ? 0 : last_mode;
    if (nk == 0) weight_pass<ELT>(sh, ring, P, rt, rd, 0, c_lo, c_hi, xp);
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
      y = draw<ELT>(sh, P, rt, rd, wmode, c_lo, c_hi, static_cast<double>(sh.u[0]) * sh.total, sh.base[rank],
                    sh.next == 1);
    if (tid == 0) sh.xs[xp].y = y;
    __syncthreads();
    exchange(sh, xp, cs);
    if (tid == 0) {
      sh.y = sh.owner >= 0 ? sh.got[sh.owner].y : -1;
      sh.st = -1;
    }
    __syncthreads();
  }

  if (tid == 0 && lead) {
    const int st = sh.st < 0 ? 0 : sh.st;
    if (st == 0) {
      P.out_tokens[rb + sh.len] = sh.y;
      P.out_len[b] = sh.len + 1;
    } else {
      P.out_len[b] = 0;
    }
    if (P.status) P.status[b] = st;
  }
  __syncthreads();
  if (sh.st > 0 && lead) {
    for (int j = tid; j < M; j += kTreeThreads) {
      P.out_tokens[rb + j] = -1;
      P.out_nodes[rb + j] = -1;
    }
  }
  cluster_sync();                     // no CTA leaves while a peer may still read its slots
}

}  // namespace
}  // namespace sv

extern "C" sv_status spec_verify_tree(int B, int max_nodes, int V, sv_dtype dtype, const void* target_logits,
                                      const void* draft_logits, const int32_t* parents, const int32_t* tokens,
                                      const int32_t* n_nodes, const float* uniforms, float temperature,
                                      int32_t* out_tokens, int32_t* out_nodes, int32_t* out_len, int32_t* status,
                                      float* alpha, sv_stream_t stream) {
  if (B < 0 || max_nodes < 1 || max_nodes > sv::kTreeMaxNodes || V < 1 || V > sv::kTreeMaxChunks * sv::kChunkElems)
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
  const int ring = elt == 2 ? sv::Chunks<2>::kRingBytes : sv::Chunks<4>::kRingBytes;
  // Once per device and kernel: the ring needs more than the default 48 KB
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
  // better spent on slices of its rows
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
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(B) * static_cast<unsigned>(cs), 1, 1);
  cfg.blockDim = dim3(sv::kTreeThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(ring);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  sv::NvtxRange range("spec_verify_tree");
  return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
