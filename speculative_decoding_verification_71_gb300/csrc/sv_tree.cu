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
// One CTA walks one sequence.  Each visited node costs one pass over its
// target row (and draft row, if it has children) for the row maximum and
// log-sum of 2^(z c), one more pass over both rows per rejected child (the
// residual mass, with the sums of 256-logit chunks kept for the draw), and
// one pass for a bonus draw; the later passes find the rows in L2.  Only
// the rows the walk visits are read.  Every reduction runs in a fixed order,
// so the result is deterministic.

#include <cuda_runtime.h>

#include <cmath>
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

// Per-CTA scratch for the walk.
struct TreeShared {
  int par[kTreeMaxNodes], tok[kTreeMaxNodes];
  float u[kTreeMaxNodes];
  int kids[kTreeMaxNodes];
  int nkids, n, cur, len, st, next, y;
  float csum[kTreeMaxChunks];        // chunk sums of the last weight pass
  double S[kTreeMaxNodes + 1];       // S[i]: mass after the i-th rejection at this node
  float invS[kTreeMaxNodes + 1];
  int fb[kTreeMaxNodes + 1];         // 1: that rejection kept r (zero residual)
  float wm[kTreeWarps], ws[kTreeWarps], wmd[kTreeWarps], wsd[kTreeWarps];
  int wbad[kTreeWarps], widx[kTreeWarps];
  float Kt, St, Kd, Sd;              // row statistics of the current node
  float invSt, invSd;
  double total;                      // mass of the last weight pass
};

// Running (max, sum 2^(z c - fl(max c))) of one lane, updated by 8 logits.
__device__ __forceinline__ void online8(const float (&z)[8], float c2, float& m, float& K, float& s, int& bad) {
  float vm = -INFINITY;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    bad |= (z[j] != z[j]) || (z[j] == INFINITY);
    vm = fmaxf(vm, z[j]);
  }
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

// CTA-wide combination of the lanes' (m, K, s): returns through the shared
// struct (Kout = fl(M c), Sout = sum 2^(z c - Kout)), in warp order.
__device__ void combine_stats(TreeShared& sh, float m, float K, float s, float& Kout, float& Sout, float* wm,
                              float* ws, float c2) {
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
    Kout = Kall;
    Sout = (Mall == -INFINITY) ? 0.f : S;
  }
}

// The weight of one logit pair in the current weight pass.
//   mode 0: bonus weight 2^(z^t c - K^t) (unnormalised p);
//   mode 1: max(0, r_i - q) after i = nrej rejections (fb: r kept);
//   mode 2: r_i itself (the zero-residual fallback).
__device__ __forceinline__ float weight_of(const TreeShared& sh, int mode, int nrej, float zt, float zd, float c2) {
  const float pe = fast_exp2(fmaf(zt, c2, -sh.Kt));
  if (mode == 0) return pe;
  const float p = pe * sh.invSt;
  const float q = fast_exp2(fmaf(zd, c2, -sh.Kd)) * sh.invSd;
  float r = p;
  for (int h = 1; h <= nrej; ++h) r = (sh.fb[h] ? r : fmaxf(r - q, 0.f)) * sh.invS[h];
  return mode == 2 ? r : fmaxf(r - q, 0.f);
}

// Fixed-order fp64 total of the chunk sums: lane l adds chunks
// [l*per, (l+1)*per) in order, then the lanes are scanned.
__device__ __forceinline__ double chunk_total(const TreeShared& sh, int nch, int lane, double& excl, int& lo, int& hi) {
  const int per = (nch + 31) / 32;
  lo = min(lane * per, nch);
  hi = min(lo + per, nch);
  double part = 0.0;
  for (int c = lo; c < hi; ++c) part += static_cast<double>(sh.csum[c]);
  const double incl = warp_incl_scan(part, lane);
  excl = incl - part;
  return __shfl_sync(0xffffffffu, incl, 31);
}

// One pass of weights over the current node's rows: chunk sums into
// sh.csum, the fixed-order fp64 total into sh.total.
template <int ELT>
__device__ void weight_pass(TreeShared& sh, const TreeParams& P, const unsigned char* rt, const unsigned char* rd,
                            int mode, int nrej, int nch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int V = P.V;
  for (int c = warp; c < nch; c += kTreeWarps) {
    const int e0 = c * kChunkElems + lane * 8;
    float zt[8], zd[8];
    Rows<ELT>::load8(rt, e0, V, P.vec, zt);
    if (mode != 0) Rows<ELT>::load8(rd, e0, V, P.vec, zd);
    float part = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (e0 + j < V) part += weight_of(sh, mode, nrej, zt[j], mode != 0 ? zd[j] : 0.f, P.c2);
    part = warp_sum(part);
    if (lane == 0) sh.csum[c] = part;
  }
  __syncthreads();
  if (warp == 0) {
    double excl;
    int lo, hi;
    const double tot = chunk_total(sh, nch, lane, excl, lo, hi);
    if (lane == 0) sh.total = tot;
  }
  __syncthreads();
}

// Inverse CDF over the weights of the last pass with the sampling uniform
// (warp 0): the chunk from the chunk sums, then the logit from the chunk's
// recomputed weights.  Rounding that leaves the point past the weights of
// the chunk (or of the row) takes the last logit with weight there.
template <int ELT>
__device__ int draw(TreeShared& sh, const TreeParams& P, const unsigned char* rt, const unsigned char* rd, int mode,
                    int nrej, int nch) {
  const int lane = threadIdx.x & 31;
  const int V = P.V;
  double excl;
  int lo, hi;
  const double tot = chunk_total(sh, nch, lane, excl, lo, hi);
  double part = 0.0;
  for (int c = lo; c < hi; ++c) part += static_cast<double>(sh.csum[c]);
  const double t = static_cast<double>(sh.u[0]) * tot;
  int chunk = -1;
  double base = 0.0;
  const unsigned in = __ballot_sync(0xffffffffu, part > 0.0 && excl <= t && t < excl + part);
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
    // past the total: the last chunk with weight
    int last = -1;
    for (int c = lo; c < hi; ++c)
      if (sh.csum[c] > 0.f) last = c;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
    chunk = last;
    base = -1.0;   // take the chunk's last logit with weight
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
    w[j] = (e0 + j < V) ? weight_of(sh, mode, nrej, zt[j], mode != 0 ? zd[j] : 0.f, P.c2) : 0.f;
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
__global__ void __launch_bounds__(kTreeThreads, 2) tree_kernel(const TreeParams P) {
  __shared__ TreeShared sh;
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int M = P.M, V = P.V;
  const int nch = (V + kChunkElems - 1) / kChunkElems;
  const size_t row_bytes = static_cast<size_t>(V) * ELT;
  const float c2 = P.c2;
  const size_t rb = static_cast<size_t>(b) * M;

  for (int j = tid; j < M; j += kTreeThreads) {
    sh.par[j] = P.parents[rb + j];
    sh.tok[j] = P.tokens[rb + j];
    sh.u[j] = P.uniforms[rb + j];
    P.out_tokens[rb + j] = -1;
    P.out_nodes[rb + j] = -1;
    if (P.alpha) P.alpha[rb + j] = NAN;
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

  // sh.st: 0 walking, > 0 an error, -1 done
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
      for (int c = warp; c < nch; c += kTreeWarps) {
        const int e0 = c * kChunkElems + lane * 8;
        float z[8];
        Rows<ELT>::load8(rt, e0, V, P.vec, z);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          bad |= (z[j] != z[j]) || (z[j] == INFINITY);
          if (e0 + j < V && z[j] > best) {
            best = z[j];
            bi = e0 + j;
          }
        }
        if (nk > 0) {
          Rows<ELT>::load8(rd, e0, V, P.vec, z);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            bad |= (z[j] != z[j]) || (z[j] == INFINITY);
            dmax = fmaxf(dmax, z[j]);
          }
        }
      }
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
        if (anybad || bv == -INFINITY || (nk > 0 && dm == -INFINITY)) {
          sh.st = SV_ERR_NONFINITE;
        } else {
          int next = -1;
          for (int i = 0; i < nk && next < 0; ++i) {
            const int c = sh.kids[i];
            const int ok = (sh.tok[c] == bx);
            if (P.alpha) P.alpha[rb + c] = ok ? 1.f : 0.f;
            if (ok) next = c;
          }
          if (next >= 0) {
            P.out_nodes[rb + sh.len] = next;
            P.out_tokens[rb + sh.len] = sh.tok[next];
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

    // --- row statistics: one pass over the target row and, for a node with
    // children, its draft row
    {
      float mt = -INFINITY, Kt = 0.f, st = 0.f, md = -INFINITY, Kd = 0.f, sd = 0.f;
      int bad = 0;
      for (int c = warp; c < nch; c += kTreeWarps) {
        const int e0 = c * kChunkElems + lane * 8;
        float z[8];
        Rows<ELT>::load8(rt, e0, V, P.vec, z);
        online8(z, c2, mt, Kt, st, bad);
        if (nk > 0) {
          Rows<ELT>::load8(rd, e0, V, P.vec, z);
          online8(z, c2, md, Kd, sd, bad);
        }
      }
      bad = warp_or(bad);
      if (lane == 0) sh.wbad[warp] = bad;
      combine_stats(sh, mt, Kt, st, sh.Kt, sh.St, sh.wm, sh.ws, c2);
      if (nk > 0) combine_stats(sh, md, Kd, sd, sh.Kd, sh.Sd, sh.wmd, sh.wsd, c2);
      __syncthreads();
      if (tid == 0) {
        int anybad = 0;
        for (int w = 0; w < kTreeWarps; ++w) anybad |= sh.wbad[w];
        if (anybad || !(sh.St > 0.f) || (nk > 0 && !(sh.Sd > 0.f))) sh.st = SV_ERR_NONFINITE;
        sh.invSt = 1.f / sh.St;
        sh.invSd = nk > 0 ? 1.f / sh.Sd : 0.f;
      }
      __syncthreads();
      if (sh.st != 0) break;
    }

    // --- the children, in index order
    int nrej = 0, accepted = -1, last_mode = 1;
    for (int i = 0; i < nk; ++i) {
      if (tid == 0) {
        const int c = sh.kids[i];
        const long long x = sh.tok[c];
        const float zt = Vec<ELT>::scalar(rt, x), zd = Vec<ELT>::scalar(rd, x);
        const double p = static_cast<double>(fast_exp2(fmaf(zt, c2, -sh.Kt))) / static_cast<double>(sh.St);
        const double q = static_cast<double>(fast_exp2(fmaf(zd, c2, -sh.Kd))) / static_cast<double>(sh.Sd);
        double r = p;
        for (int h = 1; h <= nrej; ++h) r = (sh.fb[h] ? r : fmax(r - q, 0.0)) / sh.S[h];
        const double al = (q == 0.0) ? (r > 0.0 ? 1.0 : 0.0) : fmin(1.0, r / q);
        if (P.alpha) P.alpha[rb + c] = static_cast<float>(al);
        sh.next = (static_cast<double>(sh.u[c]) < al) ? c : -1;
      }
      __syncthreads();
      if (sh.next >= 0) {
        accepted = sh.next;
        break;
      }
      // rejected: the residual after this rejection, its mass and chunk sums
      last_mode = 1;
      weight_pass<ELT>(sh, P, rt, rd, 1, nrej, nch);
      if (!(sh.total > 0.0)) {
        last_mode = 2;                       // zero residual: keep r
        weight_pass<ELT>(sh, P, rt, rd, 2, nrej, nch);
      }
      if (tid == 0) {
        sh.S[nrej + 1] = sh.total;
        sh.invS[nrej + 1] = static_cast<float>(1.0 / sh.total);
        sh.fb[nrej + 1] = (last_mode == 2);
      }
      __syncthreads();
      nrej += 1;
    }
    if (accepted >= 0) {
      if (tid == 0) {
        P.out_nodes[rb + sh.len] = accepted;
        P.out_tokens[rb + sh.len] = sh.tok[accepted];
        sh.len += 1;
        sh.cur = accepted;
      }
      __syncthreads();
      continue;
    }

    // --- the draw: the bonus weights at a node without children, else the
    // last residual (whose chunk sums the last pass left in sh.csum)
    const int wmode = nk == 0 ? 0 : last_mode;
    const int wrej = nk == 0 ? 0 : nrej - 1;
    if (nk == 0) weight_pass<ELT>(sh, P, rt, rd, 0, 0, nch);
    if (warp == 0) {
      const int y = draw<ELT>(sh, P, rt, rd, wmode, wrej, nch);
      if (lane == 0) {
        sh.y = y;
        sh.st = -1;
      }
    }
    __syncthreads();
  }

  if (tid == 0) {
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
  if (sh.st > 0) {
    for (int j = tid; j < M; j += kTreeThreads) {
      P.out_tokens[rb + j] = -1;
      P.out_nodes[rb + j] = -1;
    }
  }
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
  const dim3 grid(static_cast<unsigned>(B)), block(sv::kTreeThreads);
  if (elt == 2) {
    if (greedy) sv::tree_kernel<2, true><<<grid, block, 0, s>>>(p);
    else sv::tree_kernel<2, false><<<grid, block, 0, s>>>(p);
  } else {
    if (greedy) sv::tree_kernel<4, true><<<grid, block, 0, s>>>(p);
    else sv::tree_kernel<4, false><<<grid, block, 0, s>>>(p);
  }
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
