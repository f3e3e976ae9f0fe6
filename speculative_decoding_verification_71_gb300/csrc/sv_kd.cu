// Reward-weighted distillation loss of the draft model and its gradient in
// the draft logits, for sm_103a.
//
// "ReSpec: Towards Optimizing Speculative Decoding in Reinforcement Learning
// Systems", Online Learner (reward-weighted KD), trains the drafter on the
// rollouts with a KL divergence to the updated target, weighted per rollout
// by a function of its reward:
//   L_b = w_b * sum_t KL(p_{b,t} || q_{b,t}),  p = softmax(z^t/T), q = softmax(z^d/T)
//   dL_b / dz^d_{b,t}(x) = w_b (q(x) - p(x)) / T.
// The map from reward to weight is the caller's: w_b is an input.
//
// Per row pair, with c = log2(e)/T, K = fl(M c) for the row maximum M,
// S = sum_x 2^(z(x) c - K) and A = sum_x 2^(z^t(x) c - K^t) (z^t(x) - z^d(x)):
//   KL = ln 2 * (c A / S^t - (K^t - K^d) - log2(S^t / S^d)),
// since log2 p(x) = z^t(x) c - K^t - log2 S^t (and likewise for q).
// Rows are independent, so a cluster of cs CTAs takes one row pair at a
// time: each CTA stages its vocabulary slice of both rows in shared memory
// (cp.async.bulk), computes its part of (M, S, A), sends it to every CTA of
// the cluster (st.async, counted on their mbarriers), combines the parts in
// rank order and, from the same shared-memory copy, writes its slice of the
// gradient.  Each logit crosses HBM once and each gradient value once.  The
// next row's first pass runs while the current row's parts are exchanged.

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/specverify.h"
#include "sv_internal.h"
#include "sv_device.cuh"

namespace sv {
namespace {

constexpr int kKdWarps = 16;                         // compute warps
constexpr int kKdThreads = (kKdWarps + 1) * 32;      // + one producer warp
constexpr int kKdXRing = 4;                          // exchange slots (rows in flight: see below)
constexpr int kKdMaxBuf = 6;                         // row buffers per CTA
constexpr int kKdMaxCluster = 16;                    // 16 is a non-portable cluster size (opted into)
constexpr int kKdBarCompute = 1;                     // named barrier of the compute warps

struct alignas(16) KdPart {
  float mt, st, a, md;         // target max, target sum, weighted difference, draft max
  float sd, pad0, pad1, pad2;  // draft sum
};
static_assert(sizeof(KdPart) == 32, "a part travels as two 16-byte stores");

struct KdCtrl {
  uint64_t full[kKdMaxBuf];    // both slices of a row staged (producer -> compute warps)
  uint64_t empty[kKdMaxBuf];   // buffer released (one arrival per compute warp)
  uint64_t xbar[kKdXRing];     // every CTA's part of a row has arrived
  KdPart xpart[kKdXRing][kKdMaxCluster];
  KdPart wpart[kKdWarps];      // per-warp parts of the current row
};
constexpr int kKdCtrlBytes = ((static_cast<int>(sizeof(KdCtrl)) + 1023) / 1024) * 1024;

struct KdParams {
  const void* target;          // [rows, V]
  const void* draft;           // [rows, V]
  const float* weights;        // [rows / t_len]
  float* row_kl;               // [rows]
  void* grad;                  // [rows, V] (GRAD only)
  int rows, t_len, V;
  float c2;                    // log2(e) / T
  float inv_T;
  int slice_elems;             // logits per CTA slice (multiple of 64)
  int slot_bytes;              // bytes of one staged row slice (multiple of 128)
  int nbuf;                    // row buffers (1 .. kKdMaxBuf)
  int bulk;                    // rows 16-byte aligned: cp.async.bulk; else plain loads
};

// A part's numbers rescaled onto the common maxima of the parts in `lane`s
// 0..n-1 (warp-wide; every lane returns the combined part).
__device__ __forceinline__ KdPart combine_parts(const KdPart& mine, bool in, int n_lanes_pow2, float c2) {
  const float mt = from_ordered_key(__reduce_max_sync(0xffffffffu, ordered_key(in ? mine.mt : -INFINITY)));
  const float md = from_ordered_key(__reduce_max_sync(0xffffffffu, ordered_key(in ? mine.md : -INFINITY)));
  const float kt = mt > -INFINITY ? __fmul_rn(mt, c2) : -INFINITY;
  const float kd = md > -INFINITY ? __fmul_rn(md, c2) : -INFINITY;
  const float kt_l = (in && mine.mt > -INFINITY) ? __fmul_rn(mine.mt, c2) : -INFINITY;
  const float kd_l = (in && mine.md > -INFINITY) ? __fmul_rn(mine.md, c2) : -INFINITY;
  const float ft = kt_l > -INFINITY ? fast_exp2(__fsub_rn(kt_l, kt)) : 0.f;
  const float fd = kd_l > -INFINITY ? fast_exp2(__fsub_rn(kd_l, kd)) : 0.f;
  float st = in && kt_l > -INFINITY ? mine.st * ft : 0.f;
  float a = in && kt_l > -INFINITY ? mine.a * ft : 0.f;
  float sd = in && kd_l > -INFINITY ? mine.sd * fd : 0.f;
  for (int o = n_lanes_pow2 >> 1; o > 0; o >>= 1) {
    st += __shfl_xor_sync(0xffffffffu, st, o);
    a += __shfl_xor_sync(0xffffffffu, a, o);
    sd += __shfl_xor_sync(0xffffffffu, sd, o);
  }
  KdPart r;
  r.mt = mt; r.md = md;
  r.st = __shfl_sync(0xffffffffu, st, 0);
  r.a = __shfl_sync(0xffffffffu, a, 0);
  r.sd = __shfl_sync(0xffffffffu, sd, 0);
  r.pad0 = r.pad1 = r.pad2 = 0.f;
  return r;
}

template <int ELT, bool GRAD>
struct KdRow {
  using V = Vec<ELT>;
  static constexpr int NV = V::N;

  const KdParams& P;
  KdCtrl& C;
  unsigned char* buf;          // nbuf x (target slice, draft slice)
  const int lane, warp, cs, rank;
  int lo, n, bytes, nvec;      // this CTA's slice: logits [lo, lo + n), bytes, 16-byte vectors

  __device__ KdRow(const KdParams& p, KdCtrl& c, unsigned char* b, int ln, int wp, int ncta, int rk)
      : P(p), C(c), buf(b), lane(ln), warp(wp), cs(ncta), rank(rk) {
    lo = min(p.V, rank * p.slice_elems);
    n = min(p.V, lo + p.slice_elems) - lo;
    bytes = n * ELT;
    nvec = (bytes + 15) / 16;
  }

  __device__ unsigned char* tslice(int b) const { return buf + static_cast<size_t>(b) * 2 * P.slot_bytes; }
  __device__ unsigned char* dslice(int b) const { return tslice(b) + P.slot_bytes; }
  __device__ uint4 vec(const unsigned char* s, int v) const { return *reinterpret_cast<const uint4*>(s + static_cast<size_t>(v) * 16); }

  // ---- producer warp: stage the slices of this cluster's rows --------------
  __device__ void stage(const unsigned char* src, unsigned char* dst, int r, uint64_t* bar) const {
    const unsigned char* row = static_cast<const unsigned char*>(src) +
                               (static_cast<size_t>(r) * P.V + lo) * static_cast<size_t>(ELT);
    if (P.bulk) {
      if (lane == 0 && bytes > 0) bulk_load(dst, row, static_cast<uint32_t>(bytes), bar);
    } else {
      const int npad = nvec * NV;
      for (int e = lane; e < npad; e += 32)
        V::store_scalar(dst, e, e < n ? V::scalar(row, e) : -INFINITY);
    }
  }

  __device__ void produce(int first, int stride, int niter, unsigned int* failed) {
    for (int i = 0; i < niter; ++i) {
      const int b = i % P.nbuf;
      const uint32_t par = static_cast<uint32_t>(i / P.nbuf) & 1u;
      int ok = 1;
      if (lane == 0) ok = mbar_wait_bounded(&C.empty[b], par ^ 1u, kDrainLimitNs) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) { if (lane == 0) atomicOr(failed, 1u); return; }
      const int r = first + i * stride;
      if (lane == 0 && P.bulk) mbar_expect_tx(&C.full[b], static_cast<uint32_t>(2 * bytes));
      stage(static_cast<const unsigned char*>(P.target), tslice(b), r, &C.full[b]);
      stage(static_cast<const unsigned char*>(P.draft), dslice(b), r, &C.full[b]);
      if (!P.bulk) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&C.full[b]);
      }
    }
  }

  // ---- compute warps ---------------------------------------------------------

  // This CTA's part of the row in buffer b, sent to every CTA of the cluster.
  __device__ void pass1_send(int b, int xs) {
    const unsigned char* ts = tslice(b);
    const unsigned char* ds = dslice(b);
    const int per_warp = (nvec + kKdWarps - 1) / kKdWarps;
    const int v0 = warp * per_warp, v1 = min(nvec, v0 + per_warp);
    // this lane's maxima (packed; NaN is passed over here and caught by the
    // sums, or below when a lane holds nothing but -inf and NaN), then its
    // sums against K = fl(M c)
    float mt = -INFINITY, md = -INFINITY;
    for (int v = v0 + lane; v < v1; v += 32) {
      const uint4 tv[1] = {vec(ts, v)}, dv[1] = {vec(ds, v)};
      mt = fmaxf(mt, V::vmax(tv));
      md = fmaxf(md, V::vmax(dv));
    }
    const float c2 = P.c2;
    // (a lane whose logits are all -inf adds nothing)
    const float kt = __fmul_rn(mt, c2), kd = __fmul_rn(md, c2);
    const bool any_t = mt != -INFINITY, any_d = md != -INFINITY;
    if (!any_t || !any_d) {
      int nan_seen = 0;
      for (int v = v0 + lane; v < v1; v += 32) {
        float zt[NV], zd[NV];
        V::unpack(vec(ts, v), zt);
        V::unpack(vec(ds, v), zd);
#pragma unroll
        for (int e = 0; e < NV; ++e) nan_seen |= (zt[e] != zt[e]) | (zd[e] != zd[e]);
      }
      if (nan_seen) { mt = NAN; md = NAN; }
    }
    float st = 0.f, a = 0.f, sd = 0.f;
    for (int v = v0 + lane; v < v1; v += 32) {
      float zt[NV], zd[NV];
      V::unpack(vec(ts, v), zt);
      V::unpack(vec(ds, v), zd);
#pragma unroll
      for (int e = 0; e < NV; ++e) {
        const float et = any_t ? fast_exp2(fmaf(zt[e], c2, -kt)) : 0.f;   // NaN logits stay NaN
        const float ed = any_d ? fast_exp2(fmaf(zd[e], c2, -kd)) : 0.f;
        st += et;
        sd += ed;
        // p(x) = 0 contributes nothing, also against q(x) = 0
        a = fmaf(et, zt[e] == -INFINITY ? 0.f : zt[e] - zd[e], a);
      }
    }
    KdPart mine;
    mine.mt = mt; mine.st = st; mine.a = a; mine.md = md; mine.sd = sd;
    mine.pad0 = mine.pad1 = mine.pad2 = 0.f;
    const KdPart w = combine_parts(mine, true, 32, c2);
    if (lane == 0) C.wpart[warp] = w;
    named_barrier_sync(kKdBarCompute, kKdWarps * 32);
    if (warp == 0) {
      KdPart wp = C.wpart[lane < kKdWarps ? lane : 0];
      const KdPart part = combine_parts(wp, lane < kKdWarps, kKdWarps, c2);
      if (lane < cs) {
        const uint32_t dst = peer(&C.xpart[xs][rank], lane);
        const uint32_t bar = peer(&C.xbar[xs], lane);
        st_async(dst, make_uint4(__float_as_uint(part.mt), __float_as_uint(part.st), __float_as_uint(part.a),
                                 __float_as_uint(part.md)), bar);
        st_async(dst + 16, make_uint4(__float_as_uint(part.sd), 0u, 0u, 0u), bar);
      }
      __syncwarp();
    }
  }

  // The row's numbers from every CTA's part (the same in every warp and CTA).
  __device__ KdPart gather(int xs, int i, bool& arrived) {
    arrived = mbar_wait_bounded(&C.xbar[xs], static_cast<uint32_t>(i / kKdXRing) & 1u, kDrainLimitNs);
    const bool in = lane < cs;
    KdPart pt = C.xpart[xs][in ? lane : 0];
    int n_pow2 = 1;
    while (n_pow2 < cs) n_pow2 <<= 1;
    return combine_parts(pt, in, n_pow2, P.c2);
  }

  // Gradient of this CTA's slice of the row in buffer b.
  __device__ void pass2(int b, int r, const KdPart& row, bool valid) {
    const unsigned char* ts = tslice(b);
    const unsigned char* ds = dslice(b);
    const float c2 = P.c2;
    const float kt = __fmul_rn(row.mt, c2), kd = __fmul_rn(row.md, c2);
    float lt, ld;
    asm("lg2.approx.f32 %0, %1;" : "=f"(lt) : "f"(row.st));
    asm("lg2.approx.f32 %0, %1;" : "=f"(ld) : "f"(row.sd));
    const float scale = P.weights[r / P.t_len] * P.inv_T;
    const float ct = valid ? -(kt + lt) : NAN;   // log2 p(x) = z c - K - log2 S, one fma
    const float cd = valid ? -(kd + ld) : NAN;   // (an invalid row writes NaN)
    unsigned char* out = static_cast<unsigned char*>(P.grad) + (static_cast<size_t>(r) * P.V + lo) * static_cast<size_t>(ELT);
    const int per_warp = (nvec + kKdWarps - 1) / kKdWarps;
    const int v0 = warp * per_warp, v1 = min(nvec, v0 + per_warp);
    for (int v = v0 + lane; v < v1; v += 32) {
      float zt[NV], zd[NV], g[NV];
      V::unpack(vec(ts, v), zt);
      V::unpack(vec(ds, v), zd);
#pragma unroll
      for (int e = 0; e < NV; ++e) {
        const float p = fast_exp2(fmaf(zt[e], c2, ct));
        const float q = fast_exp2(fmaf(zd[e], c2, cd));
        g[e] = scale * (q - p);
      }
      if (P.bulk) {
        *reinterpret_cast<uint4*>(out + static_cast<size_t>(v) * 16) = V::pack(g);
      } else {
#pragma unroll
        for (int e = 0; e < NV; ++e)
          if (v * NV + e < n) V::store_rounded(out, v * NV + e, g[e]);
      }
    }
  }

  // Two orders of the work of a row:
  //  * three or more buffers (loads issued well ahead): row i+1's first pass
  //    and part go out before row i's parts are awaited, hiding the exchange;
  //  * one or two buffers: row i is finished (exchange, KL, gradient, buffer
  //    released) before row i+1's first pass, so that the load of row i+2 into
  //    the released buffer has that first pass, an exchange and a gradient to
  //    hide behind.
  // Either way a CTA sends a row's part only after reading every part of the
  // row two before it, and a peer's part of that row was sent after the peer
  // read the row three before: at most four rows of parts are ever in the
  // four exchange slots.
  __device__ void compute(int first, int stride, int niter) {
    if (niter <= 0) return;
    const bool ahead = P.nbuf >= 3;
    mbar_wait_bounded(&C.full[0], 0u, kDrainLimitNs);
    pass1_send(0, 0);
    for (int i = 0; i < niter; ++i) {
      const int b = i % P.nbuf;
      const int xs = i % kKdXRing;
      if (ahead && i + 1 < niter) {
        const int bn = (i + 1) % P.nbuf;
        mbar_wait_bounded(&C.full[bn], static_cast<uint32_t>((i + 1) / P.nbuf) & 1u, kDrainLimitNs);
        pass1_send(bn, (i + 1) % kKdXRing);
      }
      bool arrived = true;
      const KdPart row = gather(xs, i, arrived);
      if (warp == 0 && lane == 0) mbar_expect_tx(&C.xbar[xs], static_cast<uint32_t>(cs * sizeof(KdPart)));
      const int r = first + i * stride;
      const bool valid = arrived && isfinite(row.mt) && isfinite(row.md) && isfinite(row.st) && isfinite(row.sd) &&
                         row.st > 0.f && row.sd > 0.f && !isnan(row.a);
      if (rank == 0 && warp == 0 && lane == 0) {
        // KL / ln 2 = c A / S^t - (K^t - K^d) - log2(S^t / S^d), with the very
        // K = fl(M c) and sums the exponentials were taken against
        double kl = NAN;
        if (valid) {
          const double kt = __fmul_rn(row.mt, P.c2), kd = __fmul_rn(row.md, P.c2);
          kl = 0.69314718055994530942 *
               (static_cast<double>(P.c2) * static_cast<double>(row.a) / static_cast<double>(row.st) -
                (kt - kd) - log2(static_cast<double>(row.st) / static_cast<double>(row.sd)));
        }
        P.row_kl[r] = static_cast<float>(kl);
      }
      if (GRAD) pass2(b, r, row, valid);
      __syncwarp();
      if (lane == 0) mbar_arrive(&C.empty[b]);
      if (!ahead && i + 1 < niter) {
        const int bn = (i + 1) % P.nbuf;
        mbar_wait_bounded(&C.full[bn], static_cast<uint32_t>((i + 1) / P.nbuf) & 1u, kDrainLimitNs);
        pass1_send(bn, (i + 1) % kKdXRing);
      }
    }
  }
};

template <int ELT, bool GRAD>
__global__ void __launch_bounds__(kKdThreads, 1) kd_kernel(const KdParams P, unsigned int* failed) {
  extern __shared__ __align__(1024) unsigned char smem[];
  KdCtrl& C = *reinterpret_cast<KdCtrl*>(smem);
  unsigned char* buf = smem + kKdCtrlBytes;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cs = cluster_ctas();
  if (tid == 0) {
    for (int b = 0; b < kKdMaxBuf; ++b) {
      mbar_init(&C.full[b], 1);
      mbar_init(&C.empty[b], kKdWarps);
    }
    for (int x = 0; x < kKdXRing; ++x) mbar_init(&C.xbar[x], 1);
    fence_mbar_init();
    for (int x = 0; x < kKdXRing; ++x) mbar_expect_tx(&C.xbar[x], static_cast<uint32_t>(cs * sizeof(KdPart)));
  }
  cluster_sync();
  {
    uint32_t cid, ncl;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(cid));
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(ncl));
    const int first = static_cast<int>(cid), stride = static_cast<int>(ncl);
    const int niter = first < P.rows ? (P.rows - first + stride - 1) / stride : 0;
    KdRow<ELT, GRAD> k(P, C, buf, lane, warp, cs, cluster_rank());
    if (warp == kKdWarps) k.produce(first, stride, niter, failed);
    else k.compute(first, stride, niter);
  }
  cluster_sync();   // no CTA leaves while a peer may still write into its shared memory
}

// loss[b] = w_b * sum_t row_kl[b, t], in position order.
__global__ void kd_loss_kernel(int n_seq, int t_len, const float* row_kl, const float* weights, float* loss) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= n_seq) return;
  double s = 0.0;
  for (int t = 0; t < t_len; ++t) s += static_cast<double>(row_kl[static_cast<size_t>(b) * t_len + t]);
  loss[b] = static_cast<float>(static_cast<double>(weights[b]) * s);
}

// ---------------------------------------------------------------------------
// Host side: the launch shape per device, cached
// ---------------------------------------------------------------------------

constexpr int kKdSmemLimit = 227 * 1024;

struct KdShapeKey {
  int V = 0, elt = 0, grad = 0;
};

struct KdDevice {
  bool ready = false;
  int sms = 0;
  unsigned int* failed = nullptr;   // set by a producer that gave up (bounded wait)
  // launch shapes already worked out (the occupancy queries cost host time)
  static constexpr int kCached = 8;
  KdShapeKey key[kCached];
  int shape_cs[kCached] = {0}, shape_nbuf[kCached] = {0}, shape_slice[kCached] = {0}, shape_slot[kCached] = {0};
  int shape_clusters[kCached] = {0}, shape_smem[kCached] = {0};
  int next = 0;
};
std::mutex g_kd_mutex;
KdDevice g_kd[64];

template <int ELT, bool GRAD>
const void* kd_fn() { return reinterpret_cast<const void*>(&kd_kernel<ELT, GRAD>); }

const void* kd_kernel_for(int elt, bool grad) {
  if (elt == 2) return grad ? kd_fn<2, true>() : kd_fn<2, false>();
  return grad ? kd_fn<4, true>() : kd_fn<4, false>();
}

struct KdShape {
  int cs = 0, nbuf = 0, slice_elems = 0, slot = 0, max_clusters = 0, smem = 0;
};

// The cluster (1 .. 16 CTAs) and buffer count: as many row buffers as fit,
// up to kKdMaxBuf, taking the fewest CTAs per row that still give three
// buffers (rows keep arriving while earlier ones are reduced), else the
// deepest pipeline any launchable size allows.
bool kd_shape(int V, int elt, bool with_grad, KdShape* out) {
  const void* fn = kd_kernel_for(elt, with_grad);
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    (void)cudaGetLastError();
  KdShape best;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kKdThreads, 1, 1);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  for (int c = 1; c <= kKdMaxCluster; c *= 2) {
    const int per = static_cast<int>(((static_cast<long long>(V) + c - 1) / c + 63) / 64 * 64);
    const int sbytes = static_cast<int>(((static_cast<long long>(per) * elt) + 127) / 128 * 128);
    int nb = static_cast<int>((kKdSmemLimit - kKdCtrlBytes) / (2LL * sbytes));
    if (nb > kKdMaxBuf) nb = kKdMaxBuf;
    if (nb < 1) continue;
    if (best.cs != 0 && (best.nbuf >= 3 || nb <= best.nbuf)) continue;
    const int sm = kKdCtrlBytes + nb * 2 * sbytes;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, sm) != cudaSuccess) {
      (void)cudaGetLastError();
      continue;
    }
    attr[0].val.clusterDim.x = static_cast<unsigned>(c);
    cfg.gridDim = dim3(static_cast<unsigned>(c), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(sm);
    int mc = 0;
    if (cudaOccupancyMaxActiveClusters(&mc, fn, &cfg) != cudaSuccess || mc <= 0) {
      (void)cudaGetLastError();
      continue;
    }
    best.cs = c; best.nbuf = nb; best.slice_elems = per; best.slot = sbytes; best.max_clusters = mc; best.smem = sm;
  }
  if (best.cs == 0) return false;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, best.smem) != cudaSuccess) return false;
  *out = best;
  return true;
}

}  // namespace
}  // namespace sv

extern "C" sv_status spec_kd_loss(int n_seq, int t_len, int V, sv_dtype dtype, const void* target_logits,
                                  const void* draft_logits, const float* weights, float temperature,
                                  float* row_kl, float* loss, void* grad, sv_stream_t stream) {
  using namespace sv;
  if (n_seq < 1 || t_len < 1 || V < 1) return SV_ERR_INVALID_ARG;
  if (static_cast<long long>(n_seq) * t_len > (1LL << 30)) return SV_ERR_INVALID_ARG;
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || !std::isfinite(temperature)) return SV_ERR_INVALID_ARG;
  if (!target_logits || !draft_logits || !weights || !row_kl || !loss) return SV_ERR_INVALID_ARG;
  const int elt = dtype == SV_F32 ? 4 : 2;
  const long long row_bytes = static_cast<long long>(V) * elt;
  const double c2 = 1.4426950408889634 / static_cast<double>(temperature);
  if (!(c2 < 1e30)) return SV_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  if (dev < 0 || dev >= 64) return SV_ERR_UNSUPPORTED;
  KdDevice* D = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_kd_mutex);
    KdDevice& d = g_kd[dev];
    if (!d.ready) {
      cudaDeviceProp prop;
      if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return SV_ERR_CUDA;
      if (!(prop.major == 10 && prop.minor == 3)) return SV_ERR_UNSUPPORTED;
      if (cudaMalloc(&d.failed, sizeof(unsigned int)) != cudaSuccess) return SV_ERR_CUDA;
      if (cudaMemset(d.failed, 0, sizeof(unsigned int)) != cudaSuccess) return SV_ERR_CUDA;
      d.sms = prop.multiProcessorCount;
      d.ready = true;
    }
    D = &d;
  }

  const bool with_grad = grad != nullptr;
  KdShape sh;
  {
    std::lock_guard<std::mutex> lock(g_kd_mutex);
    int hit = -1;
    for (int c = 0; c < KdDevice::kCached; ++c)
      if (D->key[c].V == V && D->key[c].elt == elt && D->key[c].grad == (with_grad ? 1 : 0) && D->shape_cs[c] > 0)
        hit = c;
    if (hit >= 0) {
      sh.cs = D->shape_cs[hit]; sh.nbuf = D->shape_nbuf[hit]; sh.slice_elems = D->shape_slice[hit];
      sh.slot = D->shape_slot[hit]; sh.max_clusters = D->shape_clusters[hit]; sh.smem = D->shape_smem[hit];
    } else {
      if (!kd_shape(V, elt, with_grad, &sh)) return SV_ERR_UNSUPPORTED;
      const int c = D->next;
      D->next = (D->next + 1) % KdDevice::kCached;
      D->key[c].V = V; D->key[c].elt = elt; D->key[c].grad = with_grad ? 1 : 0;
      D->shape_cs[c] = sh.cs; D->shape_nbuf[c] = sh.nbuf; D->shape_slice[c] = sh.slice_elems;
      D->shape_slot[c] = sh.slot; D->shape_clusters[c] = sh.max_clusters; D->shape_smem[c] = sh.smem;
    }
  }
  // the kernel's shared-memory size may have been set for another shape meanwhile
  if (cudaFuncSetAttribute(kd_kernel_for(elt, with_grad), cudaFuncAttributeMaxDynamicSharedMemorySize, sh.smem) !=
      cudaSuccess)
    return SV_ERR_CUDA;
  const int cs = sh.cs, nbuf = sh.nbuf, slice_elems = sh.slice_elems, slot = sh.slot;
  const int max_clusters = sh.max_clusters, smem = sh.smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kKdThreads, 1, 1);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  const int rows = n_seq * t_len;
  const int clusters = rows < max_clusters ? rows : max_clusters;
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * cs), 1, 1);

  KdParams p{};
  p.target = target_logits;
  p.draft = draft_logits;
  p.weights = weights;
  p.row_kl = row_kl;
  p.grad = grad;
  p.rows = rows;
  p.t_len = t_len;
  p.V = V;
  p.c2 = static_cast<float>(c2);
  p.inv_T = 1.f / temperature;
  p.slice_elems = slice_elems;
  p.slot_bytes = slot;
  p.nbuf = nbuf;
  auto aligned = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  p.bulk = (row_bytes % 16 == 0) && aligned(target_logits) && aligned(draft_logits) &&
           (grad == nullptr || aligned(grad));
  sv::NvtxRange range("spec_kd_loss");
  cudaError_t e;
  if (elt == 2)
    e = with_grad ? cudaLaunchKernelEx(&cfg, kd_kernel<2, true>, p, D->failed)
                  : cudaLaunchKernelEx(&cfg, kd_kernel<2, false>, p, D->failed);
  else
    e = with_grad ? cudaLaunchKernelEx(&cfg, kd_kernel<4, true>, p, D->failed)
                  : cudaLaunchKernelEx(&cfg, kd_kernel<4, false>, p, D->failed);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  kd_loss_kernel<<<(n_seq + 255) / 256, 256, 0, cfg.stream>>>(n_seq, t_len, row_kl, weights, loss);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

extern "C" sv_status spec_kd_launch_shape(int V, sv_dtype dtype, int with_grad, int* cluster, int* buffers,
                                          int* grid_ctas) {
  using namespace sv;
  if (V < 1 || (dtype != SV_F32 && dtype != SV_BF16)) return SV_ERR_INVALID_ARG;
  KdShape sh;
  if (!kd_shape(V, dtype == SV_F32 ? 4 : 2, with_grad != 0, &sh)) return SV_ERR_UNSUPPORTED;
  if (cluster) *cluster = sh.cs;
  if (buffers) *buffers = sh.nbuf;
  if (grid_ctas) *grid_ctas = sh.max_clusters * sh.cs;
  return SV_OK;
}
