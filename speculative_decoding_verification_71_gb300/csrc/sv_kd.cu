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
//
// Rows are independent: a persistent grid of one CTA per SM takes whole row
// pairs, row b + i * grid for CTA b.  A producer warp streams each pair
// through three 64 KB shared-memory slots with cp.async.bulk, 32 KB of the
// target row and the same 32 KB of the draft row per slot; 16 consumer warps
// fold every slot into running per-lane maxima and sums (two logits per
// f32x2 instruction).  At the row's end the warps' parts are combined, in a
// fixed order, into (M, S, A) and the KL.  For the gradient the producer
// streams the pair a second time right behind the first: those copies find
// the row in L2 (it was read a few microseconds before) and are marked first
// out of it, and the gradient leaves with streaming stores.  Each logit
// crosses HBM once and each gradient value once; no CTA waits for another.

#include <cuda_runtime.h>

#include <cfloat>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/specverify.h"
#include "sv_internal.h"
#include "sv_device.cuh"

namespace sv {
namespace {

constexpr int kKdWarps = 16;                          // consumer warps
constexpr int kKdThreads = (kKdWarps + 1) * 32;       // + the producer warp
constexpr int kKdStages = 3;                          // 64 KB staging slots
constexpr int kKdHalf = 32 * 1024;                    // one row's part of a slot
constexpr int kKdVecsPerWarp = kKdHalf / 16 / kKdWarps;   // 128 vectors of 16 bytes
constexpr int kKdVecsPerLane = kKdVecsPerWarp / 32;       // 4
constexpr int kKdBarCompute = 1;                      // named barrier of the consumer warps

struct alignas(16) KdPart {
  float mt, st, a, md;         // target max, target sum, weighted difference, draft max
  float sd, pad0, pad1, pad2;  // draft sum
};

struct KdCtrl {
  uint64_t full[kKdStages];    // slot filled (producer -> consumers)
  uint64_t empty[kKdStages];   // slot released (one arrival per consumer warp)
  KdPart wpart[2][kKdWarps];   // per-warp parts of a row (by row parity)
};
constexpr int kKdCtrlBytes = ((static_cast<int>(sizeof(KdCtrl)) + 1023) / 1024) * 1024;
constexpr int kKdSmemBytes = kKdCtrlBytes + kKdStages * 2 * kKdHalf;
static_assert(kKdSmemBytes <= 227 * 1024, "three slots must fit in one CTA");

struct KdParams {
  const void* target;          // [rows, V]
  const void* draft;           // [rows, V]
  const float* weights;        // [rows / t_len]
  float* row_kl;               // [rows]
  void* grad;                  // [rows, V] (GRAD only)
  int rows, t_len, V;
  float c2;                    // log2(e) / T
  float inv_T;
  int nchunks;                 // slots per row and pass: ceil(V * elt / kKdHalf)
  int bulk;                    // rows 16-byte aligned: cp.async.bulk; else plain loads
};

// A part's numbers rescaled onto the common maxima of the parts in lanes
// 0..n-1 (warp-wide; every lane returns the combined part).  The sums are
// added in a fixed butterfly order, so every warp that combines the same
// parts gets the same bits.
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

// Rescale a lane's running sums onto a larger maximum vm (also the first
// time: the sums start empty).
__device__ __forceinline__ void raise_max(float vm, float c2, float& m, float& k, f2& s, f2& a) {
  const float kn = __fmul_rn(vm, c2);
  const float f = m == -INFINITY ? 0.f : fast_exp2(__fsub_rn(k, kn));
  const f2 ff = pack2(f, f);
  s = mul2(s, ff);
  a = mul2(a, ff);
  m = vm;
  k = kn;
}

// 16 bytes to global memory, marked as read by nobody soon (st.global.cs).
__device__ __forceinline__ void store_streaming(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.b32 [%0], {%1, %2, %3, %4};"
               :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

template <int ELT, bool GRAD>
struct KdRows {
  using V = Vec<ELT>;
  static constexpr int NV = V::N;

  const KdParams& P;
  KdCtrl& C;
  unsigned char* ring;         // kKdStages slots of (target part, draft part)
  unsigned int* failed;        // bit 0: the producer gave up; bit 1: a consumer did
  const int lane, warp;
  const long long row_bytes;

  __device__ KdRows(const KdParams& p, KdCtrl& c, unsigned char* r, unsigned int* f, int ln, int wp)
      : P(p), C(c), ring(r), failed(f), lane(ln), warp(wp), row_bytes(static_cast<long long>(p.V) * ELT) {}

  __device__ unsigned char* slot(int s) const { return ring + static_cast<size_t>(s) * 2 * kKdHalf; }
  __device__ int chunk_bytes(int c) const {
    const long long left = row_bytes - static_cast<long long>(c) * kKdHalf;
    return static_cast<int>(left < kKdHalf ? left : kKdHalf);
  }

  // ---- producer warp ---------------------------------------------------------
  // Every row pair once (and for the gradient twice, the second time right
  // behind the first), kKdHalf bytes of each row per slot.
  __device__ void produce() {
    const uint64_t first_out = evict_first_policy();
    const int passes = GRAD ? 2 : 1;
    int q = 0;
    for (int r = blockIdx.x; r < P.rows; r += gridDim.x) {
      const unsigned char* rt = static_cast<const unsigned char*>(P.target) + static_cast<size_t>(r) * row_bytes;
      const unsigned char* rd = static_cast<const unsigned char*>(P.draft) + static_cast<size_t>(r) * row_bytes;
      for (int pass = 0; pass < passes; ++pass) {
        // a pass read again keeps its lines in L2; the last read of a row
        // marks them first out
        const bool last_read = pass == passes - 1;
        for (int c = 0; c < P.nchunks; ++c, ++q) {
          const int s = q % kKdStages;
          int ok = 1;
          if (lane == 0) ok = mbar_wait_bounded(&C.empty[s], ((q / kKdStages) & 1) ^ 1, kDrainLimitNs) ? 1 : 0;
          if (!__shfl_sync(0xffffffffu, ok, 0)) {
            if (lane == 0) atomicOr(failed, 1u);
            return;
          }
          const long long off = static_cast<long long>(c) * kKdHalf;
          const int bytes = chunk_bytes(c);
          unsigned char* dst = slot(s);
          if (P.bulk) {
            if (lane == 0) {
              mbar_expect_tx(&C.full[s], static_cast<uint32_t>(2 * bytes));
              if (last_read) {
                bulk_load_hint(dst, rt + off, static_cast<uint32_t>(bytes), &C.full[s], first_out);
                bulk_load_hint(dst + kKdHalf, rd + off, static_cast<uint32_t>(bytes), &C.full[s], first_out);
              } else {
                bulk_load(dst, rt + off, static_cast<uint32_t>(bytes), &C.full[s]);
                bulk_load(dst + kKdHalf, rd + off, static_cast<uint32_t>(bytes), &C.full[s]);
              }
            }
          } else {
            // rows not 16-byte aligned: plain loads, the last vector padded with -inf
            const long long e0 = off / ELT;
            const int n = bytes / ELT;
            const int npad = (n + NV - 1) / NV * NV;
            for (int e = lane; e < npad; e += 32) {
              V::store_scalar(dst, e, e < n ? V::scalar(rt, e0 + e) : -INFINITY);
              V::store_scalar(dst + kKdHalf, e, e < n ? V::scalar(rd, e0 + e) : -INFINITY);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&C.full[s]);
          }
        }
      }
    }
  }

  // ---- consumer warps --------------------------------------------------------

  // This lane's vectors of slot s (target, draft), -inf past the chunk; the
  // slot is released as soon as they are in registers.  False if the wait
  // gave up (every later wait is then skipped: the rows turn NaN).
  __device__ bool take(int s, int q, int c, bool& dead, uint4 (&tv)[kKdVecsPerLane], uint4 (&dv)[kKdVecsPerLane]) {
    bool ok = !dead && mbar_wait_bounded(&C.full[s], static_cast<uint32_t>(q / kKdStages) & 1u, kDrainLimitNs);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && !dead) {
      dead = true;
      if (lane == 0) atomicOr(failed, 2u);
    }
    const int nvec = (chunk_bytes(c) + 15) / 16;
    const unsigned char* src = slot(s);
#pragma unroll
    for (int j = 0; j < kKdVecsPerLane; ++j) {
      const int v = warp * kKdVecsPerWarp + j * 32 + lane;
      const bool in = v < nvec;
      tv[j] = in ? *reinterpret_cast<const uint4*>(src + static_cast<size_t>(v) * 16) : V::neg_inf();
      dv[j] = in ? *reinterpret_cast<const uint4*>(src + kKdHalf + static_cast<size_t>(v) * 16) : V::neg_inf();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&C.empty[s]);
    return ok;
  }

  __device__ void consume() {
    const float c2 = P.c2;
    const f2 cc = pack2(c2, c2);
    int q = 0, row_i = 0;
    bool dead = false;
    for (int r = blockIdx.x; r < P.rows; r += gridDim.x, ++row_i) {
      // ---- first pass: per lane, running maxima and sums against K = fl(M c)
      float mt = -INFINITY, md = -INFINITY, kt = 0.f, kd = 0.f;
      f2 st2 = 0ull, sd2 = 0ull, a2 = 0ull, unused = 0ull;
      bool lost = false;
      for (int c = 0; c < P.nchunks; ++c, ++q) {
        uint4 tv[kKdVecsPerLane], dv[kKdVecsPerLane];
        if (!take(q % kKdStages, q, c, dead, tv, dv)) lost = true;
        // NaN is passed over by the maxima and kept by the sums
        const float vt = V::vmax(tv), vd = V::vmax(dv);
        if (vt > mt) raise_max(vt, c2, mt, kt, st2, a2);
        if (vd > md) raise_max(vd, c2, md, kd, sd2, unused);
        const f2 nkt = pack2(-kt, -kt), nkd = pack2(-kd, -kd);
#pragma unroll
        for (int j = 0; j < kKdVecsPerLane; ++j) {
          f2 zt[NV / 2], zd[NV / 2];
          V::pairs(tv[j], zt);
          V::pairs(dv[j], zd);
#pragma unroll
          for (int i = 0; i < NV / 2; ++i) {
            // while a lane's maximum is -inf its K is 0 and 2^(-inf) adds 0
            const f2 et = exp2_2(fma2(zt[i], cc, nkt));
            const f2 ed = exp2_2(fma2(zd[i], cc, nkd));
            st2 = add2(st2, et);
            sd2 = add2(sd2, ed);
            // p(x) = 0 (z^t = -inf) adds nothing, also against q(x) = 0: the
            // difference is clamped to a finite value that the zero multiplies
            float d0, d1;
            unpack2(sub2(zt[i], zd[i]), d0, d1);
            a2 = fma2(et, pack2(fmaxf(d0, -FLT_MAX), fmaxf(d1, -FLT_MAX)), a2);
          }
        }
      }
      // ---- the row's numbers, the same in every warp
      float x0, x1;
      KdPart mine;
      unpack2(st2, x0, x1); mine.st = x0 + x1;
      unpack2(a2, x0, x1);  mine.a = x0 + x1;
      unpack2(sd2, x0, x1); mine.sd = x0 + x1;
      // a NaN sum is carried by the maximum (a lane whose maximum stayed
      // -inf would otherwise drop it in the combine); so is a lost wait
      mine.mt = (mine.st != mine.st || lost) ? NAN : mt;
      mine.md = (mine.sd != mine.sd || lost) ? NAN : md;
      mine.pad0 = mine.pad1 = mine.pad2 = 0.f;
      const KdPart w = combine_parts(mine, true, 32, c2);
      if (lane == 0) C.wpart[row_i & 1][warp] = w;
      named_barrier_sync(kKdBarCompute, kKdWarps * 32);
      const KdPart row = combine_parts(C.wpart[row_i & 1][lane < kKdWarps ? lane : 0], lane < kKdWarps, kKdWarps, c2);
      const bool valid = isfinite(row.mt) && isfinite(row.md) && isfinite(row.st) && isfinite(row.sd) &&
                         row.st > 0.f && row.sd > 0.f && !isnan(row.a);
      if (warp == 0 && lane == 0) P.row_kl[r] = row_kl(row, valid);
      if (GRAD) gradient(r, row, valid, q, dead);
    }
  }

  // KL / ln 2 = c A / S^t - (K^t - K^d) - log2(S^t / S^d), with the very
  // K = fl(M c) and sums the exponentials were taken against.  In fp32
  // without losing the difference: c A / S^t as hi + lo (fused multiply-add),
  // K^t - K^d and the final difference by TwoSum; the error left is that of
  // A / S^t's rounding and of the sums themselves.
  __device__ float row_kl(const KdPart& row, bool valid) const {
    if (!valid) return NAN;
    const float kt = __fmul_rn(row.mt, P.c2), kd = __fmul_rn(row.md, P.c2);
    const float q = __fdiv_rn(row.a, row.st);
    const float h1 = __fmul_rn(P.c2, q);
    if (isinf(h1)) return h1;   // q(x) = 0 where p(x) > 0: A, hence KL, is +inf
    const float l1 = __fmaf_rn(P.c2, q, -h1);
    float h2, l2, h3, l3;
    two_sum(kt, -kd, h2, l2);
    two_sum(h1, -h2, h3, l3);
    const float rest = __fadd_rn(__fsub_rn(l1, l2), l3) - log2f(__fdiv_rn(row.st, row.sd));
    return __fmul_rn(0.6931471805599453f, __fadd_rn(h3, rest));
  }

  // ---- second pass: w (q - p) / T for every logit of the row pair
  __device__ void gradient(int r, const KdPart& row, bool valid, int& q, bool& dead) {
    const float c2 = P.c2;
    const float kt = __fmul_rn(row.mt, c2), kd = __fmul_rn(row.md, c2);
    float lt, ld;
    asm("lg2.approx.f32 %0, %1;" : "=f"(lt) : "f"(row.st));
    asm("lg2.approx.f32 %0, %1;" : "=f"(ld) : "f"(row.sd));
    const float scale = P.weights[r / P.t_len] * P.inv_T;
    const float ct = valid ? -(kt + lt) : NAN;   // log2 p(x) = z c - K - log2 S, one fma
    const float cd = valid ? -(kd + ld) : NAN;   // (an invalid row writes NaN)
    const f2 cc = pack2(c2, c2), ct2 = pack2(ct, ct), cd2 = pack2(cd, cd), sc2 = pack2(scale, scale);
    unsigned char* out_row = static_cast<unsigned char*>(P.grad) + static_cast<size_t>(r) * row_bytes;
    for (int c = 0; c < P.nchunks; ++c, ++q) {
      uint4 tv[kKdVecsPerLane], dv[kKdVecsPerLane];
      take(q % kKdStages, q, c, dead, tv, dv);
      const int nvec = (chunk_bytes(c) + 15) / 16;
      unsigned char* out = out_row + static_cast<size_t>(c) * kKdHalf;
#pragma unroll
      for (int j = 0; j < kKdVecsPerLane; ++j) {
        const int v = warp * kKdVecsPerWarp + j * 32 + lane;
        f2 zt[NV / 2], zd[NV / 2];
        V::pairs(tv[j], zt);
        V::pairs(dv[j], zd);
        float g[NV];
#pragma unroll
        for (int i = 0; i < NV / 2; ++i) {
          const f2 pp = exp2_2(fma2(zt[i], cc, ct2));
          const f2 qq = exp2_2(fma2(zd[i], cc, cd2));
          unpack2(mul2(sc2, sub2(qq, pp)), g[2 * i], g[2 * i + 1]);
        }
        if (v >= nvec) continue;
        if (P.bulk) {
          store_streaming(out + static_cast<size_t>(v) * 16, V::pack(g));
        } else {
          const int n = chunk_bytes(c) / ELT;
#pragma unroll
          for (int e = 0; e < NV; ++e)
            if (v * NV + e < n) V::store_rounded(out, v * NV + e, g[e]);
        }
      }
    }
  }
};

template <int ELT, bool GRAD>
__global__ void __launch_bounds__(kKdThreads, 1) kd_kernel(const KdParams P, unsigned int* failed) {
  extern __shared__ __align__(1024) unsigned char smem[];
  KdCtrl& C = *reinterpret_cast<KdCtrl*>(smem);
  unsigned char* ring = smem + kKdCtrlBytes;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < kKdStages; ++s) {
      mbar_init(&C.full[s], 1);
      mbar_init(&C.empty[s], kKdWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  KdRows<ELT, GRAD> k(P, C, ring, failed, lane, warp);
  if (warp == kKdWarps) k.produce();
  else k.consume();
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
// Host side
// ---------------------------------------------------------------------------

struct KdDevice {
  bool ready = false;
  int sms = 0;
  unsigned int* failed = nullptr;   // set by a warp that gave up a bounded wait
  bool smem_set[4] = {false, false, false, false};
};
std::mutex g_kd_mutex;
KdDevice g_kd[64];

template <int ELT, bool GRAD>
const void* kd_fn() { return reinterpret_cast<const void*>(&kd_kernel<ELT, GRAD>); }

const void* kd_kernel_for(int elt, bool grad) {
  if (elt == 2) return grad ? kd_fn<2, true>() : kd_fn<2, false>();
  return grad ? kd_fn<4, true>() : kd_fn<4, false>();
}

// The device's record, set up once (its properties, the failure word).
sv_status kd_device(KdDevice** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  if (dev < 0 || dev >= 64) return SV_ERR_UNSUPPORTED;
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
  *out = &d;
  return SV_OK;
}

// The kernel's shared-memory limit, raised once per instance and device.
sv_status kd_prepare(KdDevice* d, int elt, bool grad) {
  const int i = (elt == 2 ? 0 : 2) + (grad ? 1 : 0);
  std::lock_guard<std::mutex> lock(g_kd_mutex);
  if (d->smem_set[i]) return SV_OK;
  if (cudaFuncSetAttribute(kd_kernel_for(elt, grad), cudaFuncAttributeMaxDynamicSharedMemorySize, kKdSmemBytes) !=
      cudaSuccess)
    return SV_ERR_CUDA;
  d->smem_set[i] = true;
  return SV_OK;
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
  if (row_bytes > (1LL << 30)) return SV_ERR_INVALID_ARG;
  const double c2 = 1.4426950408889634 / static_cast<double>(temperature);
  if (!(c2 < 1e30)) return SV_ERR_INVALID_ARG;

  KdDevice* D = nullptr;
  sv_status st = kd_device(&D);
  if (st != SV_OK) return st;
  const bool with_grad = grad != nullptr;
  if ((st = kd_prepare(D, elt, with_grad)) != SV_OK) return st;

  const int rows = n_seq * t_len;
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
  p.nchunks = static_cast<int>((row_bytes + kKdHalf - 1) / kKdHalf);
  auto aligned = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  p.bulk = (row_bytes % 16 == 0) && aligned(target_logits) && aligned(draft_logits) &&
           (grad == nullptr || aligned(grad));
  // one CTA per SM, every row to the CTA b + i * grid
  const int ctas = rows < D->sms ? rows : D->sms;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  sv::NvtxRange range("spec_kd_loss");
  if (elt == 2) {
    if (with_grad) kd_kernel<2, true><<<ctas, kKdThreads, kKdSmemBytes, s>>>(p, D->failed);
    else kd_kernel<2, false><<<ctas, kKdThreads, kKdSmemBytes, s>>>(p, D->failed);
  } else {
    if (with_grad) kd_kernel<4, true><<<ctas, kKdThreads, kKdSmemBytes, s>>>(p, D->failed);
    else kd_kernel<4, false><<<ctas, kKdThreads, kKdSmemBytes, s>>>(p, D->failed);
  }
  if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  kd_loss_kernel<<<(n_seq + 255) / 256, 256, 0, s>>>(n_seq, t_len, row_kl, weights, loss);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

extern "C" sv_status spec_kd_launch_shape(int V, sv_dtype dtype, int with_grad, int* cluster, int* buffers,
                                          int* grid_ctas) {
  using namespace sv;
  if (V < 1 || (dtype != SV_F32 && dtype != SV_BF16)) return SV_ERR_INVALID_ARG;
  (void)with_grad;
  KdDevice* D = nullptr;
  const sv_status st = kd_device(&D);
  if (st != SV_OK) return st;
  if (cluster) *cluster = 1;
  if (buffers) *buffers = kKdStages;
  if (grid_ctas) *grid_ctas = D->sms;
  return SV_OK;
}
