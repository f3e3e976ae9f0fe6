// Device helpers shared by the verification and the distillation kernels:
// PTX wrappers (mbarriers, bulk copies, L2 policies, programmatic launch),
// packed fp32 pairs, 16-byte logit vectors, warp reductions and the cluster
// (distributed shared memory) primitives.  Header-only, one copy per
// translation unit (everything here is in an unnamed namespace).
#pragma once

#include <cuda_bf16.h>
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
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
  f2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f2 exp2_2(f2 t) {
  float a, b;
  unpack2(t, a, b);
  return pack2(fast_exp2(a), fast_exp2(b));
}

// 1 - 2^d, accurate relative to the result as d -> 0 (where 1 - ex2(d)
// would cancel).  For d > -1/4 the Taylor series of
// 1 - 2^d = -(sum over n >= 1 of (d ln 2)^n / n!) up to n = 6, in Horner form
// in d with c_n = (ln 2)^n / n! (truncation below 6e-9 relative); below -1/4,
// 1 - 2^d >= 0.16 and the subtraction loses nothing.  d >= 0 gives a result
// <= 0 (or NaN for d = +inf), which callers clamp away.  The scalar and the
// packed form round identically, lane by lane.
constexpr float kSmallDelta = -0.25f;
__device__ __forceinline__ float one_minus_exp2(float d) {
  float s = __fmaf_rn(d, 1.5403530393381609e-4f, 1.3333558146428443e-3f);   // c6, c5
  s = __fmaf_rn(d, s, 9.6181291076284772e-3f);                               // c4
  s = __fmaf_rn(d, s, 5.5504108664821580e-2f);                               // c3
  s = __fmaf_rn(d, s, 2.4022650695910071e-1f);                               // c2
  s = __fmaf_rn(d, s, 6.9314718055994531e-1f);                               // c1 = ln 2
  const float small = -__fmul_rn(d, s);
  const float big = __fsub_rn(1.f, fast_exp2(d));
  return d > kSmallDelta ? small : big;
}
__device__ __forceinline__ f2 one_minus_exp2_2(f2 d) {
  // lane by lane: scalar multiply-adds take their constants as immediates,
  // where the packed form would hold six constant pairs in registers
  float d0, d1;
  unpack2(d, d0, d1);
  return pack2(one_minus_exp2(d0), one_minus_exp2(d1));
}

// The same with the series taken two lanes per f32x2 instruction (its six
// coefficient pairs live in registers: for kernels with registers to spare).
// Bit-identical to one_minus_exp2, lane by lane.
__device__ __forceinline__ f2 one_minus_exp2_2r(f2 d) {
  f2 s = fma2(d, pack2(1.5403530393381609e-4f, 1.5403530393381609e-4f),
              pack2(1.3333558146428443e-3f, 1.3333558146428443e-3f));
  s = fma2(d, s, pack2(9.6181291076284772e-3f, 9.6181291076284772e-3f));
  s = fma2(d, s, pack2(5.5504108664821580e-2f, 5.5504108664821580e-2f));
  s = fma2(d, s, pack2(2.4022650695910071e-1f, 2.4022650695910071e-1f));
  s = fma2(d, s, pack2(6.9314718055994531e-1f, 6.9314718055994531e-1f));
  float s0, s1, d0, d1;
  unpack2(mul2(d, s), s0, s1);
  unpack2(d, d0, d1);
  const float r0 = d0 > kSmallDelta ? -s0 : __fsub_rn(1.f, fast_exp2(d0));
  const float r1 = d1 > kSmallDelta ? -s1 : __fsub_rn(1.f, fast_exp2(d1));
  return pack2(r0, r1);
}

// a + b = s + e exactly (Knuth's TwoSum, six operations, no branch).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// G = (Ka - Kb) + log2(Sa / Sb), the log2 ratio of two normalisers 2^K S,
// as an unevaluated sum gh + gl: the difference of the K's is carried
// exactly, so the only roundings are those of Sa / Sb and of its log2 (a
// small number when the rows are alike).
__device__ __forceinline__ void log2_ratio(float Ka, float Sa, float Kb, float Sb, float& gh, float& gl) {
  float s1, e1, s2, e2;
  two_sum(Ka, -Kb, s1, e1);
  two_sum(s1, log2f(__fdiv_rn(Sa, Sb)), s2, e2);
  gh = s2;
  gl = __fadd_rn(e1, e2);
}

// Residual weight max(0, p - q) of one logit pair without cancellation:
// with log2 p = z_t c - K_t - L_t and log2 q = z_d c - K_d - L_d,
//   p - q = p (1 - 2^delta),  delta = log2 q - log2 p = (z_d - z_t) c + G,
// G = (K_t + L_t) - (K_d + L_d) the log2 ratio of the two normalisers, held
// as an unevaluated sum Gh + Gl of two floats.  The fused multiply-add
// rounds (z_d - z_t) c + Gh once, at the magnitude of delta itself, so delta
// (and the weight, relative to itself) stays accurate where p ~ q.  Returns
// the weight and sets p.
__device__ __forceinline__ float resid_weight(float zt, float zd, float c, float Kt, float Lt, float Gh, float Gl,
                                              float& p) {
  p = fast_exp2(__fsub_rn(__fmaf_rn(zt, c, -Kt), Lt));
  const float delta = __fadd_rn(__fmaf_rn(__fsub_rn(zd, zt), c, Gh), Gl);
  return fmaxf(__fmul_rn(p, one_minus_exp2(delta)), 0.f);
}
// The same for two pairs at once (bit-identical to the scalar form).
__device__ __forceinline__ void resid_weight2(f2 zt, f2 zd, f2 cc, f2 nkt, f2 nlt, f2 gh, f2 gl, f2& p, float& w0,
                                              float& w1) {
  p = exp2_2(add2(fma2(zt, cc, nkt), nlt));
  const f2 delta = add2(fma2(sub2(zd, zt), cc, gh), gl);
  unpack2(mul2(p, one_minus_exp2_2(delta)), w0, w1);
  w0 = fmaxf(w0, 0.f);
  w1 = fmaxf(w1, 0.f);
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
  // one fp32 value rounded to nearest-even bf16
  __device__ __forceinline__ static void store_rounded(unsigned char* base, int idx, float v) {
    reinterpret_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(v);
  }
  // eight fp32 values rounded to nearest-even bf16, in element order
  __device__ __forceinline__ static uint4 pack(const float (&v)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w[j]) : "f"(v[2 * j + 1]), "f"(v[2 * j]));
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
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
  // the same maximum, NaN if any value is NaN
  __device__ __forceinline__ static uint32_t max2_nan(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
  }
  template <int N>
  __device__ __forceinline__ static float vmax_nan(const uint4 (&r)[N]) {
    uint32_t m[4] = {r[0].x, r[0].y, r[0].z, r[0].w};
#pragma unroll
    for (int j = 1; j < N; ++j) {
      m[0] = max2_nan(m[0], r[j].x); m[1] = max2_nan(m[1], r[j].y);
      m[2] = max2_nan(m[2], r[j].z); m[3] = max2_nan(m[3], r[j].w);
    }
    const uint32_t w = max2_nan(max2_nan(m[0], m[1]), max2_nan(m[2], m[3]));
    float res;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(res) : "f"(__uint_as_float(w << 16)), "f"(__uint_as_float(w & 0xffff0000u)));
    return res;
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
  __device__ __forceinline__ static void store_rounded(unsigned char* base, int idx, float v) {
    reinterpret_cast<float*>(base)[idx] = v;
  }
  __device__ __forceinline__ static uint4 pack(const float (&v)[4]) {
    return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3]));
  }
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
  template <int N>
  __device__ __forceinline__ static float vmax_nan(const uint4 (&r)[N]) {
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < N; ++j) {
      const float a = __uint_as_float(r[j].x), b = __uint_as_float(r[j].y);
      const float c = __uint_as_float(r[j].z), d = __uint_as_float(r[j].w);
      asm("max.NaN.f32 %0, %0, %1;" : "+f"(m) : "f"(a));
      asm("max.NaN.f32 %0, %0, %1;" : "+f"(m) : "f"(b));
      asm("max.NaN.f32 %0, %0, %1;" : "+f"(m) : "f"(c));
      asm("max.NaN.f32 %0, %0, %1;" : "+f"(m) : "f"(d));
    }
    return m;
  }
};

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
// Clusters: distributed shared memory between the CTAs of one cluster
// ---------------------------------------------------------------------------

__device__ __forceinline__ int cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return static_cast<int>(r);
}
__device__ __forceinline__ int cluster_ctas() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return static_cast<int>(r);
}
// Address of shared variable `p` in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t peer(const volatile void* p, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(r) : "r"(smem_addr(const_cast<const void*>(p))), "r"(rank));
  return r;
}
// Asynchronous stores into the shared memory of a CTA of the cluster; each
// counts its bytes on an mbarrier of that CTA (complete_tx), so a receiver
// that saw the phase complete sees the data, with no fence on either side.
__device__ __forceinline__ void st_async(uint32_t addr, uint4 v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];"
               :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(bar) : "memory");
}
__device__ __forceinline__ void st_async(uint32_t addr, int v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
               :: "r"(addr), "r"(v), "r"(bar) : "memory");
}
// A plain arrival on an mbarrier of a CTA of the cluster.  No data rides on
// it: it only says that a buffer of the arriving CTA's has been read (the
// values read are already in registers) and may be written again.
__device__ __forceinline__ void mbar_arrive_peer(uint32_t addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" :: "r"(addr) : "memory");
}
// Every thread of every CTA of the cluster.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Order-preserving int view of a non-NaN float (for redux.sync max), and back.
__device__ __forceinline__ int ordered_key(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : i ^ 0x7fffffff;
}
__device__ __forceinline__ float from_ordered_key(int k) {
  return __int_as_float(k >= 0 ? k : k ^ 0x7fffffff);
}

// Wait for a phase in hardware for at most about `ns` nanoseconds (the warp
// is not scheduled meanwhile); returns whether the phase completed.
__device__ __forceinline__ bool mbar_park(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t done;
  asm volatile("{\n\t.reg .pred p;\n\t"
               "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(done) : "r"(smem_addr(bar)), "r"(parity), "r"(ns) : "memory");
  return done != 0;
}

// Barrier among `count` threads (whole warps) of the CTA on barrier `id`.
__device__ __forceinline__ void named_barrier_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(count) : "memory");
}

// Maximum that keeps NaN (PTX max.NaN).
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}


}  // namespace
}  // namespace sv
