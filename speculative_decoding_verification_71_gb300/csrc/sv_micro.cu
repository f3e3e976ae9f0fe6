// Throughput of the special-function unit's base-2 exponential
// (ex2.approx.ftz.f32, the one the verify kernels call), measured on the
// device at hand.  It is the second bound of the verify path after HBM: the
// statistics pass takes one ex2 per streamed logit, the re-read of a rejected
// pair two per logit pair.  A measurement utility beside the path; no verify
// call uses it.

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <vector>

#include "specverify.h"
#include "sv_device.cuh"

namespace sv {
namespace {

constexpr int kEx2Threads = 1024;   // 32 warps: enough independent work to keep the unit busy
constexpr int kEx2Chains = 8;       // independent exponentials in flight per thread

// Each thread iterates x <- 2^x - 3/2 on kEx2Chains independent chains; the
// map sends [-1, 0] into [-1, -1/2], so every argument stays a normal number.
// The block's elapsed SM cycles (its slowest thread) go to cycles[block].
__global__ void __launch_bounds__(kEx2Threads, 1) ex2_rate_kernel(int iters, long long* cycles, float* sink) {
  __shared__ unsigned long long tmax;
  if (threadIdx.x == 0) tmax = 0;
  float x[kEx2Chains];
#pragma unroll
  for (int j = 0; j < kEx2Chains; ++j) x[j] = -0.25f - 1e-5f * static_cast<float>((threadIdx.x * 7 + j) & 1023);
  __syncthreads();
  const long long t0 = clock64();
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < kEx2Chains; ++j) x[j] = __fsub_rn(fast_exp2(x[j]), 1.5f);
  }
  const long long dt = clock64() - t0;
  atomicMax(&tmax, static_cast<unsigned long long>(dt));
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < kEx2Chains; ++j) s += x[j];
  if (s > 0.f) sink[0] = s;   // never true (every x is negative): keeps the chains live
  __syncthreads();
  if (threadIdx.x == 0) cycles[blockIdx.x] = static_cast<long long>(tmax);
}

}  // namespace
}  // namespace sv

extern "C" {

sv_status sv_measure_ex2(int iters, double* per_sm_per_clock, double* per_second) {
  if (iters <= 0 || iters > (1 << 24) || (!per_sm_per_clock && !per_second)) return SV_ERR_INVALID_ARG;
  int dev = 0;
  cudaDeviceProp prop;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return SV_ERR_CUDA;
  // one block per SM: more than half of an SM's shared memory per block
  const int grid = prop.multiProcessorCount;
  const int smem = static_cast<int>(prop.sharedMemPerMultiprocessor / 2) + 1024;
  if (smem > static_cast<int>(prop.sharedMemPerBlockOptin)) return SV_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(sv::ex2_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return SV_ERR_CUDA;
  long long* cycles = nullptr;
  float* sink = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  sv_status st = SV_OK;
  float ms = 0.f;
  std::vector<long long> host(static_cast<size_t>(grid));
  if (cudaMalloc(&cycles, sizeof(long long) * grid) != cudaSuccess || cudaMalloc(&sink, sizeof(float)) != cudaSuccess ||
      cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
    st = SV_ERR_CUDA;
  } else {
    sv::ex2_rate_kernel<<<grid, sv::kEx2Threads, smem>>>(iters, cycles, sink);   // warm-up
    cudaEventRecord(e0);
    sv::ex2_rate_kernel<<<grid, sv::kEx2Threads, smem>>>(iters, cycles, sink);
    cudaEventRecord(e1);
    if (cudaEventSynchronize(e1) != cudaSuccess || cudaGetLastError() != cudaSuccess ||
        cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess ||
        cudaMemcpy(host.data(), cycles, sizeof(long long) * grid, cudaMemcpyDeviceToHost) != cudaSuccess)
      st = SV_ERR_CUDA;
  }
  if (st == SV_OK) {
    const double ops = static_cast<double>(sv::kEx2Threads) * iters * sv::kEx2Chains;   // per block
    std::sort(host.begin(), host.end());
    const double med = static_cast<double>(host[host.size() / 2]);
    if (!(med > 0.0) || !(ms > 0.f)) {
      st = SV_ERR_CUDA;
    } else {
      if (per_sm_per_clock) *per_sm_per_clock = ops / med;
      if (per_second) *per_second = ops * grid / (static_cast<double>(ms) * 1e-3);
    }
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (cycles) cudaFree(cycles);
  if (sink) cudaFree(sink);
  return st;
}

}  // extern "C"
