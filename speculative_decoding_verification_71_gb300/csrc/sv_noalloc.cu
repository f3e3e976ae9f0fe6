// spec_verify_noalloc: the verification without a context, for callers that
// may not allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they verify: code
// that runs under an allocator it does not own (a framework's caching
// allocator that must see every byte), code that must not synchronise the
// device (cudaMalloc/cudaFree can), or code with a fixed memory budget decided
// before it starts.  For them the workspace that sv_create would allocate
// lives here instead, in one fixed-size array in the library's device memory.
// The caller still passes every input and output buffer.
//
// The array is shared by every call on a device and keeps the last call's
// contents; the parts that must start from zero are cleared at the start of
// each call.  Calls that overlap on the GPU (different streams, or no
// ordering between them) race on it and must not be issued.

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/specverify.h"
#include "sv_internal.h"

namespace {

// Largest batch the array holds: B <= kNoAllocMaxB sequences and
// B * (k + 1) <= kNoAllocMaxRows rows.
constexpr int kNoAllocMaxB = 4096;
constexpr int kNoAllocMaxRows = 16384;

constexpr size_t align256(size_t x) { return (x + 255) / 256 * 256; }
constexpr size_t kOffSeqs = 0;
constexpr size_t kOffNSeqs = kOffSeqs + align256(sizeof(int2) * kNoAllocMaxB);
constexpr size_t kOffTicket = kOffNSeqs + 256;
constexpr size_t kOffStats = kOffTicket + 256;
constexpr size_t kOffErr = kOffStats + align256(sizeof(unsigned long long) * sv::kStatCount);
constexpr size_t kOffRows = kOffErr + 256;                      // six float arrays of kNoAllocMaxRows
constexpr size_t kRowArray = align256(sizeof(float) * kNoAllocMaxRows);
constexpr size_t kScratchBytes = kOffRows + 6 * kRowArray;      // about 420 KB

// The workspace of spec_verify_noalloc: every GPU that loads the library
// holds one copy until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

struct DeviceSetup {
  bool ready = false;
  unsigned char* scratch = nullptr;   // device address of g_noalloc_scratch
  int num_sms = 0;
  int smem = 0;
  int max_clusters[4] = {0, 0, 0, 0}; // clusters of 1, 2, 4, 8 CTAs that fit at once
};

std::mutex g_setup_mutex;
DeviceSetup g_setup[kMaxDevices];

// Once per device, with that device current: the array's device address and
// the launch shape (three 64 KB staging slots, one CTA per SM, the cluster
// size chosen per call as for a context).
sv_status setup_device(int dev, DeviceSetup** out) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  DeviceSetup& s = g_setup[dev];
  if (!s.ready) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return SV_ERR_CUDA;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return SV_ERR_CUDA;
    if (!(prop.major == 10 && prop.minor == 3)) return SV_ERR_UNSUPPORTED;
    const int smem = sv::verify_smem_bytes(3);
    if (smem > static_cast<int>(prop.sharedMemPerBlockOptin)) return SV_ERR_UNSUPPORTED;
    if (sv::prepare_verify_kernel(smem) != cudaSuccess) return SV_ERR_CUDA;
    int fit = 0;
    if (sv::query_ctas_per_sm(smem, &fit) != cudaSuccess || fit <= 0) return SV_ERR_UNSUPPORTED;
    for (int i = 0; i < 4; ++i) {
      const int c = 1 << i;
      int n = 0;
      if (sv::query_max_clusters(c, smem, &n) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
      }
      const int cap = prop.multiProcessorCount * fit / c;
      s.max_clusters[i] = n < cap ? n : cap;
    }
    if (s.max_clusters[0] <= 0) return SV_ERR_UNSUPPORTED;
    s.scratch = static_cast<unsigned char*>(ptr);
    s.num_sms = prop.multiProcessorCount;
    s.smem = smem;
    s.ready = true;
  }
  *out = &s;
  return SV_OK;
}

}  // namespace

extern "C" sv_status spec_verify_noalloc(int B, int k, int V, sv_dtype dtype,
                                         const void* target_logits, const void* draft_logits,
                                         const int32_t* draft_tokens, const int32_t* draft_len,
                                         const float* uniforms, float temperature,
                                         int32_t* out_tokens, int32_t* out_len, sv_stream_t stream) {
  // sizes first: nothing beyond the array's capacity is accepted
  if (B < 1 || B > kNoAllocMaxB || k < 0 || k > 31 || V <= 0) return SV_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * (k + 1) > kNoAllocMaxRows) return SV_ERR_INVALID_ARG;
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  const int elt = dtype == SV_F32 ? 4 : 2;
  if (static_cast<long long>(V) * elt > static_cast<long long>(sv::kMaxChunks) * sv::kChunkBytes)
    return SV_ERR_INVALID_ARG;
  if (!(temperature >= 0.f) || !std::isfinite(temperature)) return SV_ERR_INVALID_ARG;
  const bool greedy = temperature == 0.f;
  const double c2 = greedy ? 0.0 : 1.4426950408889634 / static_cast<double>(temperature);
  if (!greedy && !(c2 < 1e30)) return SV_ERR_INVALID_ARG;
  if (!target_logits || !draft_len || !out_tokens || !out_len) return SV_ERR_INVALID_ARG;
  if (k > 0 && !draft_tokens) return SV_ERR_INVALID_ARG;
  if (k > 0 && !greedy && !draft_logits) return SV_ERR_INVALID_ARG;
  if (!greedy && !uniforms) return SV_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SV_ERR_UNSUPPORTED;
  DeviceSetup* setup = nullptr;
  const sv_status st = setup_device(dev, &setup);
  if (st != SV_OK) return st;

  unsigned char* base = setup->scratch;
  sv::Workspace ws;
  ws.seqs = reinterpret_cast<int2*>(base + kOffSeqs);
  ws.n_seqs = reinterpret_cast<int*>(base + kOffNSeqs);
  ws.ticket = reinterpret_cast<int*>(base + kOffTicket);
  ws.stats = reinterpret_cast<unsigned long long*>(base + kOffStats);
  ws.err_word = reinterpret_cast<unsigned int*>(base + kOffErr);
  ws.m_t = reinterpret_cast<float*>(base + kOffRows + 0 * kRowArray);
  ws.L_t = reinterpret_cast<float*>(base + kOffRows + 1 * kRowArray);
  ws.mass = reinterpret_cast<float*>(base + kOffRows + 2 * kRowArray);
  ws.m_d = reinterpret_cast<float*>(base + kOffRows + 3 * kRowArray);
  ws.L_d = reinterpret_cast<float*>(base + kOffRows + 4 * kRowArray);
  ws.alpha = reinterpret_cast<float*>(base + kOffRows + 5 * kRowArray);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the counters and the error word must start from zero (the work list and
  // the ticket are rebuilt by the first kernel of the call)
  if (cudaMemsetAsync(base + kOffStats, 0, kOffRows - kOffStats, s) != cudaSuccess) return SV_ERR_CUDA;
  // the staging shape may have been lowered for this function by a context
  if (sv::prepare_verify_kernel(setup->smem) != cudaSuccess) return SV_ERR_CUDA;

  sv::VerifyParams p{};
  p.target = target_logits;
  p.draft = draft_logits;
  p.tokens = draft_tokens;
  p.draft_len = draft_len;
  p.uniforms = uniforms;
  p.out_tokens = out_tokens;
  p.out_len = out_len;
  p.B = B;
  p.k = k;
  p.V = V;
  p.elt = elt;
  p.greedy = greedy ? 1 : 0;
  p.c2 = static_cast<float>(c2);
  p.stages = 3;
  const bool aligned = (reinterpret_cast<uintptr_t>(target_logits) & 15u) == 0 &&
                       (draft_logits == nullptr || (reinterpret_cast<uintptr_t>(draft_logits) & 15u) == 0);
  p.bulk = ((static_cast<long long>(V) * elt) % 16 == 0) && aligned;
  p.wait_limit_ns = sv::kDrainLimitNs;
  p.ws = ws;
  p.cluster = sv::auto_cluster(B, static_cast<long long>(V) * elt, setup->num_sms, setup->max_clusters);
  const int fit = setup->max_clusters[__builtin_ctz(static_cast<unsigned>(p.cluster))];
  const int ctas = (B < fit ? B : fit) * p.cluster;
  return sv::launch_verify(p, ctas, setup->smem, s) == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
