// Internal declarations shared by the verification kernels and the C ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

constexpr int kThreads = 256;           // threads per CTA of the verify kernel
constexpr int kMaxCluster = 16;         // largest cluster (non-portable size)
constexpr int kMaxStages = 4;           // staging buffers per CTA
constexpr int kNoReject = 0x7fffffff;   // "no rejection seen" in rej_min
constexpr int kCtrlBytes = 2048;        // control block at the start of shared memory
constexpr long long kDrainLimitNs = 1000000000LL;  // second wait: always 1 s

// Counters kept on the device (unsigned long long each).
enum StatSlot {
  kStatSequences = 0,   // sequences finalised without error
  kStatProposed,        // sum k_b
  kStatAccepted,        // sum a_b
  kStatEmitted,         // sum (a_b + 1)
  kStatSpecOff,         // k_b == 0
  kStatZeroResidual,    // residual mass exactly zero
  kStatErrorSeqs,       // sequences that emitted nothing because of an error
  kStatCount
};

// Workspace owned by the context.  The plan kernel that starts every call
// resets the per-sequence words and the ticket counter.
struct Workspace {
  int* done;        // [max_B]   items of the sequence finished so far
  int* rej_min;     // [max_B]   smallest rejecting draft index, kNoReject if none
  int* seq_err;     // [max_B]   OR of (1 << code) for the sequence
  int* y_slot;      // [max_B * (max_k + 1)]  token drawn at each position
  int2* items;      // [max_B * (max_k + 1)]  work list: {b, (pos << 1) | is_pair}
  int* n_items;     // [1]       entries in the work list
  int* ticket;      // [1]       next work-list entry to hand out
  float* m_t;       // [max_B * (max_k + 1)]  target row maximum (debug)
  float* L_t;       // [max_B * (max_k + 1)]  log2 sum 2^(z c - fl(m c)) (debug)
  float* m_d;       // [max_B * max_k]
  float* L_d;       // [max_B * max_k]
  float* alpha;     // [max_B * max_k]        min(1, p/q) (debug)
  float* mass;      // [max_B * (max_k + 1)]  S of the draw (debug)
  unsigned long long* stats;  // [kStatCount]
  unsigned int* err_word;     // sticky OR of (1 << code)
};

struct VerifyParams {
  const void* target;   // [B, k+1, V]
  const void* draft;    // [B, k, V]
  const int* tokens;    // [B, k]
  const int* draft_len; // [B]
  const float* uniforms;// [B, k+1]
  int* out_tokens;      // [B, k+1]
  int* out_len;         // [B]
  int B, k, V;
  int elt;              // bytes per logit: 4 (fp32) or 2 (bf16)
  int greedy;           // T == 0
  float c2;             // log2(e) / T
  int slice;            // logits per CTA (multiple of 8)
  int stages;           // staging buffers per CTA (2..kMaxStages)
  int bulk;             // 1: rows staged with cp.async.bulk; 0: plain loads
  long long wait_limit_ns;
  Workspace ws;
};

// Launchers (sv_kernels.cu).
cudaError_t launch_verify(const VerifyParams& p, int cluster, int clusters, int smem_bytes, cudaStream_t s);
cudaError_t prepare_verify_kernel(int smem_bytes, int cluster);
cudaError_t query_max_active_clusters(int cluster, int smem_bytes, int* out);
cudaError_t launch_compact(int B, int k, const int* out_tokens, const int* out_len,
                           int* packed, int* offsets, cudaStream_t s);
cudaError_t launch_debug(const Workspace& ws, int B, int k, int greedy, float inv_T, double* lse_t,
                         double* lse_d, double* accept_prob, double* mass, cudaStream_t s);
cudaError_t launch_init_workspace(const Workspace& ws, int max_B, cudaStream_t s);

// Shared-memory bytes the verify kernel needs for `stages` buffers of a
// target/draft slice pair of `slice` logits each.
inline int row_bytes_padded(int slice, int elt) { return ((slice * elt + 127) / 128) * 128; }
inline int verify_smem_bytes(int slice, int elt, int stages) {
  return kCtrlBytes + stages * 2 * row_bytes_padded(slice, elt);
}

}  // namespace sv
