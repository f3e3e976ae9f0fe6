// Internal declarations shared by the verification kernels and the C ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

namespace sv {

// A named NVTX range over the host code that enqueues a kernel (header-only
// NVTX v3: a no-op unless a profiler is attached), so that a timeline or an
// ncu --nvtx filter can tell the library's launches apart.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

constexpr int kConsumerWarps = 16;                      // warps that compute
constexpr int kWalkers = 2;                             // walker warps (walks of different sequences overlap)
constexpr int kThreads = (kConsumerWarps + 2 + kWalkers) * 32;   // + producer, control and walker warps
constexpr int kVecsPerLane = 8;                         // 16-byte vectors per lane and chunk
constexpr int kVecsPerWarp = kVecsPerLane * 32;         // 256 x 16 B per warp and chunk
constexpr int kChunkBytes = kVecsPerWarp * 16 * kConsumerWarps;  // one staging slot: 64 KB
constexpr int kMaxChunks = 16;                          // rows up to 1 MiB
constexpr int kMaxStages = 16;                          // staging slots per CTA
constexpr long long kDrainLimitNs = 1000000000LL;       // second wait: always 1 s
constexpr int kMaxCluster = 8;                          // CTAs sharing one sequence (portable limit)
// Timeline slots per CTA: 0 grid wait done, 1 first chunk, 2 last chunk,
// 3 control warp done, 4 walker done, 5 CTA end, 6 chunks consumed,
// 7 prologue start.
constexpr int kTimelineSlots = 8;

// Counters kept on the device (unsigned long long each).
enum StatSlot {
  kStatSequences = 0,   // sequences finalised without error
  kStatProposed,        // sum k_b
  kStatAccepted,        // sum a_b
  kStatEmitted,         // sum (a_b + 1)
  kStatSpecOff,         // k_b == 0
  kStatZeroResidual,    // residual mass exactly zero
  kStatErrorSeqs,       // sequences that emitted nothing because of an error
  kStatRowsSkipped,     // early exit: needed rows not read
  kStatCount
};

// Workspace owned by the context.
struct Workspace {
  int2* seqs;       // [max_B]   work list {b, k_b}, longest first
  int* n_seqs;      // [1]       entries in the work list
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

// Workspace of the row-streaming schedule (sv_pieces.cu), owned by the
// context.  A sequence's rows are target 0, draft 0, ..., target k_b; a
// piece is 64 KB of one row (np per row), a re-read half-piece 16 KB of each
// row of a pair (nr per row).
struct PiecesWs {
  float4* rec;       // [max_B * (2 max_k + 1) * np]  a piece's (M, S about fl(M c), token logit, flags), at
                     //   ((b (2k + 1) + row of the sequence) np + piece); greedy (M, argmax, 0, flags)
  float2* bseg;      // [max_B * np * 16]  bonus rows: each warp segment's (fl(m c), sum)
  int4* job;         // [max_B]       a rejected pair to draw from: (sampling uniform's bits, b, a, k_b)
  float4* jobn;      // [max_B]       ... its (K_t, L_t, Gh, Gl)
  int* njobs;        // [1]
  float4* bonus;     // [max_B]       a fully accepted sequence's bonus row: (call number's bits, K, L, s)
  int* epoch;        // [1]           the call number (counted by each call's statistics kernel)
  float* rmass;      // [max_B * nr * 16]  per job, each re-read segment's sum of max(0, p - q)
  float* pmass;      // [max_B * nr * 16]  ... and of p (zero-residual fallback)
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
  int stages;           // staging slots per CTA (2..kMaxStages)
  int bulk;             // 1: rows staged with cp.async.bulk; 0: plain loads
  int cluster;          // CTAs per cluster: each takes one slice of every row (1, 2, 4 or 8)
  int early_exit;       // 1: rows after a decided rejection are not read
  int diag;             // 1: per-row diagnostics (row maxima, log-sums, alpha, draw masses) are written
  long long wait_limit_ns;
  Workspace ws;
  // optional per-CTA timestamps (global timer, ns) of the cluster kernel,
  // kTimelineSlots per CTA and, after the last CTA's, the plan kernel's
  // start and end: null when not asked for
  unsigned long long* timeline;
  // row streaming (sv_pieces.cu) instead of the cluster kernel when set
  int pieces;
  int np;               // 64 KB pieces per row
  int nr;               // 16 KB half-pieces per row (re-reads)
  int ctas;             // grid of the streaming kernels (one CTA per SM)
  PiecesWs pw;
};

// Launchers (sv_kernels.cu).
cudaError_t launch_verify(const VerifyParams& p, int ctas, int smem_bytes, cudaStream_t s);
cudaError_t prepare_verify_kernel(int smem_bytes);
cudaError_t query_ctas_per_sm(int smem_bytes, int* out);
cudaError_t query_max_clusters(int cluster, int smem_bytes, int* out);
cudaError_t launch_compact(int B, int k, const int* out_tokens, const int* out_len,
                           int* packed, int* offsets, cudaStream_t s);
cudaError_t launch_debug(const Workspace& ws, int B, int k, int greedy, float inv_T, double* lse_t,
                         double* lse_d, double* accept_prob, double* mass, cudaStream_t s);
cudaError_t launch_init_workspace(const Workspace& ws, cudaStream_t s);

// Shared-memory bytes of the verify kernel with `stages` staging slots.
int verify_smem_bytes(int stages);

// The row-streaming schedule (sv_pieces.cu).
constexpr int kPiecesMaxB = 2048;                         // sequences per call
int pieces_smem_bytes();
int pieces_threads();                                       // threads of the streaming kernels
cudaError_t prepare_pieces_kernel();
cudaError_t launch_pieces(const VerifyParams& p, cudaStream_t s);   // after plan_kernel
// 64 KB pieces and 16 KB re-read half-pieces per row of V logits of elt bytes.
constexpr int kRowsHalfBytes = kChunkBytes / 4;          // a re-read slot: this much of each row of a pair
inline void pieces_shape(int V, int elt, int& np, int& nr) {
  const long long row = static_cast<long long>(V) * elt;
  np = static_cast<int>((row + kChunkBytes - 1) / kChunkBytes);
  nr = static_cast<int>((row + kRowsHalfBytes - 1) / kRowsHalfBytes);
}

// Cluster size chosen when the caller leaves it open.  A sequence is the
// unit of work of a cluster, so with few sequences per cluster the last ones
// to finish leave most SMs idle; splitting every row over more CTAs makes the
// units smaller.  Slices stay at 32 KB or more, and a size is only taken if
// its clusters still cover nearly every SM (max_clusters[i]: clusters of
// 2^i CTAs that fit at once).
inline int auto_cluster(int B, long long row_bytes, int num_sms, const int (&max_clusters)[4]) {
  int best = 1;
  for (int i = 1, c = 2; c <= kMaxCluster; ++i, c *= 2) {
    if (static_cast<long long>(B) * c > 4LL * num_sms) break;
    if (row_bytes / c < 32 * 1024) break;
    if (max_clusters[i] * c * 10 < num_sms * 9) continue;
    best = c;
  }
  return best;
}

}  // namespace sv
