/*
 * specverify: lossless speculative-sampling verification on one GPU (sm_103a).
 *
 * The operation.  A drafter proposes k tokens per sequence; the target model
 * scores them in one forward pass; the verifier accepts or rejects the drafts
 * from the target's probability distribution so that the rollout keeps the
 * target policy's output distribution exactly ("Accelerating RL Post-Training
 * Rollouts via System-Integrated Speculative Decoding", §2 core mechanism:
 * drafting, verification in one forward pass, rejection sampling).  The
 * verifier checks all drafts together and rewrites from the first wrong token
 * ("Online Draft Co-Training for Speculative Decoding in Large-Scale,
 * Long-Context RL Post-Training", the stenographer/proof-reader analogy).
 * The pages do not write the rule down; this library implements the standard
 * speculative-sampling rule, which is the reading their exactness claim needs:
 *
 *   p_i = softmax(z^t_i / T),  q_i = softmax(z^d_i / T)
 *   draft i is accepted iff u_i < min(1, p_i(x_i) / q_i(x_i));
 *   the first rejection a ends the round;
 *   if a < k_b the token at a is drawn from max(0, p_a - q_a) (normalised),
 *   else a bonus token is drawn from p_{k_b};
 *   draws are inverse CDF in ascending token id with the sequence's one
 *   sampling uniform s_b = u_{b,k}: y = min{x : s_b * S < C(x)}.
 *
 * Per-sequence draft lengths k_b in [0, k] are allowed; k_b = 0 turns
 * speculation off for that sequence, which then emits one token sampled from
 * p_0 ("EfficientRollout: System-Aware Self-Speculative Decoding for RL
 * Rollouts", abstract: system-aware SD toggle policy).  T == 0 is greedy:
 * a draft is accepted iff it is the first argmax of p_i, and the emitted
 * token is the first argmax of the decided target row.
 *
 * Memory.  Every tensor argument is caller-owned DEVICE memory, row-major and
 * contiguous.  The context owns a fixed workspace allocated by sv_create;
 * spec_verify itself allocates nothing.  One context serves one stream at a
 * time and is not thread-safe.
 *
 * Errors.  Problems visible on the host (NULL pointers, sizes beyond the
 * context's limits, a bad temperature) return an error code synchronously and
 * launch nothing.  Problems found on the device (a draft length outside
 * [0,k], a drafted token outside [0,V), NaN or +inf in a row that is read, a
 * read row that is all -inf) mark only the affected sequence: it emits
 * nothing (out_len 0, tokens -1), and the code's bit is set in a sticky
 * device error word that spec_verify_stats returns.
 *
 * Determinism.  The library draws no random numbers: all randomness comes
 * from `uniforms`.  Reductions run in a fixed order, so repeated calls on the
 * same inputs give bitwise identical outputs.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *sv_stream_t;

typedef enum {
    SV_OK = 0,
    SV_ERR_INVALID_ARG = 1,   /* host-side argument check failed; nothing launched */
    SV_ERR_BAD_DRAFT_LEN = 2, /* device: some draft_len[b] outside [0, k] */
    SV_ERR_BAD_TOKEN = 3,     /* device: some drafted token outside [0, V) */
    SV_ERR_NONFINITE = 4,     /* device: NaN/+inf in a read row, or a read row all -inf */
    SV_ERR_TIMEOUT = 5,       /* device: a bounded wait for staged logits expired */
    SV_ERR_CUDA = 6,          /* a CUDA runtime call failed (see sv_last_cuda_error) */
    SV_ERR_UNSUPPORTED = 7    /* the device or configuration is not supported */
} sv_status;

typedef enum { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;

typedef struct sv_ctx sv_ctx;

/* Running counters since the last reset (spec_verify_stats).  The pages track
 * accepted length ("Accelerating RL Post-Training Rollouts ...", §4 draft
 * initialisation; "ReSpec", GAP 2 / Fig. 4) without defining it, so both
 * readings are reported: mean_accepted = sum a_b / sequences (accepted
 * drafts) and mean_emitted = sum (a_b + 1) / sequences (tokens emitted per
 * round, the usual "tau"). */
typedef struct {
    double mean_emitted;       /* sum(a_b + 1) / sequences */
    double mean_accepted;      /* sum(a_b) / sequences */
    double accept_rate;        /* drafts_accepted / drafts_proposed (0 if none) */
    long long calls;           /* spec_verify calls counted */
    long long sequences;       /* sequences verified without a device error */
    long long drafts_proposed; /* sum k_b */
    long long drafts_accepted; /* sum a_b */
    long long emitted;         /* sum (a_b + 1) */
    long long spec_off;        /* sequences with k_b == 0 */
    long long zero_residual;   /* rejections whose residual mass was exactly 0 */
    long long error_sequences; /* sequences that emitted nothing because of a device error */
    unsigned int error_bits;   /* OR of (1 << code) over device errors seen */
    long long rows_skipped;    /* early exit: needed logit rows not read (each row once) */
} sv_stats;

/* Human-readable name of a status code (static string). */
const char *sv_status_string(sv_status s);

/* Message of the last CUDA error seen by this context ("" if none).
 * ctx may be NULL for errors raised by sv_create. */
const char *sv_last_cuda_error(const sv_ctx *ctx);

/* Create a context for batches of up to max_B sequences, up to max_k drafts
 * each, vocabulary V and logit dtype `dtype`, on the current CUDA device.
 * Allocates the fixed device workspace (O(max_B * (max_k + 1)) words) and
 * chooses the launch configuration.  *ctx receives the handle.
 * Limits: max_k <= 31; V * sizeof(dtype) <= 1 MiB.
 * Errors: SV_ERR_INVALID_ARG (sizes <= 0 or too large, NULL ctx),
 * SV_ERR_UNSUPPORTED (no sm_100-family device), SV_ERR_CUDA. */
sv_status sv_create(sv_ctx **ctx, int max_B, int max_k, int V, sv_dtype dtype);

/* Release the context and its workspace.  NULL is accepted. */
sv_status sv_destroy(sv_ctx *ctx);

/*
 * Verify one round of drafts for B sequences (asynchronous on `stream`).
 *
 *   target_logits  [B, k+1, V] dtype   target rows; row (b, i) scores position
 *                                      i; row (b, k_b) is the bonus row.  Rows
 *                                      i > k_b are never read.
 *   draft_logits   [B, k, V]   dtype   drafter rows q; rows i >= k_b are never
 *                                      read.  May be NULL when k == 0 or T == 0.
 *   draft_tokens   [B, k]      int32   x_{b,i}; entries i >= k_b are ignored.
 *   draft_len      [B]         int32   k_b in [0, k].
 *   uniforms       [B, k+1]    float   in [0,1): columns 0..k-1 are the accept
 *                                      tests, column k the sampling uniform.
 *   temperature    T >= 0, finite; T == 0 is greedy (uniforms unused).
 *   out_tokens     [B, k+1]    int32   written: accepted drafts, then the
 *                                      sampled token, then -1 padding.
 *   out_len        [B]         int32   written: a_b + 1 (0 on a device error).
 *
 * Requires 1 <= B <= max_B, 0 <= k <= max_k.  Rows are read with 16-byte
 * bulk copies when V * sizeof(dtype) is a multiple of 16 and the logit
 * pointers are 16-byte aligned, and with plain loads otherwise.
 * The inputs must be complete when the call is enqueued: under row
 * streaming the call's first kernel starts reading them (not the workspace,
 * not the outputs) while the previous kernel on the stream finishes, when
 * that kernel allows its dependents an early start (this library's last
 * kernel of a call does; kernels launched without programmatic dependent
 * launch, such as PyTorch's, never do).
 * Returns SV_OK once the work is enqueued; device-side problems are reported
 * by spec_verify_stats.
 */
sv_status spec_verify(sv_ctx *ctx, int B, int k,
                      const void *target_logits, const void *draft_logits,
                      const int32_t *draft_tokens, const int32_t *draft_len,
                      const float *uniforms, float temperature,
                      int32_t *out_tokens, int32_t *out_len,
                      sv_stream_t stream);

/*
 * Compact the outputs of a verification into one packed token list
 * (asynchronous on `stream`): offsets[b] = sum_{b' < b} out_len[b'],
 * offsets[B] = total, packed[offsets[b] + j] = out_tokens[b, j] for
 * j < out_len[b].  All pointers are device memory; packed must hold
 * B * (k+1) entries (the worst case).  Requires 1 <= B <= max_B.
 */
sv_status spec_verify_compact(sv_ctx *ctx, int B, int k,
                              const int32_t *out_tokens, const int32_t *out_len,
                              int32_t *packed, int32_t *offsets,
                              sv_stream_t stream);

/*
 * Diagnostics recording (off by default).  While on, spec_verify also writes
 * the per-row values spec_verify_debug returns (one more global store per
 * row and draw, and a reset of the arrays per call); off, those stores are
 * skipped.  on must be 0 or 1, else SV_ERR_INVALID_ARG.
 */
sv_status sv_set_diagnostics(sv_ctx *ctx, int on);

/*
 * Per-row diagnostics of the LAST spec_verify call on this context, for
 * parity checks (asynchronous on `stream`; device pointers; any may be NULL).
 * SV_ERR_INVALID_ARG unless that call ran with diagnostics on
 * (sv_set_diagnostics) and B and k match it:
 *   lse_t      [B, k+1] double  log-sum-exp of z^t_i / T for rows i <= k_b
 *   lse_d      [B, k]   double  log-sum-exp of z^d_i / T for rows i < k_b
 *   accept_prob[B, k]   double  min(1, p_i(x_i)/q_i(x_i)) for i < k_b
 *   mass       [B, k+1] double  total weight S of the draw computed at
 *                               position i (NaN where no draw was computed)
 * Entries that do not apply (padding rows, T == 0, sequences with a device
 * error) are NaN.
 */
sv_status spec_verify_debug(sv_ctx *ctx, int B, int k, double *lse_t, double *lse_d,
                            double *accept_prob, double *mass, sv_stream_t stream);

/* Synchronise `stream`, then read the running counters and the sticky device
 * error word into *out.  Returns SV_OK, or the lowest-numbered device error
 * code seen since the last reset, or SV_ERR_CUDA. */
sv_status spec_verify_stats(sv_ctx *ctx, sv_stream_t stream, sv_stats *out);

/* Clear the counters and the device error word (asynchronous on `stream`). */
sv_status spec_verify_reset_stats(sv_ctx *ctx, sv_stream_t stream);

/* Tuning and introspection.  A cluster of 1, 2, 4 or 8 CTAs verifies one
 * sequence at a time: each CTA takes an equal slice of every row's vocabulary
 * and streams it through a ring of 64 KB shared-memory slots, and the CTAs
 * combine their slices through distributed shared memory.
 * sv_set_pipeline picks the number of slots (2..16) and how many CTAs share
 * an SM (0: as many as fit); (0, 0) restores the automatic choice.
 * sv_set_cluster fixes the cluster size (1, 2, 4 or 8), or 0 (the default)
 * to choose it on every call from the batch size and the row length.  Both
 * return SV_ERR_INVALID_ARG for values outside these ranges and
 * SV_ERR_UNSUPPORTED, keeping the previous setting, when the shape cannot be
 * launched on this device.  sv_get_config reports the current shape and
 * cluster setting, and the most CTAs the persistent grid can have;
 * sv_launch_shape the cluster size and grid a call with batch B would use.
 * Any output pointer may be NULL. */
sv_status sv_set_pipeline(sv_ctx *ctx, int stages, int ctas_per_sm);
sv_status sv_set_cluster(sv_ctx *ctx, int cluster);
sv_status sv_get_config(const sv_ctx *ctx, int *stages, int *ctas_per_sm, int *threads,
                        int *smem_bytes, int *grid_ctas, int *cluster);
sv_status sv_launch_shape(const sv_ctx *ctx, int B, int *cluster, int *grid_ctas);

/* Which schedule runs a call.  Two compute the same rule with the same
 * arithmetic:
 *   SV_KERNEL_CLUSTER  the cluster kernel described above: a sequence at a
 *                      time per cluster of CTAs;
 *   SV_KERNEL_PIECES   row streaming: every needed row is cut into 64 KB
 *                      pieces spread evenly over one CTA per SM (no exchange
 *                      between CTAs); then one warp per sequence takes the
 *                      tests and the bonus draw, the rejected pairs are read
 *                      again (spread over the SMs the same way), and one warp
 *                      per rejected pair draws.  Four launches per call, per
 *                      2048 sequences (a larger batch runs as consecutive
 *                      calls of at most 2048 sequences on the stream).  It
 *                      needs 16-byte aligned rows (V * sizeof(dtype) a
 *                      multiple of 16, aligned bases), rows of at most 1 MiB,
 *                      early exit off and no fixed cluster size; a call that
 *                      does not qualify runs the cluster kernel.
 *   SV_KERNEL_AUTO     (default) row streaming where it qualifies, the
 *                      faster of the two on every measured workload; else
 *                      the cluster kernel.
 * sv_set_kernel returns SV_ERR_INVALID_ARG for another value;
 * sv_kernel_for reports the kernel a call with batch B would run on
 * 16-byte aligned rows. */
typedef enum { SV_KERNEL_AUTO = 0, SV_KERNEL_CLUSTER = 1, SV_KERNEL_PIECES = 2 } sv_kernel;
sv_status sv_set_kernel(sv_ctx *ctx, int kernel);
sv_status sv_kernel_for(const sv_ctx *ctx, int B, int *kernel);

/* Launch shape of row streaming's two streaming kernels (statistics and
 * re-read): threads per CTA, dynamic shared memory per CTA and the grid (one
 * CTA per SM); the decision and draw kernels run one warp per sequence or
 * job.  SV_ERR_UNSUPPORTED if this context cannot run row streaming (rows
 * over 1 MiB, or too little shared memory); SV_ERR_INVALID_ARG for a NULL
 * context.  Any output pointer may be NULL. */
sv_status sv_rows_shape(const sv_ctx *ctx, int *threads, int *smem_bytes, int *grid_ctas);

/* Per-CTA timeline of the cluster kernel (measurement aid, off by default;
 * calls that run row streaming write nothing).
 * timeline: device buffer of `capacity` unsigned 64-bit words, or NULL to
 * turn it off.  A call whose grid has G CTAs (sv_launch_shape) and for which
 * capacity >= (G + 1) * 8 writes, per CTA g, the global timer in ns at
 * [g*8 + 0] the end of its wait for the work list, [+1] its first chunk,
 * [+2] its last chunk (both as consumer warp 0 takes them), [+3] its control
 * warp done, [+4] its walker warp done, [+5] its end, [+6] the chunks it
 * consumed, [+7] its start; and at [G*8 + 0] and [G*8 + 1] the start and end
 * of the work-list kernel.  Calls on a smaller buffer write nothing.  The
 * buffer stays the caller's; SV_ERR_INVALID_ARG for a negative capacity or a
 * buffer with capacity 0. */
sv_status sv_set_timeline(sv_ctx *ctx, unsigned long long *timeline, int capacity);

/* Early exit (off by default): rows of a sequence after its first rejection
 * are not read once the rejection is decided.  The outputs are the same; the
 * diagnostics of the rows not read stay NaN.  With one CTA per sequence the
 * rest of a sequence is dropped as soon as its rejection is known; in a
 * cluster the decision on pair i spares the rows from pair i + E on, E fixed
 * by the row length (about 32 64 KB chunks of every CTA's slice), so that
 * every CTA skips the same rows.  Reading stops before the bonus row too.  The bytes read then fall
 * below "every needed row once": report such runs apart from that metric.
 * on: 0 or 1 (else SV_ERR_INVALID_ARG). */
sv_status sv_set_early_exit(sv_ctx *ctx, int on);

/* Reward-weighted distillation loss of the draft model and its gradient in
 * the draft logits ("ReSpec: Towards Optimizing Speculative Decoding in
 * Reinforcement Learning Systems", Online Learner, reward-weighted KD):
 *   L_b = w_b * sum_t KL(p_{b,t} || q_{b,t}),
 *   p = softmax(z^t / T) (the updated target), q = softmax(z^d / T) (draft),
 *   grad_{b,t}(x) = dL_b / dz^d_{b,t}(x) = w_b (q(x) - p(x)) / T.
 * The page weights the KL by a function of the rollout's reward without
 * fixing it: w_b = w(r_b) is computed by the caller.
 *   target_logits, draft_logits  [n_seq, t_len, V] dtype, device, contiguous
 *   weights                      [n_seq] fp32 device
 *   temperature                  > 0 (else SV_ERR_INVALID_ARG)
 *   row_kl                       [n_seq, t_len] fp32 device, out
 *   loss                         [n_seq] fp32 device, out
 *   grad                         [n_seq, t_len, V] dtype device, out (bf16:
 *                                rounded to nearest even), or NULL for the
 *                                loss alone (one read of the logits)
 * A row pair holding NaN or +inf, or a row that is all -inf, gives a NaN
 * KL, NaN gradient and NaN loss for its rollout; a masked draft logit (-inf)
 * where the target has mass gives KL = +inf.  Asynchronous on `stream`; no
 * context and no allocation per call (the first call on a device allocates
 * one word).  Deterministic: every sum is taken in a fixed order.  One CTA
 * per SM takes whole row pairs; with the gradient each pair is streamed twice,
 * the second time from L2.  Rows whose V * sizeof(dtype) is a multiple of 16
 * with 16-byte aligned bases (and gradient) are staged with bulk copies,
 * others with plain loads.  Rows of more than 1 GiB are SV_ERR_INVALID_ARG. */
sv_status spec_kd_loss(int n_seq, int t_len, int V, sv_dtype dtype, const void *target_logits,
                       const void *draft_logits, const float *weights, float temperature,
                       float *row_kl, float *loss, void *grad, sv_stream_t stream);

/* The launch shape spec_kd_loss uses for rows of V logits of `dtype` (with or
 * without the gradient): CTAs per row (always 1), 64 KB staging slots per CTA,
 * and the most CTAs of the persistent grid (the SM count).  Any output
 * pointer may be NULL. */
sv_status spec_kd_launch_shape(int V, sv_dtype dtype, int with_grad, int *cluster, int *buffers,
                               int *grid_ctas);

/* Test hook: the limit, in nanoseconds, of each bounded wait for staged logits
 * (default 1 s).  0 makes every wait report expiry, so every sequence that
 * reads a row ends with SV_ERR_TIMEOUT; the copies are still drained (with a
 * 1 s bound) before the shared memory is reused.  Negative restores the
 * default. */
sv_status sv_set_wait_limit_ns(sv_ctx *ctx, long long ns);

/* Measurement utility (no page defines it; no verify call uses it): the
 * throughput of the special-function unit's base-2 exponential on the current
 * device, the second bound of the verify path after HBM bandwidth (the
 * statistics pass takes one ex2.approx per streamed logit, the re-read of a
 * rejected pair two per logit pair).  One 1024-thread block per SM iterates
 * `iters` times (1 <= iters <= 2^24) over 8 independent exponentials per
 * thread.  Writes the exponentials per SM per SM clock (the median block,
 * from its cycle counter) and per second (the whole grid, from CUDA events),
 * either pointer may be NULL but not both.  Synchronous: it allocates and
 * frees its own scratch and runs on the legacy default stream.  Returns
 * SV_ERR_CUDA if a CUDA call fails. */
sv_status sv_measure_ex2(int iters, double *per_sm_per_clock, double *per_second);

/*
 * spec_verify without a context, for callers that may not allocate device
 * memory (the pages describe no such entry point; it is a property of this
 * library).  Code running under an allocator it does not own, code that must
 * not synchronise the device, or code with a memory budget fixed in advance
 * cannot call sv_create, which allocates its workspace with cudaMalloc.  This
 * entry point keeps that workspace in one fixed array of about 420 KB in the
 * library's own device memory (every GPU that loads the library holds a copy
 * until the process exits) and calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *
 * Arguments are those of spec_verify, with the vocabulary V and the logit
 * dtype passed directly; inputs and outputs are caller-owned device buffers
 * as there.  Limits: 1 <= B <= 4096, 0 <= k <= 31, B * (k+1) <= 16384,
 * V * sizeof(dtype) <= 1 MiB; larger requests return SV_ERR_INVALID_ARG and
 * launch nothing.  Device-side errors show in the outputs only (out_len 0,
 * tokens -1 for the affected sequences); there are no counters.
 *
 * The first call on a device sets that device up (the array's device address
 * and the launch shape); make that first call before any stream capture.
 * Every call on a device shares the array: calls that may overlap on the GPU
 * (on different streams without ordering between them) race on it and give
 * wrong results; order them on one stream.
 */
sv_status spec_verify_noalloc(int B, int k, int V, sv_dtype dtype,
                              const void *target_logits, const void *draft_logits,
                              const int32_t *draft_tokens, const int32_t *draft_len,
                              const float *uniforms, float temperature,
                              int32_t *out_tokens, int32_t *out_len,
                              sv_stream_t stream);

/* ------------------------------------------------------------------------
 * Tree verification.
 *
 * "ReSpec: Towards Optimizing Speculative Decoding in Reinforcement Learning
 * Systems" (GAP 1) describes an SD configuration by its rounds, a branching
 * factor and a draft length per round, without a rule for verifying
 * branching drafts.  The rule implemented (recursive rejection sampling, the
 * multi-candidate form of spec_verify's rule, exact when the children of a
 * node are independent draws from the drafter's q at that node):
 *   at node j (starting at the root, node 0) let r = p_j = softmax(z^t_j / T);
 *   test the children c of j in index order: accept c (token x) iff
 *     u[b, c] < min(1, r(x) / q_j(x)) (r(x) > 0 = q_j(x) accepts);
 *     after a rejection r <- max(0, r - q_j) / S with S its mass (if S = 0, r
 *     is kept);
 *   an accepted child emits its token and the walk moves to it;
 *   if every child of j is rejected, y is drawn from the last residual; at a
 *     node without children y is the bonus token drawn from p_j;
 *   the draw is the inverse CDF in ascending token id with s = u[b, 0].
 * A chain (one child per node) is exactly spec_verify.  temperature == 0:
 * accept the first child whose token is the first argmax of z^t_j; y is that
 * argmax where none is.
 *
 * Layout (device memory, caller-owned; M = max_nodes <= SV_TREE_MAX_NODES):
 *   target_logits [B, M, V]: row j = target logits after the path to node j;
 *   draft_logits  [B, M, V]: row j = the drafter's logits from which node j's
 *                 children were drawn (read only for nodes with children);
 *   parents [B, M] (0 <= parents[b, j] < j for 1 <= j < n_nodes[b]; entry 0
 *   unused), tokens [B, M] (entry 0 unused), n_nodes [B] in [1, M],
 *   uniforms [B, M] in [0, 1) (column 0 samples, column j tests child j);
 *   out_tokens, out_nodes [B, M] (-1 padded): the accepted tokens and their
 *   nodes, then y (out_nodes has no entry for y); out_len [B] = accepted + 1;
 *   status [B] (may be NULL): SV_OK, SV_ERR_BAD_DRAFT_LEN (n_nodes or a
 *   parent out of range), SV_ERR_BAD_TOKEN, SV_ERR_NONFINITE (NaN or +inf in
 *   a row the walk reads, or such a row all -inf); a sequence with an error
 *   emits nothing (out_len 0, tokens -1);
 *   alpha [B, M] (may be NULL): min(1, r(x)/q(x)) of each tested child, NaN
 *   for the others (greedy: 1 or 0).
 * Only the rows on the walk are read.  A cluster of up to 8 CTAs walks each
 * sequence (each streams a slice of every row); the size is chosen from B
 * and the SM count, and the result is deterministic for a given B.  No
 * context and no workspace: the call allocates nothing and can be captured
 * in a CUDA graph.  The first call on a device (per dtype, and for sampling
 * and greedy separately) sets the kernel's shared-memory limit and queries
 * the cluster sizes that fit: make it before any stream capture.  Not
 * thread-safe on that first call.  Host-checkable errors (sizes, dtype,
 * temperature < 0 or not finite, NULL pointers) return SV_ERR_INVALID_ARG
 * and launch nothing.  V <= 524288.  The inputs must be complete when the
 * call is enqueued: a call's walks may start while the previous kernel on
 * the stream finishes, when that kernel allows its dependents an early start
 * (a previous tree call does); the outputs are written only after that
 * kernel is complete, so consecutive calls may share output buffers.
 * ------------------------------------------------------------------------ */

#define SV_TREE_MAX_NODES 64

sv_status spec_verify_tree(int B, int max_nodes, int V, sv_dtype dtype,
                           const void *target_logits, const void *draft_logits,
                           const int32_t *parents, const int32_t *tokens, const int32_t *n_nodes,
                           const float *uniforms, float temperature,
                           int32_t *out_tokens, int32_t *out_nodes, int32_t *out_len,
                           int32_t *status, float *alpha, sv_stream_t stream);

/* ------------------------------------------------------------------------
 * Draft-length controller and speculation toggle.
 *
 * "EfficientRollout: System-Aware Self-Speculative Decoding for RL Rollouts"
 * (abstract): speculation is switched on only in the regimes where it pays
 * for the system, and the draft length follows the drafter's acceptance.
 * "ReSpec: Towards Optimizing Speculative Decoding in Reinforcement Learning
 * Systems" (Adaptive Server): a performance model profiled offline gives, per
 * batch size, the speed of each SD configuration; at run time the effective
 * batch size picks the configuration, and large batches decode without
 * speculation.  The pages give no formulas; the rule used here:
 *
 *   observe: a verified round of sequence b (draft length k_b > 0, emitted
 *     length a + 1) tested a + r drafts, r = 1 if a < k_b; the per-slot
 *     counts decay: A <- decay A + a, N <- decay N + (a + r);
 *   alpha_b = (A + prior_alpha * prior_weight) / (N + prior_weight), or
 *     prior_alpha while N + prior_weight = 0;
 *   expected tokens of a round of n drafts: E_n(alpha) = sum_{j=0..n} alpha^j;
 *   round time T(B, n): the caller's profiled table, linear in B between two
 *     profiled batch sizes, the nearest end row outside them;
 *   SV_CTRL_BATCH: n* = argmax_n sum_b E_n(alpha_b) / T(B, n) over
 *     n = 0..max_k (smallest n on ties) for every row; n* = 0 switches
 *     speculation off for the round;
 *   SV_CTRL_PER_SEQUENCE: n_b = argmax_n E_n(alpha_b) / T(B, n).
 * B is the number of rows of the choose call: the active batch size.
 *
 * State: fp64 A and N per sequence slot, on the device, owned by the
 * controller.  A decode loop runs spec_verify -> spec_ctrl_observe (its
 * draft_len and out_len) -> spec_ctrl_choose (next round's draft lengths,
 * which spec_verify accepts as they are) with no host round trip; every call
 * is stream-ordered, allocates nothing and can be captured in a CUDA graph.
 * One controller per stream; not thread-safe.
 *
 * Arrays marked "device" are caller-owned memory of the controller's device
 * (checked for NULL only, as for spec_verify).
 *
 * Errors: host-checkable errors return SV_ERR_INVALID_ARG and launch
 * nothing.  Errors found on the device set a sticky word read by
 * spec_ctrl_status: a slot id outside [0, n_slots) or named twice in one
 * observe call (SV_ERR_INVALID_ARG; the row is skipped, and choose gives it
 * draft length 0), a draft length outside [0, max_k] or an emitted length
 * outside [0, k_b + 1] (SV_ERR_BAD_DRAFT_LEN; skipped).  A row with emitted
 * length 0 (a sequence the verifier rejected) or draft length 0 carries no
 * acceptance information and is skipped without an error.
 * ------------------------------------------------------------------------ */

#define SV_CTRL_MAX_POINTS 12    /* profiled batch sizes in the round-time table */

typedef enum { SV_CTRL_BATCH = 0, SV_CTRL_PER_SEQUENCE = 1 } sv_ctrl_mode;

typedef struct sv_ctrl sv_ctrl;

/* n_slots sequence slots (1..2^24), draft lengths 0..max_k (max_k <= 31).
 * Allocates the state (zero: every slot at the prior) on the current device.
 * Defaults: decay 0.9, prior_alpha 0.5, prior_weight 2, SV_CTRL_BATCH; no
 * round-time table (spec_ctrl_choose fails until one is set). */
sv_status spec_ctrl_create(sv_ctrl **ctrl, int n_slots, int max_k);
sv_status spec_ctrl_destroy(sv_ctrl *ctrl);

/* The profiled round-time table (host memory, copied): batch_sizes
 * [n_points] strictly increasing and >= 1, round_time [n_points][max_k + 1]
 * row-major, finite and > 0, any time unit (n = 0 is a round without
 * speculation: one target step).  1 <= n_points <= SV_CTRL_MAX_POINTS.
 * Takes effect for the choose calls issued after it. */
sv_status spec_ctrl_set_cost(sv_ctrl *ctrl, int n_points, const int *batch_sizes, const double *round_time);

/* decay in (0, 1], prior_alpha in [0, 1], prior_weight >= 0 and finite. */
sv_status spec_ctrl_set_params(sv_ctrl *ctrl, double decay, double prior_alpha, double prior_weight,
                               sv_ctrl_mode mode);

/* Put slots back at the prior: seq_ids == NULL resets every slot and clears
 * the error word; otherwise the n slots of seq_ids (device [n]) are reset. */
sv_status spec_ctrl_reset(sv_ctrl *ctrl, int n, const int32_t *seq_ids, sv_stream_t stream);

/* Add one verified round of B rows (device arrays [B]: slot ids, the draft
 * lengths the round was verified with and spec_verify's out_len).
 * 0 <= B <= n_slots. */
sv_status spec_ctrl_observe(sv_ctrl *ctrl, int B, const int32_t *seq_ids, const int32_t *draft_len,
                            const int32_t *out_len, sv_stream_t stream);

/* Draft lengths of the next round for its B active rows: next_draft_len
 * (device [B]) receives n* (batch mode) or n_b (per-sequence mode); choice
 * (device, one int32, may be NULL) receives n* or the largest n_b, so
 * choice == 0 means the round runs without speculation. */
sv_status spec_ctrl_choose(sv_ctrl *ctrl, int B, const int32_t *seq_ids, int32_t *next_draft_len,
                           int32_t *choice, sv_stream_t stream);

/* The acceptance estimate alpha_b of B slots (device [B] fp64; NaN for a bad
 * id). */
sv_status spec_ctrl_alpha(sv_ctrl *ctrl, int B, const int32_t *seq_ids, double *alpha, sv_stream_t stream);

/* Synchronises the stream and returns the sticky device error: SV_OK,
 * SV_ERR_INVALID_ARG or SV_ERR_BAD_DRAFT_LEN (SV_ERR_CUDA if the copy
 * failed). */
sv_status spec_ctrl_status(sv_ctrl *ctrl, sv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
