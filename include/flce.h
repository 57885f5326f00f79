/*
 * flce.h -- C ABI of libflce.so: fused linear cross-entropy on one GB300
 * (sm_103a) GPU.
 *
 * The operation ("fused-linear-ce" model card, trl-lib: §Full signature,
 * §Metrics for free, §Algorithm):
 *
 *   lin_ij  = hidden_i . weight_j + bias_j                 (i < N, j < V)
 *   u_ij    = logit_scale * lin_ij
 *   z_ij    = softcap * tanh(u_ij / softcap)   if softcap > 0, else u_ij
 *   lse_i   = log sum_j exp(z_ij),   p_ij = exp(z_ij - lse_i)
 *   loss_i  = lse_i - z_{i,t_i}      (0 when t_i == ignore_index)
 *   loss    = sum_i loss_i / n_valid ("mean") | sum_i loss_i ("sum") | loss_i ("none")
 *   mean_token_accuracy = #{valid i : argmax_j z_ij == t_i} / n_valid
 *   entropy             = sum_{valid i} (lse_i - sum_j p_ij z_ij) / n_valid   (nats)
 *
 * and its backward (§Algorithm: the logits are recomputed and the logit
 * gradient is the softmax minus the one-hot target):
 *
 *   D_ij          = g_i (p_ij - [j == t_i]) * logit_scale * (1 - tanh^2(u_ij/softcap))
 *   grad_hidden   = D @ weight,  grad_weight = D^T @ hidden,  grad_bias = sum_i D_ij
 *
 * with g_i = grad_out/n_valid ("mean"), grad_out ("sum") or grad_out[i]
 * ("none"), and g_i = 0 on ignored rows. n_valid counts rows whose target is
 * not ignore_index. The N x V logit matrix is never stored: the forward keeps
 * per-(row, vocabulary tile) softmax statistics, the backward recomputes the
 * logits one vocabulary chunk at a time.
 *
 * Conventions shared by every entry point:
 *   - Every pointer argument except `p` is a DEVICE pointer on the current
 *     CUDA device; `p` is a host pointer read during the call only.
 *   - The caller owns all memory, including the workspace. The library never
 *     allocates or frees device memory and never synchronises the stream:
 *     every kernel is enqueued on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and the call returns before the work completes.
 *   - Tensors are dense row-major: hidden [N,H], weight [V,H], bias [V],
 *     targets int64 [N]. hidden, weight and bias share `p->dtype`.
 *   - FLCE_BF16 and FLCE_F16 need H % 8 == 0 and 16-byte aligned
 *     hidden/weight/bias pointers (tensor-memory-accelerator row pitch rule);
 *     FLCE_F32 needs 4-byte alignment. Violations return FLCE_ERR_UNSUPPORTED
 *     before any launch.
 *   - Dtypes: FLCE_BF16 and FLCE_F16 run on the tensor cores (bf16 or fp16
 *     products, fp32 accumulation). FLCE_F32 runs on the tensor cores too,
 *     each operand split into three bf16 parts that sum to it exactly and each
 *     product formed from six part products (within about 2^-23 of it), when
 *     H % 8 == 0 and the parts' workspace stays under 40 % of one fp32 N x V
 *     matrix; otherwise on fp32 FFMA kernels. Both meet the same fp32 bars.
 *   - Argument errors are detected on the host, before any launch, and
 *     return a non-OK status; flce_last_error() then describes the problem.
 *     A failed launch returns FLCE_ERR_CUDA.
 *   - Errors that only the device can see are ORed into `*err_word` (when it
 *     is non-NULL) asynchronously: FLCE_DEVERR_TARGET_RANGE for a target
 *     outside [0,V) that is not ignore_index (that row's loss is NaN and it
 *     gets no gradient), FLCE_DEVERR_TIMEOUT when a kernel's bounded wait
 *     expired (results are then invalid). The caller zeroes the word and
 *     reads it after its own synchronisation.
 *   - No C++ exception crosses this interface. Entry points are thread-safe;
 *     calls that share a workspace must be ordered on one stream.
 */
#ifndef FLCE_H
#define FLCE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum flce_status {
  FLCE_OK = 0,
  FLCE_ERR_INVALID_ARG = 1,   /* bad shape, option, or NULL required pointer */
  FLCE_ERR_UNSUPPORTED = 2,   /* valid but not supported (alignment, GPU arch) */
  FLCE_ERR_WORKSPACE = 3,     /* workspace smaller than *_workspace_size() or misaligned */
  FLCE_ERR_CUDA = 4,          /* a CUDA runtime/driver call or launch failed */
  FLCE_ERR_DEVICE_TIMEOUT = 5 /* reserved for callers that translate FLCE_DEVERR_TIMEOUT */
} flce_status;

typedef enum flce_dtype { FLCE_F32 = 0, FLCE_BF16 = 1, FLCE_F16 = 2 } flce_dtype;

typedef enum flce_reduction {
  FLCE_RED_NONE = 0,
  FLCE_RED_SUM = 1,
  FLCE_RED_MEAN = 2
} flce_reduction;

/* Bits of the device error word. */
#define FLCE_DEVERR_TARGET_RANGE 1
#define FLCE_DEVERR_TIMEOUT 2

/* Problem description (host struct, copied during the call).
 *   n, h, v            tokens, hidden size, vocabulary size (n >= 0, h >= 1, v >= 1)
 *   dtype              flce_dtype of hidden, weight and bias
 *   has_bias           0 or 1
 *   ignore_index       target value that marks an ignored row (default -100)
 *   logit_scale        multiplies the linear logits (finite)
 *   softcap            > 0 enables z = softcap*tanh(u/softcap); <= 0 disables
 *   reduction          flce_reduction
 *   grad_weight_dtype  dtype of grad_weight: FLCE_F32, or equal to dtype
 *   vocab_chunk        backward vocabulary chunk width; 0 picks the default:
 *                      equal chunks of whole 256-column tiles, at least five
 *                      of them (one per tile for a vocabulary of fewer than
 *                      five tiles), more where an N x chunk dlogits buffer
 *                      would exceed 512 MiB. The buffer is the largest
 *                      workspace item, so a smaller chunk lowers peak memory
 *                      at some cost in speed. Rounded up to a multiple of 256
 *   flags              OR of FLCE_SKIP_IGNORED_ROWS; 0 for none
 *   label_smoothing    eps in [0, 1]: cross-entropy against the target
 *                      distribution (1-eps)*onehot + eps/V, i.e.
 *                      loss_i = (1-eps)(lse_i - z_{i,t_i}) + eps(lse_i - mean_j z_ij)
 *   z_loss             lam >= 0: lam * lse_i^2 is added to each non-ignored row
 *   reserved           must be 0
 * With label smoothing and z-loss the logit gradient is
 *   g_i (p_ij (1 + 2 lam lse_i) - (1-eps)[j == t_i] - eps/V).
 * Both options are named in the CuTe-DSL FLCE pull request's feature list
 * (Liger-Kernel #1287, Summary); the forms above are the plain readings.
 */
typedef struct flce_problem {
  int64_t n, h, v;
  int32_t dtype;
  int32_t has_bias;
  int64_t ignore_index;
  float logit_scale;
  float softcap;
  int32_t reduction;
  int32_t grad_weight_dtype;
  int64_t vocab_chunk;
  int32_t flags;
  float label_smoothing;
  float z_loss;
  int32_t reserved;
} flce_problem;

/* Leave rows whose target is ignore_index out of every contraction (bf16 and
 * fp16 paths; the fp32 path computes every row either way). The non-ignored rows are
 * gathered, in their original order, into the workspace, and the GEMMs run
 * over them alone: ignored rows contribute nothing to the loss or to any
 * gradient, so their logits are never needed. Loss, metrics and gradients are
 * unchanged; loss_rows and correct_rows of ignored rows are 0 as without the
 * flag, but lse_rows and entropy_rows of ignored rows are not computed (NaN).
 * Grad_hidden rows of ignored rows are written as 0. */
#define FLCE_SKIP_IGNORED_ROWS 1

/* Bytes of device workspace flce_forward() needs for `p` (0 if `p` is
 * invalid). Following §Algorithm (the vocabulary is swept in tiles, each
 * folded into a running log-sum-exp), the workspace holds the per-(row,
 * vocabulary tile) statistics that the merge combines: about
 * N * ceil(V/256) * 16 bytes (20 with label smoothing). */
size_t flce_forward_workspace_size(const flce_problem* p);

/* Forward pass. Cite: §Algorithm (forward), §Metrics for free.
 *   hidden [N,H], weight [V,H], bias [V] (NULL unless p->has_bias), targets [N]
 *   loss_rows    [N] fp32 out: per-row loss (0 on ignored rows)       required
 *   lse_rows     [N] fp32 out: per-row log-sum-exp, kept for backward required
 *   correct_rows [N] int32 out: 1 where argmax == target (valid rows) nullable
 *   entropy_rows [N] fp32 out: per-row softmax entropy in nats       nullable
 *   loss_out     scalar fp32 out: the reduced loss; required for "sum" and
 *                "mean", ignored (may be NULL) for "none"
 *   metrics_out  [2] fp32 out: {mean_token_accuracy, entropy}; NULL skips
 *                them. Loss outputs are bit-identical either way.
 *   n_valid      scalar int32 out: rows whose target != ignore_index  required
 *   err_word     scalar int32, ORed with FLCE_DEVERR_* bits           nullable
 *   workspace    >= flce_forward_workspace_size(p) bytes, 256-byte aligned
 * With n_valid = 0, "mean" gives NaN loss and NaN metrics. */
flce_status flce_forward(const flce_problem* p, const void* hidden,
                         const void* weight, const void* bias,
                         const int64_t* targets, float* loss_rows,
                         float* lse_rows, int32_t* correct_rows,
                         float* entropy_rows, float* loss_out,
                         float* metrics_out, int32_t* n_valid,
                         int32_t* err_word, void* workspace,
                         size_t workspace_bytes, void* stream);

/* Forward pass that allocates nothing and takes no workspace. The method's
 * pages have no counterpart to it; it exists for callers that cannot call
 * cudaMalloc and have no workspace to hand in: for example a host framework
 * whose memory pool owns the whole device and refuses allocations from
 * libraries, or a latency-bound loop where a cudaMalloc (which may
 * synchronise the device) is not allowed.
 *   Arguments and outputs are those of flce_forward() without `workspace`
 *   and `workspace_bytes`; results are the same as flce_forward's.
 *   Scratch: a fixed 16 MiB array inside the library, held by every GPU that
 *   loads the library until the process exits. A problem is accepted when
 *   flce_forward_workspace_size(p) <= 16 MiB, and otherwise rejected with
 *   FLCE_ERR_UNSUPPORTED before any launch. For bf16 at H = 4096,
 *   V = 128256 that is N <= 2089 tokens; with FLCE_SKIP_IGNORED_ROWS, whose
 *   gathered copy of the kept hidden rows adds N * H * 2 bytes, N <= 1033
 *   (N <= 919 with label smoothing as well).
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current, and so does the first
 *   call after the device's context was destroyed and re-created (for
 *   example by cudaDeviceReset); make that first call before any stream
 *   capture.
 *   All calls share the one array, which keeps the last call's contents:
 *   calls whose work overlaps on the GPU (for example on two streams without
 *   ordering between them) race and corrupt each other's results. Order them
 *   on one stream. */
flce_status flce_forward_noalloc(const flce_problem* p, const void* hidden,
                                 const void* weight, const void* bias,
                                 const int64_t* targets, float* loss_rows,
                                 float* lse_rows, int32_t* correct_rows,
                                 float* entropy_rows, float* loss_out,
                                 float* metrics_out, int32_t* n_valid,
                                 int32_t* err_word, void* stream);

/* Bytes of device workspace flce_backward() needs for `p` (0 if invalid):
 * the dlogits buffer of one vocabulary chunk (N x chunk, in the input type for
 * FLCE_BF16 / FLCE_F16; fp32 for FLCE_F32 on FFMA kernels, or three bf16 parts
 * on the tensor cores, which also hold the bf16 parts of hidden and of the
 * chunk's weight rows), an fp32 [N,H] grad_hidden accumulator when there is
 * more than one chunk on the tensor-core path, and fp32 grad_bias partial sums
 * when has_bias. */
size_t flce_backward_workspace_size(const flce_problem* p);

/* Backward pass: all three gradients. Cite: §Algorithm (backward: recompute
 * each logit tile, form p - onehot, grad_hidden = (p - onehot) @ weight,
 * grad_weight = (p - onehot)^T @ hidden); §Full signature ("hidden, weight
 * and bias all receive gradients").
 *   hidden, weight, bias, targets   as for flce_forward (same values)
 *   lse_rows    [N] fp32 in: from flce_forward on the same inputs   required
 *   n_valid     scalar int32 in: from flce_forward                   required
 *   grad_out    fp32 in: scalar d(objective)/d(loss) for "sum"/"mean",
 *               [N] per-row upstream gradients for "none"            required
 *   grad_hidden [N,H] out, dtype p->dtype                            required
 *   grad_weight [V,H] out, dtype p->grad_weight_dtype                required
 *   grad_bias   [V] out, dtype p->dtype; required iff p->has_bias
 *   err_word    as for flce_forward                                  nullable
 *   workspace   >= flce_backward_workspace_size(p) bytes, 256-byte aligned
 * Outputs are overwritten, not accumulated into. */
flce_status flce_backward(const flce_problem* p, const void* hidden,
                          const void* weight, const void* bias,
                          const int64_t* targets, const float* lse_rows,
                          const int32_t* n_valid, const float* grad_out,
                          void* grad_hidden, void* grad_weight,
                          void* grad_bias, int32_t* err_word, void* workspace,
                          size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Fused linear KL divergence (FusedLinearKLDivLoss pull request, Liger-Kernel
 * #1423, Summary and Details): the vocabulary projection followed by
 * KL(Q || P) against an explicit target distribution Q (teacher
 * probabilities), without materialising the N x V logits:
 *
 *   z_ij   = (hidden_i . weight_j + bias_j) / temperature
 *   loss_i = sum_j q_ij (log max(q_ij, eps) - (z_ij - lse_i))     (counted rows)
 *          = sum_j q_ij (log max(q_ij, eps) - z_ij) + lse_i * sum_j q_ij
 *   D_ij   = g_i (p_ij * sum_k q_ik - q_ij) / temperature          (d loss / d lin)
 *
 * Rows whose label equals ignore_index are not counted (labels may be NULL:
 * every row counts). Reductions follow torch.nn.KLDivLoss: batchmean divides
 * the sum by the counted rows, mean by counted rows * V; none returns the
 * per-row losses and takes per-row upstream gradients. The same kernels as
 * the cross-entropy run underneath; conventions are those of flce_forward /
 * flce_backward above.
 */
typedef enum flce_kl_reduction {
  FLCE_KL_NONE = 0,
  FLCE_KL_SUM = 1,
  FLCE_KL_BATCHMEAN = 2,
  FLCE_KL_MEAN = 3
} flce_kl_reduction;

/*   n, h, v, dtype, has_bias, grad_weight_dtype, vocab_chunk, flags
 *                      as in flce_problem (target_probs has the input dtype)
 *   ignore_index       label value of rows left out (used only with labels)
 *   temperature        > 0: the student logits are divided by it
 *   eps                > 0: clamp inside log q (so that 0 * log 0 adds 0)
 *   reduction          flce_kl_reduction
 *   reserved           must be 0 */
typedef struct flce_kl_problem {
  int64_t n, h, v;
  int32_t dtype;
  int32_t has_bias;
  int64_t ignore_index;
  float temperature;
  float eps;
  int32_t reduction;
  int32_t grad_weight_dtype;
  int64_t vocab_chunk;
  int32_t flags;
  int32_t reserved;
} flce_kl_problem;

/* Bytes of device workspace flce_kl_forward() needs (0 if `p` is invalid). */
size_t flce_kl_forward_workspace_size(const flce_kl_problem* p);

/* KL forward. target_probs [N,V] (input dtype), labels [N] int64 (nullable).
 *   loss_rows [N] fp32 out (0 on uncounted rows)                     required
 *   lse_rows  [N] fp32 out: log-sum-exp of z, kept for the backward   required
 *   qsum_rows [N] fp32 out: sum_j q_ij, kept for the backward         required
 *   loss_out  scalar fp32 out (not written for FLCE_KL_NONE)
 *   n_counted scalar int32 out: rows counted                          required
 * With FLCE_SKIP_IGNORED_ROWS and labels, uncounted rows are left out of
 * the contractions (their lse and qsum are then NaN). */
flce_status flce_kl_forward(const flce_kl_problem* p, const void* hidden,
                            const void* weight, const void* bias,
                            const void* target_probs, const int64_t* labels,
                            float* loss_rows, float* lse_rows, float* qsum_rows,
                            float* loss_out, int32_t* n_counted,
                            int32_t* err_word, void* workspace,
                            size_t workspace_bytes, void* stream);

/* Bytes of device workspace flce_kl_backward() needs (0 if `p` is invalid). */
size_t flce_kl_backward_workspace_size(const flce_kl_problem* p);

/* KL backward: grad_hidden, grad_weight, grad_bias as in flce_backward, from
 * the forward's lse_rows, qsum_rows and n_counted; grad_out is a scalar, or
 * [N] for FLCE_KL_NONE. */
flce_status flce_kl_backward(const flce_kl_problem* p, const void* hidden,
                             const void* weight, const void* bias,
                             const void* target_probs, const int64_t* labels,
                             const float* lse_rows, const float* qsum_rows,
                             const int32_t* n_counted, const float* grad_out,
                             void* grad_hidden, void* grad_weight,
                             void* grad_bias, int32_t* err_word,
                             void* workspace, size_t workspace_bytes,
                             void* stream);

/* ------------------------------------------------------------------------
 * Self-test of the bounded waits (not part of the method; the pages describe
 * no such check). Every pipeline wait of the kernels gives up after a time
 * budget, records FLCE_DEVERR_TIMEOUT in the error word and returns instead
 * of spinning forever. This call exercises exactly those wait routines on an
 * mbarrier that nothing arrives on, with a budget of budget_s seconds
 * (0 < budget_s <= 1): once in a single CTA and once in a pair of CTAs (the
 * cluster-scope wait). On completion of the stream's work, *err_word has
 * FLCE_DEVERR_TIMEOUT set and result[0..2] (int32, device) are 0: each wait
 * gave up. Nothing faults; the context stays usable.
 *   err_word  int32 device scalar, ORed into (not cleared)
 *   result    int32 device [3]                                           */
flce_status flce_selftest_wait_timeout(int32_t* err_word, int32_t* result,
                                       double budget_s, void* stream);

/* ------------------------------------------------------------------------
 * Per-kernel timing, for measurement tools (not part of the method; the
 * pages describe no profiler). While enabled, every kernel launch made by
 * flce_forward / flce_backward on the calling process is bracketed by two
 * CUDA events recorded on the caller's stream, so the launch sequence and
 * its stream ordering are unchanged. Up to FLCE_PROFILE_MAX_RECORDS launches
 * are recorded; later ones are counted in `dropped`. The events are created
 * on the current device the first time profiling is enabled.
 */
#define FLCE_PROFILE_MAX_RECORDS 8192
#define FLCE_PROFILE_NAME_LEN 40

typedef struct flce_kernel_time {
  char name[FLCE_PROFILE_NAME_LEN]; /* kernel role, e.g. "fwd_stats" */
  int32_t launches;                 /* launches recorded since the last collect */
  double total_ms;                  /* summed event-to-event time of those launches */
} flce_kernel_time;

/* Turn recording on (1) or off (0). Enabling clears earlier records. */
flce_status flce_profile_enable(int enable);

/* Synchronise on the recorded events, write up to `max_entries` per-kernel
 * totals (one entry per kernel role, in first-launch order) and clear the
 * record. Returns the number of entries written, or -1 on a CUDA error.
 * `*dropped` (nullable) receives the launches not recorded. */
int flce_profile_collect(flce_kernel_time* out, int max_entries, int32_t* dropped);

/* Static text for a status code. */
const char* flce_status_string(flce_status s);

/* Description of the last non-OK status returned on the calling thread
 * (empty string if none). Valid until the next call on that thread. */
const char* flce_last_error(void);

/* 1 if the current CUDA device can run this library's kernels (compute
 * capability 10.3, i.e. sm_103a), else 0. */
int flce_device_supported(void);

#ifdef __cplusplus
}
#endif

#endif /* FLCE_H */
