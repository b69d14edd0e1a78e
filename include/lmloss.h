/*
 * lmloss: fused LM-head loss forward + backward over a [T, V] logit matrix,
 * for one NVIDIA GB300 GPU (sm_103a).
 *
 * One call computes, sharing one softmax pass per row:
 *   - cross-entropy in the collapse-free form NLL = softplus(lse_{j!=t} z_j - z_t)
 *       [torchtitan PR 5661 "fix softmax collapse with improved CE perf",
 *        commit message, "Numerics (TP > 1 only)"];
 *   - z-loss alpha * lse^2
 *       [xtuner PR 1963 "[FSDP][Loss] Switch gradient reduction to SUM", z-loss diff];
 *   - optional forward-KL distillation against teacher logits, and
 *   - optional GSPO sequence-level clipped aggregation over packed segments
 *       [Fast-LLM PR 552 "Fuse GSPO into the monolithic compiled loss (#507)",
 *        "Why it needed special handling" and "Approach"],
 * reduced either as a token mean or as a SUM over the caller's global
 * denominator [xtuner PR 1963, description], and writes the gradient
 * d(total)/d(logits) once, optionally over the logits in place.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE memory owned by the caller, row-major.
 *     The library never frees or retains them past the call.
 *   - Calls are asynchronous on the given stream; no entry point synchronises
 *     the device except lmloss_get_device_error and lmloss_get_timing.
 *   - Argument errors are detected on the host and returned synchronously
 *     before anything is launched.  Data errors found on the device (a target
 *     outside [0, V) that is not -100, a segment id >= num_segments, a GSPO
 *     log-ratio sum out of range, a bounded wait that expired) are recorded in
 *     the handle's device error word; the affected rows' losses and gradients
 *     are NaN.  Read the word with lmloss_get_device_error after syncing.
 *   - One handle per stream: two calls on one handle must not overlap.
 */
#ifndef LMLOSS_H
#define LMLOSS_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LMLOSS_OK = 0,
    LMLOSS_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size, ld < V, ...        */
    LMLOSS_ERR_UNSUPPORTED = 2,   /* valid but not served: a launch shape that does not fit, */
                                  /* a row too long to stage (see lmloss_forward_backward),  */
                                  /* T >= 2^30, a shard call with a teacher or policy term    */
    LMLOSS_ERR_CUDA = 3,          /* a CUDA runtime call failed                            */
    LMLOSS_ERR_BAD_TARGET = 4,    /* device: target not in [0, V) and not -100             */
    LMLOSS_ERR_BAD_SEGMENT = 5,   /* device: segment id >= num_segments                    */
    LMLOSS_ERR_RANGE = 6,         /* device: GSPO log-ratio sum beyond +-2^31              */
    LMLOSS_ERR_TIMEOUT = 7        /* device: a bounded wait on a copy expired              */
} lmloss_status;

typedef enum { LMLOSS_BF16 = 0, LMLOSS_FP32 = 1 } lmloss_dtype;

typedef enum {
    LMLOSS_REDUCE_SUM = 0,        /* every term scaled by 1 / denominator                  */
    LMLOSS_REDUCE_TOKEN_MEAN = 1  /* token terms / #active tokens, GSPO / #non-empty segs   */
} lmloss_reduction;

#define LMLOSS_IGNORE_INDEX (-100)

typedef struct lmloss_ctx* lmloss_handle;

/*
 * Arguments of one call.  Zero-initialise, then fill what is used.
 *
 * Layout: logits, teacher_logits and grad_out are [T, ld] row-major arrays of
 * `dtype` (bf16 or fp32) whose first V columns are used; all three share ld.
 * Elements must be naturally aligned, and teacher_logits / grad_out must sit at
 * the same address modulo 16 bytes as logits (true for any two buffers from
 * one allocator with the same ld).
 *
 * Row r is ACTIVE iff targets[r] != -100 and (loss_mask == NULL or
 * loss_mask[r] != 0).  Inactive rows add nothing and get an all-zero gradient
 * [torchtitan PR 5661, "Numerics": ignored labels are zeroed by the mask].
 */
typedef struct {
    const void* logits;          /* [T, ld] dtype                                          */
    int64_t T;                   /* rows (tokens), >= 0                                    */
    int64_t V;                   /* vocabulary columns, >= 1                               */
    int64_t ld;                  /* row stride in elements, >= V                           */
    int32_t dtype;               /* lmloss_dtype                                           */
    int32_t reduction;           /* lmloss_reduction                                       */
    const int64_t* targets;      /* [T] target column, or -100 to ignore the row           */
    const uint8_t* loss_mask;    /* [T] or NULL                                            */

    float ce_weight;             /* weight of the CE term (0 for pure GSPO)                */
    float z_alpha;               /* z-loss alpha; 0 disables                               */

    const void* teacher_logits;  /* [T, ld] dtype, or NULL to disable distillation         */
    float kl_weight;             /* weight of KL(q || p^tau), q = softmax(teacher / tau),   */
                                 /*     p^tau = softmax(logits / tau)                      */
    float temperature;           /* distillation temperature tau: finite and > 0 with a    */
                                 /*     teacher (ignored without one)                      */

    const int32_t* segment_ids;  /* [T] GSPO segment of each row, -1 = none; NULL disables */
    int32_t num_segments;        /* segments in this call, <= the handle's max_segments    */
    const float* advantages;     /* [num_segments] per-segment advantage A_i               */
    const float* old_logprobs;   /* [T] behaviour-policy log-prob of each target           */
    float clip_eps_low;          /* ratio clipped to [1 - clip_eps_low, 1 + clip_eps_high] */
    float clip_eps_high;

    double denominator;          /* SUM reduction: every term is divided by this (> 0)     */

    void* grad_out;              /* [T, ld] dtype; == logits writes in place; NULL = none  */
    float* loss_out;             /* [5] total, ce, z, kl, policy (GSPO or GRPO), each      */
                                 /*     after its scale                                    */
    float* logp_out;             /* optional [T]: log p_target = -NLL (0 on inactive rows) */
    float* lse_out;              /* optional [T]: logsumexp of the row (0 on inactive)     */
    float* kl_out;               /* optional [T]: per-row KL (0 on inactive / no teacher)  */
    int64_t* count_out;          /* optional [2]: active rows, non-empty GSPO segments     */
    int32_t* seg_count_out;      /* optional [num_segments]: active tokens per segment     */
    float* seg_ratio_out;        /* optional [num_segments]: s_i = exp(mean log-ratio)     */
    uint8_t* seg_flag_out;       /* optional [num_segments]: 1 iff gradient flows via s_i  */
    float* seg_loss_out;         /* optional [num_segments]: L_i before the GSPO scale     */

    const float* token_advantages; /* [T] GRPO per-token advantages, or NULL: token-level  */
                                 /* clipped surrogate -min(rho A, clamp(rho) A) with        */
                                 /* rho = exp(logp - old_logprobs), clip_eps_low/high,     */
                                 /* scaled like the CE term; exclusive with segment_ids    */
    float* entropy_out;          /* optional [T]: entropy of softmax(logits) (0 inactive)  */
} lmloss_args;

/* What the last call launched (for tuning and for benchmark bookkeeping). */
typedef struct {
    int32_t launches;            /* kernels launched by the call                           */
    int32_t path;                /* 0 fused single-read, 1 stats-only, 2 GSPO three-phase  */
    int32_t cluster;             /* CTAs per row in the fused kernel                       */
    int32_t threads;             /* threads per CTA of the main kernel                     */
    int32_t nbuf;                /* staging buffers per CTA in the fused kernel (1 or 2)   */
    int32_t grid;                /* CTAs of the main kernel                                */
    int32_t smem_bytes;          /* dynamic shared memory per CTA of the main kernel       */
    int32_t reserved;
} lmloss_call_info;

/* Create a handle on `device`: allocates the workspace for calls with up to
 * max_T rows and max_segments GSPO segments (40 B per row plus about 40 B per
 * segment) and the device error word.  The caller owns the handle. */
lmloss_status lmloss_create(lmloss_handle* handle, int device, int64_t max_T, int32_t max_segments);

/* Free the handle and its workspace.  Synchronises the handle's device. */
lmloss_status lmloss_destroy(lmloss_handle handle);

/* Host-only validation of `args` (no CUDA call).  Returns what
 * lmloss_forward_backward would return before launching anything, except
 * for the handle's capacity limits. */
lmloss_status lmloss_check_args(const lmloss_args* args);

/*
 * Loss and gradient for one batch, asynchronous on `stream`.  The call makes
 * no host synchronisation and no allocation, so it may be captured into a CUDA
 * graph and replayed (the graph then reads whatever the captured buffers hold).
 *
 * Paths:
 *   - no GSPO, grad_out != NULL: one fused kernel reads every active row once
 *     (staged in shared memory across a thread-block cluster), reduces its
 *     max / non-target sum / teacher statistics through distributed shared
 *     memory, and writes the gradient once;
 *   - no GSPO, grad_out == NULL: forward statistics only;
 *   - GSPO: statistics pass, segment seam, gradient pass (the seam must see
 *     every row of a segment before any gradient, so the logits are read twice)
 *     [Fast-LLM PR 552, "Approach": GSPO's backward follows its eager seam].
 * A teacher combines with every other term, GSPO included (its gradient pass
 * reads the teacher's row statistics back from the workspace).
 * Row length: a row is staged across at most 16 CTAs, each slice in one CTA's
 * shared memory (227 KB on GB300), so V is at most 1,835,008 for bf16 logits
 * (917,504 with a teacher) and half that for fp32; a longer row returns
 * LMLOSS_ERR_UNSUPPORTED before anything is launched.  Vocabularies beyond that
 * go through the vocabulary-shard calls below.
 * loss_out is written on every path.  The gradient is
 *   s * (ce_weight (p - onehot) + 2 z_alpha lse p + kl_weight (p^tau - q) / tau)
 *     + c_r (p - onehot)
 * with s the token scale, c_r the row's GSPO (or GRPO) coefficient, and the
 * distillation term the derivative of kl_weight KL(q || p^tau) (Fast-LLM PR 552,
 * the list of combinable losses, names distillation; read as the forward KL at
 * temperature tau with no tau^2 factor, so tau = 1 gives kl_weight (p - q)); it
 * is rounded to nearest-even into dtype.
 */
lmloss_status lmloss_forward_backward(lmloss_handle handle, const lmloss_args* args, cudaStream_t stream);

/*
 * lmloss_forward_backward for logits that are in host memory: the call copies
 * them into the device buffer args->logits (and the teacher's into
 * args->teacher_logits) itself, in chunks of chunk_rows rows (0: T / 8, at
 * most 64 chunks), on a stream of the handle's own, and launches each chunk's
 * staged-row kernel on `stream` as soon as that chunk has landed, so the
 * kernels run under the copies of the chunks after them and the call takes
 * little more than the copies.
 *
 * host_logits (host_teacher) hold the same [T, ld] rows as the device buffer;
 * host_teacher is non-NULL exactly when args->teacher_logits is.  The copies
 * overlap only from pinned memory (cudaHostAlloc / cudaHostRegister).  Every
 * other pointer in args is device memory as for lmloss_forward_backward; the
 * gradient may be written in place into args->logits.  The copies start after
 * the work already queued on `stream`; the whole call is complete when `stream`
 * reaches its end.  Results are bitwise those of lmloss_forward_backward on the
 * same data (each row's computation does not depend on the chunking, and the
 * token-mean count and the loss reduction run once over all rows).
 *
 * With GSPO (segment_ids) the chunks run the statistics pass; the segment step
 * and the gradient pass, which need every row's log-prob, follow once all rows
 * are in.  The first call creates the copy stream and 65 events (freed by
 * lmloss_destroy), so it belongs before any stream capture; later calls can be
 * captured in a CUDA graph (the copy stream joins the capture through the
 * events, and a replay copies whatever the host buffers hold then).
 * lmloss_set_timing records nothing for this call.
 */
lmloss_status lmloss_forward_backward_host(lmloss_handle handle, const lmloss_args* args, const void* host_logits,
                                           const void* host_teacher, int64_t chunk_rows, cudaStream_t stream);

/* Read and clear the device error word.  Synchronises the handle's device.
 * Returns LMLOSS_OK when no device-side data error occurred since the last read. */
lmloss_status lmloss_get_device_error(lmloss_handle handle);

/* Human-readable name of a status. */
const char* lmloss_status_string(lmloss_status status);

/* Override the fused kernel's launch shape: cluster size (1..16), threads per
 * CTA (128, 256, 512 or 1024) and rows staged per CTA (1 or 2); other values are
 * LMLOSS_ERR_INVALID_ARG, and 0 keeps the automatic choice.  Shapes that do not
 * fit are rejected at the next call with LMLOSS_ERR_UNSUPPORTED. */
lmloss_status lmloss_set_launch_config(lmloss_handle handle, int cluster, int threads, int nbuf);

/* When enabled (which also resets the record), each call records a pair of
 * CUDA events on its stream around its main kernel(s), up to 4096 calls.
 * lmloss_get_timing waits for the last pair and returns the summed elapsed
 * time of every recorded call and how many calls were recorded. */
lmloss_status lmloss_set_timing(lmloss_handle handle, int enable);
lmloss_status lmloss_get_timing(lmloss_handle handle, float* total_ms, int32_t* calls);

/* Failure-detection self-test (diagnostic; synchronises the device): runs the
 * bounded wait that guards every copy in the kernels on a barrier that nothing
 * arrives at, giving up after limit_cycles SM clock cycles.  Returns
 * LMLOSS_ERR_TIMEOUT when the wait gave up as it should (LMLOSS_OK if it
 * somehow completed), with the device still usable. */
lmloss_status lmloss_selftest_bounded_wait(lmloss_handle handle, long long limit_cycles);

/* Launch shape and kernel count of the last call on this handle. */
lmloss_status lmloss_get_call_info(lmloss_handle handle, lmloss_call_info* info);

/*
 * Allocation-free variant of lmloss_forward_backward.  The pages have no
 * counterpart: it is for callers that may not allocate device memory once they
 * are running, such as an inference-engine plugin whose enqueue step must not
 * allocate, or a service that plans all of its device memory at start-up,
 * because cudaMalloc can synchronise the device and can fail under memory
 * pressure.
 *
 * Same arguments, results and asynchrony as lmloss_forward_backward, on the
 * current device, without a handle.  It allocates nothing: its workspace is a
 * fixed array of about 2.8 MB inside this library, which every GPU that loads
 * the library holds until the process exits.  Limits: T <= LMLOSS_NOALLOC_MAX_T
 * rows and, with GSPO, num_segments <= LMLOSS_NOALLOC_MAX_SEGMENTS; a larger
 * call returns LMLOSS_ERR_INVALID_ARG before anything is launched.
 *
 * The first call on a device looks up the array's device address and the
 * device's SM limits, and clears the array (no allocation; it synchronises
 * that device once); make that first call before any stream capture.  The
 * address is kept for the life of the process: after cudaDeviceReset on a
 * device the module is reloaded elsewhere, so do not call this entry point on
 * that device again.  Every call on a device shares the one array, which keeps the last
 * call's contents, so calls that overlap on the GPU (other streams, other host
 * threads) race and must be serialised by the caller.  Device-side data errors
 * show up only as NaN losses and gradients: there is no handle to read them from.
 */
#define LMLOSS_NOALLOC_MAX_T 65536
#define LMLOSS_NOALLOC_MAX_SEGMENTS 4096
lmloss_status lmloss_forward_backward_noalloc(const lmloss_args* args, cudaStream_t stream);

/* ---- Vocabulary-split rows (the vocabulary of each row spread over K shards)
 *
 * torchtitan PR 5661, "Numerics (TP > 1 only)": with the vocabulary split over
 * devices, each shard drops the target from its own sum of exponentials and
 * only per-row statistics are combined.  Here the K shards are K separate
 * [T, V_k] logit matrices on one GPU, holding the columns [v0_k, v0_k + V_k)
 * of a V_total-wide vocabulary.  Three steps, in order, on one handle, with no
 * other call on that handle in between (the merge leaves the rows' statistics
 * in its workspace for the gradient step); cross-entropy and z-loss only (a
 * teacher, GSPO, GRPO, the entropy or per-row KL: LMLOSS_ERR_UNSUPPORTED).
 *
 * lmloss_shard_stats: for each active row, the shard's maximum over its
 *   non-target columns, the sum of e^(z - max) over them, the target logit if
 *   the shard holds the target column and 1.0 / 0.0 for "holds it", into
 *   part_out[4 T] (device, fp32, caller-owned).  `args` describes the shard:
 *   logits [T, ld] with V = V_k columns, targets in global column numbers
 *   [0, V_total).  grad_out and loss_out are ignored.
 * lmloss_shard_merge: merges the K shards' partials (parts: host array of K
 *   <= 16 device pointers) in shard order into each row's NLL and lse; writes
 *   loss_out (CE and z-loss with the call's reduction; the KL and policy slots
 *   are 0), logp_out / lse_out / count_out if given.  `args`: T, V = V_total,
 *   targets, loss_mask, ce_weight, z_alpha, reduction, denominator; logits are
 *   not read.  A row whose target no shard holds sets LMLOSS_ERR_BAD_TARGET.
 * lmloss_shard_grad: writes the shard's gradient (grad_out, [T, ld], may alias
 *   the shard's logits) from the merged statistics: the same bits as a
 *   whole-row call would give each column, up to the order of the merge. */
lmloss_status lmloss_shard_stats(lmloss_handle handle, const lmloss_args* args, int64_t v0, int64_t V_total,
                                 float* part_out, cudaStream_t stream);
lmloss_status lmloss_shard_merge(lmloss_handle handle, const lmloss_args* args, const float* const* parts,
                                 int32_t K, cudaStream_t stream);
lmloss_status lmloss_shard_grad(lmloss_handle handle, const lmloss_args* args, int64_t v0, int64_t V_total,
                                cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LMLOSS_H */
