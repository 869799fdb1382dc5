/*
 * hess.h -- C ABI of the GB300 calibration-Hessian library (libgptq_hess.so).
 *
 * The library accumulates the layer-input Gram matrix ("Hessian") that GPTQ
 * and QQQ weight quantization collect during calibration,
 *
 *     H = (2 / N) * sum_t x_t x_t^T ,   N = number of token vectors,
 *
 * and the batched 16x16 per-block "local Hessian".  Everything runs on one
 * CUDA device (sm_103a); every entry point is a plain C function taking host
 * scalars, device pointers and a CUDA stream.  No call takes or returns a
 * framework type.
 *
 * Sources of the operations (page title, then section):
 *   [P1] GPTQModel PR #2979 "fix(qqq): per-device Hessian partials for
 *        balanced multi-GPU calibration", Summary: H = (2/n) sum x x^T with
 *        n counting token vectors, not batches.
 *   [P2] GPTQModel PR #2981 "fix(qqq): accumulate Hessian in-place per device
 *        to reduce memory", Changes and Validation: an accumulator allocated
 *        once, in-place accumulation with no per-batch d x d temporary, the
 *        closed form 2/N X^T X, empty batches.
 *   [P3] NVIDIA Model-Optimizer PR #3002, "What does this PR do?":
 *        hessian_input_dtype float32 / bfloat16 (bf16 inputs, fp32 output,
 *        products exact in fp32), Hessian stored in float32 either way; the
 *        local_hessian 16x16 per-block Hessians built the same way.
 *   [P4] GPTQModel wiki "QQQ", Concepts (Quadratic error compensation):
 *        scale by 2 / total_samples; damping adds damp_percent*mean(diag H)
 *        to the diagonal (quantization pass, step 3); "Quantizer API and
 *        results": the returned damp is that absolute value.
 *
 * Conventions shared by every call
 *   - Status: every call returns hess_status; on failure hess_last_error()
 *     returns a thread-local message.  Invalid arguments are rejected before
 *     anything is enqueued.
 *   - Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *     default stream).  Work is enqueued asynchronously on it.
 *   - Devices: a handle belongs to the device that was current at create;
 *     later calls must be made with that device current.
 *   - Threads: calls on one handle are serialised by a per-handle mutex.
 *   - Memory: device memory is allocated only by the *_create calls (and
 *     freed by *_destroy); no other call allocates device memory [P2].
 */
#ifndef GPTQ_QQQ_HESS_H
#define GPTQ_QQQ_HESS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HESS_ABI_VERSION 1

typedef struct hess_ctx* hess_t;             /* one per layer being calibrated */
typedef struct local_hess_ctx* local_hess_t; /* one per local_hessian target */
typedef struct imatrix_ctx* imatrix_t;       /* per-column sum of squares */
typedef void* hess_stream_t;                 /* a cudaStream_t */

/* Element type of an activation batch [P3: hessian_input_dtype]. */
typedef enum {
    HESS_BF16 = 0, /* bfloat16: tensor-core products, exact in fp32 */
    HESS_F32 = 1   /* float32: its own kernel, fp32-accurate products */
} hess_dtype;

typedef enum {
    HESS_OK = 0,
    HESS_ERR_INVALID = 1,     /* bad argument (NULL, negative size, misaligned, ...) */
    HESS_ERR_UNSUPPORTED = 2, /* valid but not supported (d % 8 != 0, block != 16, ...) */
    HESS_ERR_OOM = 3,         /* device or host allocation failed (create only) */
    HESS_ERR_CUDA = 4,        /* a CUDA call failed; see hess_last_error() */
    HESS_ERR_TIMEOUT = 5,     /* a device-side wait ran out; results are invalid */
    HESS_ERR_NOT_PD = 6,      /* gptq_prepare: the damped Hessian has no fp32 Cholesky factor */
    HESS_ERR_INTERNAL = 7     /* a kernel's index guard failed (a library defect): the access
                                 was skipped and the results are invalid; reported like a
                                 timeout (hess_sync, or the calls that report a timeout) */
} hess_status;

/* Options for hess_set_option. */
typedef enum {
    HESS_OPT_FLUSH_TOKENS = 1,    /* pending tokens that trigger a flush (default 65536) */
    HESS_OPT_MAX_PENDING = 2,     /* pending batches that trigger a flush (1..192, default 192) */
    HESS_OPT_CHUNK_TOKENS = 3,    /* tokens per tensor-memory chunk before the compensated
                                     on-chip sum takes it; each chunk alternates 16-token
                                     steps between two chains (128..65536, multiple of 128,
                                     default 384).  Tensor-core accumulation rounds toward
                                     zero, so longer chunks bias H low: at 384, channels whose
                                     diagonal is 80x the mean diagonal come out ~2.4e-5 of the
                                     mean diagonal low.  fp32 batches use chunks of a sixth
                                     of this, in 32-token steps (64 by default). */
    HESS_OPT_WAIT_TIMEOUT_NS = 4, /* limit of every device-side wait, ns (default 2e9; 0 makes
                                     any wait that is not already satisfied give up) */
    HESS_OPT_SPLIT_K = 5,         /* token slabs per flush; 0 = automatic (default) */
    HESS_OPT_GRID = 6,            /* persistent CTAs per flush; 0 = one per SM (default) */
    HESS_OPT_PAIR_KERNEL = 7,     /* bf16: 0 = tiles of 128x128, one SM each (default),
                                     1 = tiles of 256x128 on pairs of SMs (fewer operand
                                     bytes per SM; faster with long chunks) */
    HESS_OPT_FOLD_EVERY = 8,      /* 1..64, default 8: the accumulator keeps each entry as two
                                     fp32 parts; most flushes add only to the low part (half
                                     the accumulator bytes of a small flush, and large flushes
                                     run as one balanced slab), and at most this many minus one
                                     flushes' sums wait in the low part before they are folded
                                     into the high part (by the next small flush, or by a pass of
                                     its own before a large one).  1 = every flush updates both
                                     parts exactly (large flushes then use split-K). */
    HESS_OPT_OVERLAP_LAUNCHES = 9 /* 1 (default): a flush's kernel is launched so that it may
                                     be scheduled while the kernel before it in the stream
                                     ends (programmatic dependent launch); it sets itself up
                                     there and waits for that kernel's memory before reading
                                     X or the accumulator.  0: plain stream order. */
} hess_option;

/* ------------------------------------------------------------------------ */
/* Full Hessian                                                              */

/* Create an accumulator for inputs of width d (features).  Allocates the
 * on-device accumulator once [P2: "allocate the partial buffer once"] on the
 * current device and zeroes it (synchronously).  The accumulator keeps each
 * entry S[i][j] (i <= j) of the running Gram as an unevaluated sum of two
 * fp32 values, about 48 significant bits: 4 * d * (d + 128) bytes
 * (69 MB at d = 4096).
 *   d      : features, 1..32768; d % 8 == 0 is required (each token row must
 *            be a multiple of 16 bytes), else HESS_ERR_UNSUPPORTED.
 *   out    : receives the handle (host pointer, non-NULL).
 * Errors: INVALID (d <= 0, out NULL), UNSUPPORTED, OOM, CUDA. */
hess_status hess_create(int64_t d, hess_t* out);

/* Add one batch of activations [P1, P2, P3].
 *   X        : device pointer, row-major [n_tokens, d], contiguous, 16-byte
 *              aligned, element type `dtype`.  May be NULL when n_tokens==0.
 *   n_tokens : rows of the flattened [-1, d] input; N += n_tokens [P1].
 *              0 is a no-op that does not change N [P2].
 *   dtype    : HESS_BF16 or HESS_F32.
 *   stream   : the stream X was produced on.
 * The batch is queued; it is summed by the next flush, which happens when
 * the queue holds HESS_OPT_MAX_PENDING batches or HESS_OPT_FLUSH_TOKENS
 * tokens, when the dtype changes, or in hess_flush / hess_materialize.
 * X is BORROWED until that flush has been enqueued and has run: the caller
 * keeps it alive and unmodified, in stream order, until then.
 * hess_pending_batches() tells how many of the most recent batches are
 * still queued after a call returns.
 * Errors: INVALID (NULL handle, n_tokens < 0, NULL X with n_tokens > 0,
 * unknown dtype, X not 16-byte aligned, X not device memory of the
 * handle's device or managed memory), CUDA, UNSUPPORTED (a tensor map of the
 * flush this call triggered could not be built).  A call that fails leaves
 * no trace: its batch is neither queued nor counted, and batches queued
 * before it stay queued for the next flush. */
hess_status hess_add_batch(hess_t h, const void* X, int64_t n_tokens, int32_t dtype,
                           hess_stream_t stream);

/* Sum every queued batch into the accumulator now (one fused pass per dtype
 * run), enqueued on `stream`, which first waits for the streams the batches
 * were added on.  No-op when nothing is queued.  If the pass cannot be built
 * (UNSUPPORTED: a tensor map the driver refuses), nothing is enqueued and the
 * batches stay queued. */
hess_status hess_flush(hess_t h, hess_stream_t stream);

/* Flush, then write the damped Hessian [P4]:
 *     H_out[i][j] = H_out[j][i] = fp32(S[i][j] * (2/N))          (i < j)
 *     H_out[i][i] = fp32(S[i][i] * (2/N) + damp),
 *     damp        = damp_percent * mean_i(S[i][i] * (2/N))        (fp64)
 * Diagonal entries are rounded once from fp64; off-diagonal entries come
 * within one ulp of the correctly rounded value (fp32 arithmetic with an
 * exact product).  H_out is bit-exactly symmetric.  With N == 0 it is all
 * zeros and damp = 0.
 *   H_out          : device pointer, row-major [d, d] fp32, 16-byte aligned.
 *   damp_percent   : in [0, 1).  (QQQ validates (0,1) and defaults to 0.005;
 *                    0 returns the undamped H.)
 *   damp_value_out : HOST pointer or NULL.  When non-NULL the call waits for
 *                    `stream` and stores fp32(damp) there.
 * The accumulator is not consumed: more batches may follow.
 * Timeouts: a device-side wait that ran out in this handle's kernels is
 * reported (HESS_ERR_TIMEOUT) by this call when damp_value_out is non-NULL
 * (it waits).  With NULL the call does not wait: it enqueues a copy of the
 * handle's status word to pinned host memory, and the first later
 * hess_add_batch, hess_flush or hess_materialize that finds that copy
 * complete reports the timeout, before doing anything else; so does every
 * call after it, until hess_reset or hess_import_state.  hess_sync reports
 * it at once.
 * Errors: INVALID (also for H_out that is not device memory of the
 * handle's device or managed memory), CUDA, TIMEOUT (above).  Every other
 * entry point that takes a device buffer (imatrix_add, imatrix_read,
 * local_hess_add, local_hess_read, local_hess_compute_noalloc, and the
 * gptq_* calls) refuses host memory the same way, before any launch. */
hess_status hess_materialize(hess_t h, float* H_out, double damp_percent, hess_stream_t stream,
                             float* damp_value_out);

/* N: token vectors added so far (queued ones included) [P1]. */
int64_t hess_token_count(hess_t h);
/* Number of the most recently added batches that are still queued. */
int64_t hess_pending_batches(hess_t h);
/* Kernels this handle has launched so far (flush passes, fold passes,
 * materializations, merges into it), or -1 for NULL.  A diagnostic count; it
 * is not reset by hess_reset. */
int64_t hess_kernel_launches(hess_t h);
/* Width d of the handle, or -1 for NULL. */
int64_t hess_dim(hess_t h);

/* Wait for `stream`, then report a device-side timeout recorded by any
 * kernel of this handle since the last reset (HESS_ERR_TIMEOUT), else OK.
 * After a timeout, hess_add_batch, hess_flush and hess_materialize fail
 * with HESS_ERR_TIMEOUT until hess_reset. */
hess_status hess_sync(hess_t h, hess_stream_t stream);

/* Drop queued batches, zero the accumulator (on `stream`) and set N = 0. */
hess_status hess_reset(hess_t h, hess_stream_t stream);

/* Set an hess_option.  Values out of range give HESS_ERR_INVALID. */
hess_status hess_set_option(hess_t h, int32_t option, int64_t value);

/* Free the handle (synchronises its device).  NULL is a no-op. */
hess_status hess_destroy(hess_t h);

/* Partials and copies                                                      */

/* dst += src: the accumulated sums and token counts of two handles of the
 * same width on the same device (per-device partials merged before the 2/N
 * scale [P1 Summary; P2 Changes: "merge per-device partials"]).  Both queues
 * are flushed on `stream` first; src is left as it was.  Enqueued on
 * `stream`.  Errors: INVALID (NULL, same handle, widths differ),
 * UNSUPPORTED (different devices), CUDA. */
hess_status hess_merge(hess_t dst, hess_t src, hess_stream_t stream);

/* A new, independent handle holding src's sums, token count and options
 * (shared-input dedup hands each follower a private copy of the leader's
 * Hessian: GPTQModel PR #3052, "adopt_hessian_from").  src is flushed first.
 * Allocates like hess_create; the copy is enqueued on `stream`. */
hess_status hess_clone(hess_t src, hess_t* out, hess_stream_t stream);

/* Checkpoint and resume.  The pages checkpoint only the quantized model; a
 * long calibration run also wants to save its partial Gram and token count
 * and resume later, so these calls have no counterpart on the pages.
 * The state is the accumulator in the library's own layout: an opaque blob of
 * hess_state_bytes(h) bytes (the accumulator, then 16 bytes that name the
 * library version and how far the low parts have been folded), valid for a
 * handle of the same width d and a library of the same HESS_ABI_VERSION.
 * A run exported and resumed gives bit for bit the H of the same run
 * uninterrupted. */
int64_t hess_state_bytes(hess_t h);  /* 0 for a NULL handle */

/* Flush, then copy the state to `dst` (host or device memory, `bytes` >=
 * hess_state_bytes(h)) on `stream`, and store the token count N in
 * *n_tokens_out (host pointer, non-NULL).  With pageable host memory the copy
 * is synchronous; otherwise the caller synchronises `stream` before reading
 * dst.  Errors: INVALID (NULL, bytes too small), CUDA. */
hess_status hess_export_state(hess_t h, void* dst, int64_t bytes, hess_stream_t stream,
                              int64_t* n_tokens_out);

/* Replace the handle's state by a blob from hess_export_state and set N to
 * n_tokens.  Batches still queued are dropped (as by hess_reset); `src` is
 * read on `stream`, and the call waits for its trailer.  Errors: INVALID
 * (NULL, bytes != hess_state_bytes(h), n_tokens < 0, a trailer that does
 * not name this library version), CUDA. */
hess_status hess_import_state(hess_t h, const void* src, int64_t bytes, int64_t n_tokens,
                              hess_stream_t stream);

/* ------------------------------------------------------------------------ */
/* imatrix statistic [P3: "a per-column sum of squares, not a GEMM"]        */

/* out[i] = sum over all added tokens of X[t][i]^2, accumulated in fp64 and
 * returned as fp32.  d % 8 == 0; X row-major [n_tokens, d], 16-byte aligned,
 * bf16 or fp32; n_tokens == 0 is a no-op. */
hess_status imatrix_create(int64_t d, imatrix_t* out);
hess_status imatrix_add(imatrix_t h, const void* X, int64_t n_tokens, int32_t dtype,
                        hess_stream_t stream);
hess_status imatrix_read(imatrix_t h, float* out, hess_stream_t stream);
int64_t imatrix_token_count(imatrix_t h);
hess_status imatrix_reset(imatrix_t h, hess_stream_t stream);
hess_status imatrix_destroy(imatrix_t h);

/* ------------------------------------------------------------------------ */
/* Local (16x16 per-block) Hessian [P3: local_hessian]                      */

/* Create a per-block accumulator: d features split into d/block blocks.
 *   block : must be 16; d % block == 0 is required, else UNSUPPORTED. */
hess_status local_hess_create(int64_t d, int32_t block, local_hess_t* out);

/* L_b += X_b^T X_b for every block b of `block` consecutive features, in one
 * pass over X; N += n_tokens (0 is a no-op).
 *   X      : device pointer, row-major [n_tokens, d] bf16, 16-byte aligned.
 *   d, block, dtype : must match the handle (dtype HESS_BF16).
 * X need only stay alive until this call's work has run on `stream`. */
hess_status local_hess_add(local_hess_t h, const void* X, int64_t n_tokens, int64_t d,
                           int32_t block, int32_t dtype, hess_stream_t stream);

/* out[b][i][j] = fp32(L_b[i][j] * (2/N)), no damping (this Hessian is never
 * inverted [P3]); symmetric per block; zeros when N == 0.
 *   out : device pointer, [d/block, block, block] fp32. */
hess_status local_hess_read(local_hess_t h, float* out, hess_stream_t stream);

int64_t local_hess_token_count(local_hess_t h);
/* Same as hess_sync for the local accumulator. */
hess_status local_hess_sync(local_hess_t h, hess_stream_t stream);
hess_status local_hess_reset(local_hess_t h, hess_stream_t stream);
hess_status local_hess_destroy(local_hess_t h);

/* One batch's local Hessian with no device allocation.  (No counterpart on
 * the source pages: this is a library convenience.)
 * For callers that must not allocate device memory while they run: those
 * whose device memory is reserved up front by a pooling allocator, so that a
 * cudaMalloc would fail or fragment the pool, and those whose runtime forbids
 * the implicit synchronisation that cudaMalloc/cudaFree can cause.
 *   out[b][i][j] = fp32(X_b^T X_b [i][j] * (2/n_tokens))  for this batch only,
 *   the same values local_hess_create + local_hess_add + local_hess_read give
 *   for a fresh handle; zeros when n_tokens == 0.
 *   X     : device pointer, row-major [n_tokens, d] bf16, 16-byte aligned.
 *   out   : device pointer, [d/16, 16, 16] fp32.
 *   block : 16; dtype : HESS_BF16.
 * Limit: d <= 16384 (the scratch holds 1,024 blocks); larger d gives
 * HESS_ERR_UNSUPPORTED with a message naming the limit.
 * Scratch: a 2 MiB fixed device array inside the library, held by every GPU
 * that loads it until the process exits and shared by every call on that
 * device.  Each call clears what it uses, but calls whose GPU work overlaps
 * (unordered streams) race on it and give wrong results.
 * Set-up: the first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  The call is asynchronous on `stream`; a
 * device-side wait that runs out leaves `out` invalid and is not reported. */
hess_status local_hess_compute_noalloc(const void* X, int64_t n_tokens, int64_t d, int32_t block,
                                       int32_t dtype, float* out, hess_stream_t stream);

/* ------------------------------------------------------------------------ */

/* Message of the last failed call on this thread ("" if none). */
const char* hess_last_error(void);
/* HESS_ABI_VERSION of the loaded library. */
int32_t hess_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GPTQ_QQQ_HESS_H */
