/*
 * gptq.h -- C ABI of the quantization pass that consumes the calibration
 * Hessian (libgptq_hess.so; status codes, streams and devices as in hess.h).
 *
 * Source (page title, then section):
 *   [Q1] GPTQModel wiki "QQQ", Concepts, Quadratic error compensation: the
 *        quantization pass (1) copies the weight to an fp32 working matrix,
 *        (2) neutralises dead input columns, (3) adds
 *        damp_percent * mean(diag H) to the diagonal, (4) takes the upper
 *        Cholesky factor U of the inverse damped Hessian, (5) quantizes the
 *        columns in order, propagating each scaled error into the columns
 *        after it, in blocks of 128 columns.
 *   [Q2] Same page, "Whole-row and grouped weight quantization": group_size
 *        -1 gives one symmetric scale per output row and signed 4-bit codes;
 *        group_size 128 gives one scale per 128 consecutive input columns and
 *        centered unsigned 4-bit codes.
 *   [Q3] Same page, "Quantizer API and results": the returned damping value
 *        is the absolute damp_percent * mean(diag H); the reported loss is
 *        the summed Hessian-scaled column error divided by the token count.
 *
 * Readings where the pages are silent:
 *   - dead column i: H_ii == 0; it gets H_ii = 1 and W[:, i] = 0 before the
 *     damping mean is taken;
 *   - whole-row scale s = max|w_row| / 7, code = clamp(rint(w / s), -8, 7);
 *     grouped scale s = 2 max|w_group| / 15, taken when the group's first
 *     column is reached, code = clamp(rint(w / s) + 8, 0, 15) - 8; an all-zero
 *     row or group uses max = 1; rint rounds half to even; Wq = s * code;
 *   - scaled error err_i = (w_i - Wq_i) / U_ii, loss = sum err_i^2 / 2.
 *
 * Arithmetic: fp32 throughout (the working-matrix precision of [Q1]); the
 * damping mean and the loss sum are accumulated in fp64.  The codes come
 * from fp32 divisions and round-to-nearest-even, so a different factor (an
 * fp64 one, say) can move a value across a rounding boundary and change a
 * code and the errors after it.
 */
#ifndef GPTQ_QQQ_GPTQ_H
#define GPTQ_QQQ_GPTQ_H

#include "hess.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gptq_ctx* gptq_t; /* workspace of one input width d */

/* Every device pointer below must be device memory of the handle's device
 * (or managed memory): host memory, pageable or pinned, and another
 * device's memory are refused with HESS_ERR_INVALID before any launch. */

/* Allocate the workspace for inputs of width d (a multiple of 128, at most
 * 32768) and weights of up to max_rows output rows: two d x d fp32 matrices
 * plus max_rows x (d + 129) fp32.  d % 128 != 0 gives HESS_ERR_UNSUPPORTED. */
hess_status gptq_create(int64_t d, int64_t max_rows, gptq_t* out);

/* Steps 2-4 [Q1] on a materialized, undamped Hessian.
 *   H        : device pointer, row-major d x d fp32, symmetric (e.g. the
 *              output of hess_materialize with damp_percent = 0), 16-byte
 *              aligned; read only.
 *   n_tokens : the Hessian's token count N, kept for the loss average [Q3].
 *   damp_percent : in [0, 1), else HESS_ERR_INVALID.
 *   damp_value_out : host pointer or NULL; receives damp_percent * mean(diag)
 *              after the dead-column fix [Q3].
 * The factor U (d x d, upper, U^T U = inv(H + damp I)) stays in the handle
 * for gptq_quantize.  The call waits for `stream`.  A pivot that is <= 0 or
 * not finite in the fp32 factorization gives HESS_ERR_NOT_PD and leaves no
 * factor. */
hess_status gptq_prepare(gptq_t g, const float* H, int64_t n_tokens, double damp_percent,
                         hess_stream_t stream, float* damp_value_out);

/* gptq_prepare on the current sums of a Hessian handle (flushes it,
 * materializes it undamped inside the workspace and takes its token count).
 * The Hessian's width must equal the workspace's. */
hess_status gptq_prepare_hess(gptq_t g, hess_t h, double damp_percent, hess_stream_t stream,
                              float* damp_value_out);

/* Copy the factor U of the last successful prepare to U_out (device, d x d
 * row-major fp32; zeros below the diagonal).  Asynchronous on `stream`. */
hess_status gptq_read_factor(gptq_t g, float* U_out, hess_stream_t stream);

/* Step 1 and step 5 [Q1, Q2] for one weight matrix with the prepared factor.
 * Several weights that read the same layer input may share one prepare.
 *   W          : device pointer, row-major [rows, d] (output channel by input
 *                column), HESS_BF16 or HESS_F32, 16-byte aligned; read only.
 *   rows       : 0 <= rows <= max_rows.
 *   group_size : -1 (whole row) or 128; anything else HESS_ERR_UNSUPPORTED.
 *   Wq_out     : device [rows, d] fp32, the dequantized weights, 16-byte aligned.
 *   scales_out : device fp32, [rows, d / 128] (grouped) or [rows] (whole row).
 *   codes_out  : device [rows, d] int8 in [-8, 7] with Wq = scale * code, or
 *                NULL; 16-byte aligned.
 *   avg_loss_out : host pointer or NULL; receives the summed loss divided by
 *                the prepared token count (the plain sum when it is 0) [Q3];
 *                when given, the call waits for `stream`.
 * Without a successful prepare: HESS_ERR_INVALID. */
hess_status gptq_quantize(gptq_t g, const void* W, int32_t w_dtype, int64_t rows, int32_t group_size,
                          float* Wq_out, float* scales_out, int8_t* codes_out, hess_stream_t stream,
                          double* avg_loss_out);

/* Free the workspace (waits for the device).  NULL is a no-op. */
hess_status gptq_destroy(gptq_t g);

#ifdef __cplusplus
}
#endif

#endif /* GPTQ_QQQ_GPTQ_H */
