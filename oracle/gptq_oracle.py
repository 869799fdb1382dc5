"""Float64 CPU oracle of the quantization pass that consumes the Hessian.

TEST INFRASTRUCTURE ONLY (imported by ``tests/`` alone; shares no code with
the CUDA library).

GPTQModel wiki "QQQ", Concepts (Quadratic error compensation), the
quantization pass:
  1. copy the weight to an fp32 (here: float64) working matrix;
  2. neutralize dead input columns of the Hessian/weight pair;
  3. add damp_percent * mean(diag(H)) to the diagonal;
  4. compute an upper Cholesky factor of the inverse damped Hessian;
  5. quantize successive columns and propagate their scaled errors into the
     remaining columns, in blocks of 128 columns.
Same page, "Quantizer API and results": the damping value returned is the
absolute damp_percent * mean(diag(H)); the loss is the summed
Hessian-scaled column error.

Readings (the pages do not spell these out):
  * dead column: diag(H)_i == 0; it gets H_ii = 1 and W[:, i] = 0;
  * the mean diagonal for damping is taken after the dead-column fix;
  * error of column i: (w_i - q_i) / U_ii, propagated as
    W[:, j] -= err * U_ij for j > i (within the block at once, beyond the
    block after it);
  * loss = sum over columns and rows of (w - q)^2 / U_ii^2 / 2, and the
    reported average divides that sum by the Hessian's token count (same
    page, "Quantizer API and results");
  * "Whole-row and grouped weight quantization" (same page): whole-row
    (group_size = -1) codes are signed 4-bit with one symmetric scale per
    row, s = max|w_row| / 7, q = clamp(round(w / s), -8, 7); grouped
    (group_size = 128) codes are centered unsigned 4-bit with
    s = 2 max|w_group| / 15, q = clamp(round(w / s) + 8, 0, 15); an all-zero
    row or group uses max = 1; round is to nearest even; the whole-row scale
    is found once, before any column is quantized; a group's scale is found
    when its first column is reached (from the error-updated weights).
Parity pins: tests/test_gptq_oracle_pins.py.
"""

from __future__ import annotations

import numpy as np

__all__ = ["gptq_quantize", "upper_cholesky_of_inverse", "quantize_column"]

BLOCK = 128


def upper_cholesky_of_inverse(H: np.ndarray) -> np.ndarray:
    """U upper triangular with U^T U = H^{-1} (step 4)."""
    Hinv = np.linalg.inv(H)
    L = np.linalg.cholesky(Hinv)  # Hinv = L L^T, L lower
    return L.T


def _scale(absmax, bits_levels):
    m = np.where(absmax > 0, absmax, 1.0)
    return m / bits_levels


def quantize_column(w, s, grouped: bool, dtype=np.float64):
    """Dequantized value and code of one column (vector over rows)."""
    w = np.asarray(w, dtype=dtype)
    s = np.asarray(s, dtype=dtype)
    if grouped:
        q = np.clip(np.rint(w / s) + 8, 0, 15)
        return (s * (q - 8)).astype(dtype), q
    q = np.clip(np.rint(w / s), -8, 7)
    return (s * q).astype(dtype), q


def gptq_quantize(H, W, damp_percent: float, group_size: int = 128, dtype=np.float64, U=None,
                  n_tokens=None):
    """Run steps 1-5.  Returns dict(Wq, codes, scales, damp, loss, avg_loss, U, dead, Wpre).

    `dtype` is the arithmetic of steps 5 (float64 by default; float32 to take
    the quantization decisions in the kernel's precision).  `U` may be given
    to reuse a factor computed elsewhere.  `codes` are the signed 4-bit
    values c with Wq = scale * c (grouped codes stored centered: c = q - 8).
    `avg_loss` is loss / n_tokens when n_tokens is given and positive.
    `Wpre[:, i]` is the value column i held when it was quantized.
    """
    H = np.array(H, dtype=np.float64)
    W = np.array(W, dtype=np.float64)  # step 1: working copy
    d = H.shape[0]
    if group_size not in (-1, BLOCK):
        raise ValueError("group_size must be -1 or 128")
    if d % BLOCK:
        raise ValueError("d must be a multiple of 128")
    # step 2: dead input columns
    dead = np.diagonal(H) == 0
    H[dead, dead] = 1.0
    W[:, dead] = 0.0
    # step 3: damping
    damp = damp_percent * float(np.mean(np.diagonal(H)))
    H[np.diag_indices(d)] += damp
    # step 4
    if U is None:
        U = upper_cholesky_of_inverse(H)
    U = np.asarray(U, dtype=np.float64)
    Uw = U.astype(dtype)
    Ww = W.astype(dtype)
    rows = W.shape[0]
    grouped = group_size == BLOCK
    n_groups = d // BLOCK if grouped else 1
    scales = np.zeros((rows, n_groups), dtype=dtype)
    if not grouped:
        scales[:, 0] = _scale(np.max(np.abs(Ww), axis=1), 7.0)
    Wq = np.zeros_like(Ww)
    codes = np.zeros(Ww.shape, dtype=np.int8)
    Wpre = np.zeros_like(Ww)
    loss = 0.0
    # step 5: blocks of 128 columns
    for b0 in range(0, d, BLOCK):
        b1 = b0 + BLOCK
        Err = np.zeros((rows, BLOCK), dtype=dtype)
        if grouped:
            scales[:, b0 // BLOCK] = _scale(np.max(np.abs(Ww[:, b0:b1]), axis=1), 7.5)
        s = scales[:, b0 // BLOCK if grouped else 0]
        for i in range(b0, b1):
            w = Ww[:, i]
            Wpre[:, i] = w
            wq, q = quantize_column(w, s, grouped, dtype)
            Wq[:, i] = wq
            codes[:, i] = (q - 8) if grouped else q
            dii = Uw[i, i]
            err = ((w - wq) / dii).astype(dtype)
            loss += float(np.sum(((w - wq).astype(np.float64) / float(dii)) ** 2) / 2.0)
            Ww[:, i + 1:b1] -= np.outer(err, Uw[i, i + 1:b1]).astype(dtype)
            Err[:, i - b0] = err
        if b1 < d:
            Ww[:, b1:] -= (Err @ Uw[b0:b1, b1:]).astype(dtype)
    avg_loss = loss / n_tokens if n_tokens else None
    return {"Wq": Wq, "codes": codes, "scales": scales, "damp": damp, "loss": loss,
            "avg_loss": avg_loss, "U": U, "dead": dead, "Wpre": Wpre}
