"""Float64 CPU oracle for the calibration Hessian (layer-input Gram).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it.  It shares no code with the CUDA
library (no kernels, headers, helpers or tables); both sides only see the
same seeded input values.

Every function is a plain restatement of what the pages define, in float64,
with no blocking, fusion or reordering beyond a library matmul:

* Accumulation.  "fix(qqq): per-device Hessian partials for balanced
  multi-GPU calibration" (GPTQModel PR #2979), Summary: the Hessian is
  ``H = (2 / n) * sum_t x_t x_t^T`` where n counts token vectors, not
  batches.  "fix(qqq): accumulate Hessian in-place per device to reduce
  memory" (GPTQModel PR #2981), Validation: the accumulated result must equal
  the closed form ``2/N * X^T X`` over a single batch, several batches and
  empty batches.
* Scaling and damping.  GPTQModel wiki "QQQ", Concepts / Quadratic error
  compensation: the merged Gram is scaled by ``2 / total_samples``; the
  quantization pass then adds ``damp_percent * mean(diag(H))`` to the
  diagonal (step 3).  Same page, "Quantizer API and results": the value
  handed back is the absolute damping ``damp_percent * mean(diag(H))``.
* Local Hessian.  NVIDIA Model-Optimizer PR #3002 ("What does this PR do?",
  the ``local_hessian`` bullet): 16x16 per-block Hessians over 16-feature
  blocks, built "the same way" as the GPTQ Hessian.  Reading taken here: the
  same ``2/N`` scaling, and no damping (that Hessian is never inverted).

Inputs are float64 arrays holding exactly the values the GPU sees (a bf16 or
fp32 tensor widened exactly to float64 by the caller).

Parity status: every function below is pinned by ``tests/test_oracle_pins.py``
(exact rational brute force, the worked example of GPTQModel PR #3052,
closed forms and invariants); none is "parity unpinned".
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "GramOracle",
    "LocalGramOracle",
    "gram_columns",
    "column_sum_of_squares",
]


def _as_tokens(X: np.ndarray, d: int) -> np.ndarray:
    """Flatten an activation batch to ``[n_tokens, d]`` float64.

    Token counting follows GPTQModel PR #2979 (Summary) and the QQQ wiki
    (Concepts): every row of the flattened ``[-1, d]`` input is one sample.
    """
    X = np.asarray(X, dtype=np.float64)
    if X.ndim == 1:
        if d != X.shape[0] and X.size != 0:
            raise ValueError("1-D input must have d entries")
        X = X.reshape(-1, d)
    X = X.reshape(-1, X.shape[-1])
    if X.shape[1] != d:
        raise ValueError(f"feature width {X.shape[1]} != {d}")
    return X


class GramOracle:
    """Running float64 Gram ``S = sum_t x_t x_t^T`` and token count ``N``.

    ``add_batch`` mirrors the accumulate step of GPTQModel PR #2979/#2981:
    ``S += X^T X`` and ``N += rows(X)``; an empty batch changes neither
    (PR #2981, Validation: "empty batches").
    """

    def __init__(self, d: int):
        if d <= 0:
            raise ValueError("d must be positive")
        self.d = int(d)
        self.S = np.zeros((self.d, self.d), dtype=np.float64)
        self.N = 0

    def add_batch(self, X: np.ndarray) -> None:
        X = _as_tokens(X, self.d)
        n = X.shape[0]
        if n == 0:
            return
        self.S += X.T @ X
        self.N += n

    def hessian(self) -> np.ndarray:
        """``H = (2/N) * S`` (QQQ wiki, Concepts; PR #2979 Summary).

        With no tokens the Hessian is all zeros (an uncalled accumulator,
        GPTQModel PR #3052 tests: "uncalled leader -> zero H").
        """
        if self.N == 0:
            return np.zeros_like(self.S)
        return self.S * (2.0 / self.N)

    def materialize(self, damp_percent: float) -> tuple[np.ndarray, float]:
        """Scale by ``2/N``, then add ``damp_percent * mean(diag(H))``.

        Order of operations follows the QQQ wiki: the Gram is scaled when it
        is materialized (Concepts), and the quantization pass damps the
        scaled matrix (step 3).  Returns ``(H_damped, damp_value)`` where
        ``damp_value = damp_percent * mean(diag(H))`` ("Quantizer API and
        results": the seventh result is this absolute value).
        """
        H = self.hessian()
        mean_diag = float(np.mean(np.diagonal(H))) if self.N else 0.0
        damp = float(damp_percent) * mean_diag
        H = H.copy()
        H[np.diag_indices(self.d)] += damp
        return H, damp


class LocalGramOracle:
    """Per-block 16x16 Grams for ``local_hessian`` (Model-Optimizer PR #3002).

    Block ``b`` covers features ``[block*b, block*(b+1))`` and accumulates
    ``L_b += X_b^T X_b``.  Reading: the result is scaled by ``2/N`` like the
    full Hessian, and is not damped.
    """

    def __init__(self, d: int, block: int = 16):
        if d <= 0 or block <= 0 or d % block:
            raise ValueError("d must be a positive multiple of block")
        self.d, self.block = int(d), int(block)
        self.nb = self.d // self.block
        self.S = np.zeros((self.nb, self.block, self.block), dtype=np.float64)
        self.N = 0

    def add_batch(self, X: np.ndarray) -> None:
        X = _as_tokens(X, self.d)
        n = X.shape[0]
        if n == 0:
            return
        for b in range(self.nb):
            Xb = X[:, b * self.block:(b + 1) * self.block]
            self.S[b] += Xb.T @ Xb
        self.N += n

    def read(self) -> np.ndarray:
        if self.N == 0:
            return np.zeros_like(self.S)
        return self.S * (2.0 / self.N)


def gram_columns(batches, cols) -> tuple[np.ndarray, int]:
    """Selected columns of the unscaled Gram: ``S[:, cols]`` and ``N``.

    The same definition as :class:`GramOracle` restricted to a subset of
    output columns, so full-width workloads can be checked entry by entry
    without forming the whole ``d x d`` float64 matrix.
    """
    cols = np.asarray(cols, dtype=np.int64)
    S = None
    N = 0
    for X in batches:
        X = np.asarray(X, dtype=np.float64)
        X = X.reshape(-1, X.shape[-1])
        if X.shape[0] == 0:
            continue
        part = X.T @ X[:, cols]
        S = part if S is None else S + part
        N += X.shape[0]
    return S, N


def column_sum_of_squares(batches) -> tuple[np.ndarray, int]:
    """``sum_t x_{t,i}^2`` for every feature i, and N.

    This is the diagonal of the unscaled Gram written as a sum of squares,
    which is all the mean-diagonal damping term needs.
    """
    out = None
    N = 0
    for X in batches:
        X = np.asarray(X, dtype=np.float64)
        X = X.reshape(-1, X.shape[-1])
        if X.shape[0] == 0:
            continue
        sq = np.einsum("ti,ti->i", X, X)
        out = sq if out is None else out + sq
        N += X.shape[0]
    return out, N
