"""Shared helpers for the GPU parity tests (tolerances and comparisons)."""

import numpy as np
import torch

from gptq_qqq_calibration_gb300.synthetic import make_batch, to_float64

# Tolerances, relative to the mean of the oracle's diagonal: bf16 inputs
# 5e-5, fp32 inputs 1e-5.  Local blocks are graded per block against the
# mean of that block's diagonal.
TOL_BF16 = 5e-5
TOL_F32 = 1e-5


def rel_err(H_gpu, H_ref):
    H_gpu = np.asarray(H_gpu, dtype=np.float64)
    m = float(np.mean(np.diagonal(H_ref)))
    return float(np.abs(H_gpu - H_ref).max() / m)


def block_rel_err(L_gpu, L_ref):
    worst = 0.0
    for b in range(L_ref.shape[0]):
        m = float(np.mean(np.diagonal(L_ref[b])))
        if m == 0.0:
            assert not np.any(L_gpu[b]), b
            continue
        worst = max(worst, float(np.abs(np.asarray(L_gpu[b], np.float64) - L_ref[b]).max() / m))
    return worst


def batches(d, counts, seed, profile="normal", dtype=torch.bfloat16, device="cuda"):
    for b, n in enumerate(counts):
        yield make_batch(int(n), d, 1_000_000 * seed + b, profile=profile, profile_seed=seed,
                         dtype=dtype, device=device)


def host(X):
    return to_float64(X)
