"""Seeded synthetic calibration activations.

This module only draws numbers: it holds none of the Hessian arithmetic, so
both the CUDA path and the float64 oracle can be fed from it.  The recipes
follow the workloads the pages describe for the Hessian GEMM (NVIDIA
Model-Optimizer PR #3002, Testing: about 360 batches of 1 to 2,000 tokens at
widths 2,560 and 4,096; ``local_hessian`` at 32K tokens and 4,096 features):

* token counts of a ragged stream: ``numpy.random.default_rng(seed)``
  integers in ``[lo, hi]``;
* values: ``torch.randn`` from a ``torch.Generator`` seeded with
  ``1_000_000 * workload_seed + batch_index``, times a per-channel scale,
  then rounded to bf16 (round to nearest even) for the bf16 path, or kept in
  fp32 for the fp32-input path;
* per-channel structure: 1 % outlier channels x20, log-uniform std in
  [0.1, 10], or 1 % Student-t(3) channels ``z / sqrt(chi2_3 / 3)``.

No dataset is used: these stand in for the calibration activations the pages
capture from real models.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

__all__ = [
    "Workload",
    "WORKLOADS",
    "ragged_token_counts",
    "channel_profile",
    "make_batch",
    "to_float64",
]


def ragged_token_counts(seed: int, n_batches: int, lo: int = 1, hi: int = 2000) -> np.ndarray:
    """Token counts of a ragged calibration stream, uniform on [lo, hi]."""
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, size=n_batches).astype(np.int64)


def channel_profile(kind: str, d: int, seed: int) -> tuple[Optional[np.ndarray], Optional[np.ndarray]]:
    """Per-channel structure of a workload.

    Returns ``(scale, heavy_mask)``: a float64 per-channel multiplier (or None
    for unit scale) and a boolean mask of Student-t(3) channels (or None).
    """
    rng = np.random.default_rng(10_000 + seed)
    if kind == "normal":
        return None, None
    if kind == "outlier":
        k = int(round(0.01 * d))
        idx = rng.permutation(d)[:k]
        scale = np.ones(d)
        scale[idx] = 20.0
        return scale, None
    if kind == "loguniform":
        u = rng.uniform(math.log(0.1), math.log(10.0), size=d)
        return np.exp(u), None
    if kind == "student_t":
        k = max(1, int(round(0.01 * d)))
        idx = rng.permutation(d)[:k]
        mask = np.zeros(d, dtype=bool)
        mask[idx] = True
        return None, mask
    if kind == "student_t_every16":
        mask = np.zeros(d, dtype=bool)
        mask[::16] = True
        return None, mask
    raise ValueError(f"unknown channel profile {kind!r}")


def make_batch(
    n: int,
    d: int,
    seed: int,
    *,
    profile: str = "normal",
    profile_seed: int = 0,
    dtype: torch.dtype = torch.bfloat16,
    device="cpu",
) -> torch.Tensor:
    """One ``[n, d]`` activation batch, row-major and contiguous.

    Values are drawn in fp32 on ``device`` and rounded once to ``dtype``.
    The same ``(seed, device)`` always gives the same tensor.
    """
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    x = torch.randn((n, d), generator=g, device=dev, dtype=torch.float32)
    scale, heavy = channel_profile(profile, d, profile_seed)
    if heavy is not None and n > 0:
        cols = torch.from_numpy(np.nonzero(heavy)[0]).to(dev)
        chi = torch.randn((n, cols.numel(), 3), generator=g, device=dev, dtype=torch.float32)
        chi2 = (chi * chi).sum(-1)
        x[:, cols] = x[:, cols] / torch.sqrt(chi2 / 3.0)
    if scale is not None:
        x = x * torch.from_numpy(scale.astype(np.float32)).to(dev)
    return x.to(dtype).contiguous()


def to_float64(t: torch.Tensor) -> np.ndarray:
    """Exact widening of a bf16 / fp16 / fp32 tensor to a float64 array."""
    return t.detach().to("cpu").to(torch.float64).numpy()


@dataclasses.dataclass(frozen=True)
class Workload:
    """A named calibration workload: width, token counts and value recipe."""

    name: str
    d: int
    token_counts: tuple
    profile: str
    seed: int
    damp_percent: float = 0.01
    local: bool = False

    @property
    def n_tokens(self) -> int:
        return int(sum(self.token_counts))

    def batch_seed(self, b: int) -> int:
        return 1_000_000 * self.seed + b

    def batch(self, b: int, *, dtype=torch.bfloat16, device="cpu") -> torch.Tensor:
        return make_batch(
            int(self.token_counts[b]), self.d, self.batch_seed(b),
            profile=self.profile, profile_seed=self.seed, dtype=dtype, device=device,
        )

    def scaled(self, n_batches: Optional[int] = None, counts: Optional[Sequence[int]] = None) -> "Workload":
        """The same recipe with fewer batches or other token counts."""
        tc = tuple(counts) if counts is not None else self.token_counts[: n_batches]
        return dataclasses.replace(self, token_counts=tuple(int(c) for c in tc))


def _ragged(seed: int) -> tuple:
    return tuple(int(c) for c in ragged_token_counts(seed, 360))


WORKLOADS = {
    # Single linear layer: 4 batches of 128 tokens, N(0,1), damp 1 %.
    "d256_4x128": Workload("d256_4x128", 256, (128,) * 4, "normal", 1, damp_percent=0.01),
    # Ragged stream at width 2,560 with 1 % outlier channels x20.
    "d2560_ragged360_outlier": Workload("d2560_ragged360_outlier", 2560, _ragged(2), "outlier", 2),
    # Ragged stream at width 4,096, per-channel std log-uniform in [0.1, 10].
    "d4096_ragged360_loguniform": Workload("d4096_ragged360_loguniform", 4096, _ragged(3), "loguniform", 3),
    # Large batches: 16 updates of 32,768 tokens at width 4,096.
    "d4096_16x32768": Workload("d4096_16x32768", 4096, (32768,) * 16, "normal", 4),
    # local_hessian: 8 updates of 32,768 tokens, 1 % Student-t(3) channels.
    "local_d4096_8x32768": Workload("local_d4096_8x32768", 4096, (32768,) * 8, "student_t", 5, local=True),
}


def make_weight(rows: int, d: int, seed: int, *, dtype: torch.dtype = torch.float32, device="cpu") -> torch.Tensor:
    """A ``[rows, d]`` linear-layer weight (output channel by input column).

    Entries are N(0, 0.02^2), the usual initialisation scale of transformer
    projections, with 1 % of the input columns scaled by 8 (salient columns)
    so that group maxima differ across groups.  Drawn in fp32, rounded once
    to ``dtype``.
    """
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    w = 0.02 * torch.randn((rows, d), generator=g, device=dev, dtype=torch.float32)
    rng = np.random.default_rng(20_000 + int(seed))
    cols = rng.permutation(d)[: max(1, d // 100)]
    w[:, torch.from_numpy(cols).to(dev)] *= 8.0
    return w.to(dtype).contiguous()
