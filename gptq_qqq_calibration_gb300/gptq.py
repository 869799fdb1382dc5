"""Python binding of the quantization pass in ``include/gptq.h``.

Argument marshalling only: every step (dead columns, damping, the factor of
the inverse Hessian, the blockwise quantization) runs in the library's CUDA
kernels.  Functions carry the C names; ``GPTQ`` wraps a workspace handle.
"""

from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _lib
from ._lib import HESS_BF16, HESS_F32, check

__all__ = ["gptq_create", "gptq_prepare", "gptq_prepare_hess", "gptq_read_factor", "gptq_quantize",
           "gptq_destroy", "GPTQ"]

_W_DTYPES = {torch.bfloat16: HESS_BF16, torch.float32: HESS_F32}


def _stream(stream) -> int:
    return (stream if stream is not None else torch.cuda.current_stream()).cuda_stream


def _dev(t: torch.Tensor, name: str, dtype=None) -> int:
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def gptq_create(d: int, max_rows: int) -> int:
    g = ctypes.c_void_p()
    check(_lib.load().gptq_create(int(d), int(max_rows), ctypes.byref(g)))
    return g.value


def gptq_prepare(g: int, H: torch.Tensor, n_tokens: int, damp_percent: float, stream=None) -> float:
    v = ctypes.c_float()
    check(_lib.load().gptq_prepare(g, _dev(H, "H", torch.float32), int(n_tokens), float(damp_percent),
                                   _stream(stream), ctypes.byref(v)))
    return float(v.value)


def gptq_prepare_hess(g: int, h: int, damp_percent: float, stream=None) -> float:
    v = ctypes.c_float()
    check(_lib.load().gptq_prepare_hess(g, h, float(damp_percent), _stream(stream), ctypes.byref(v)))
    return float(v.value)


def gptq_read_factor(g: int, U_out: torch.Tensor, stream=None) -> None:
    check(_lib.load().gptq_read_factor(g, _dev(U_out, "U_out", torch.float32), _stream(stream)))


def gptq_quantize(g: int, W: torch.Tensor, group_size: int, Wq_out: torch.Tensor, scales_out: torch.Tensor,
                  codes_out: Optional[torch.Tensor] = None, stream=None, want_loss: bool = True):
    if W.dtype not in _W_DTYPES:
        raise ValueError(f"W must be bfloat16 or float32, got {W.dtype}")
    rows = W.shape[0] if W.dim() == 2 else 0
    loss = ctypes.c_double()
    check(_lib.load().gptq_quantize(
        g, _dev(W, "W"), _W_DTYPES[W.dtype], int(rows), int(group_size),
        _dev(Wq_out, "Wq_out", torch.float32), _dev(scales_out, "scales_out", torch.float32),
        _dev(codes_out, "codes_out", torch.int8) if codes_out is not None else None,
        _stream(stream), ctypes.byref(loss) if want_loss else None))
    return float(loss.value) if want_loss else None


def gptq_destroy(g: int) -> None:
    check(_lib.load().gptq_destroy(g))


class GPTQ:
    """Quantization workspace for one input width d (a multiple of 128).

    ``prepare`` takes a materialized Hessian (or a ``Hessian`` object) and
    keeps the factor; ``quantize`` then runs the pass for any number of
    weights of that input width.
    """

    def __init__(self, d: int, max_rows: int):
        self.d, self.max_rows = int(d), int(max_rows)
        self.handle = gptq_create(self.d, self.max_rows)
        self.damp = None

    def prepare(self, H, damp_percent: float, n_tokens: Optional[int] = None, stream=None) -> float:
        if isinstance(H, torch.Tensor):
            if n_tokens is None:
                raise ValueError("n_tokens is required with a materialized H")
            self.damp = gptq_prepare(self.handle, H, n_tokens, damp_percent, stream)
        else:
            self.damp = gptq_prepare_hess(self.handle, H.handle, damp_percent, stream)
        return self.damp

    def factor(self, stream=None) -> torch.Tensor:
        U = torch.empty((self.d, self.d), dtype=torch.float32, device="cuda")
        gptq_read_factor(self.handle, U, stream)
        return U

    def quantize(self, W: torch.Tensor, group_size: int = 128, codes: bool = True, stream=None,
                 want_loss: bool = True) -> dict:
        rows = W.shape[0]
        Wq = torch.empty((rows, self.d), dtype=torch.float32, device="cuda")
        n_groups = self.d // 128 if group_size == 128 else 1
        scales = torch.empty((rows, n_groups), dtype=torch.float32, device="cuda")
        cd = torch.empty((rows, self.d), dtype=torch.int8, device="cuda") if codes else None
        loss = gptq_quantize(self.handle, W, group_size, Wq, scales, cd, stream, want_loss)
        return {"Wq": Wq, "scales": scales, "codes": cd, "avg_loss": loss, "damp": self.damp}

    def close(self) -> None:
        if self.handle:
            gptq_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
