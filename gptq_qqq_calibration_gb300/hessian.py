"""Python binding of the C ABI in ``include/hess.h``.

Argument marshalling only: tensors become device pointers and sizes, the
current torch stream becomes the ``cudaStream_t``; every step of the
computation runs in the library's CUDA kernels.  There is no CPU path.

Functions carry the C names (``hess_create``, ``hess_add_batch``, ...);
``Hessian`` and ``LocalHessian`` wrap a handle and keep every queued batch
alive until the library has consumed it.
"""

from __future__ import annotations

import ctypes
import threading
from typing import Optional

import torch

from . import _lib
from ._lib import HESS_BF16, HESS_F32, HessError, check

__all__ = [
    "HESS_BF16", "HESS_F32", "HessError",
    "hess_create", "hess_add_batch", "hess_flush", "hess_materialize", "hess_token_count",
    "hess_pending_batches", "hess_kernel_launches", "hess_sync", "hess_reset", "hess_set_option",
    "hess_destroy",
    "local_hess_create", "local_hess_add", "local_hess_read", "local_hess_token_count",
    "local_hess_sync", "local_hess_reset", "local_hess_destroy",
    "hess_merge", "hess_clone", "hess_state_bytes", "hess_export_state", "hess_import_state",
    "imatrix_create", "imatrix_add", "imatrix_read",
    "imatrix_token_count", "imatrix_reset", "imatrix_destroy",
    "Hessian", "LocalHessian", "IMatrix",
]

_DTYPES = {torch.bfloat16: HESS_BF16, torch.float32: HESS_F32}


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    if stream is not None:
        return stream.cuda_stream
    # the raw handle of the current stream, without building a Stream object
    return torch._C._cuda_getCurrentRawStream(torch.cuda.current_device())


def _tokens_view(X: torch.Tensor, d: int) -> tuple:
    if not X.is_cuda:
        raise ValueError("X must be a CUDA tensor")
    if X.dtype not in _DTYPES:
        raise ValueError(f"X must be bfloat16 or float32, got {X.dtype}")
    if X.shape[-1] != d:
        raise ValueError(f"last dimension {X.shape[-1]} != d = {d}")
    if not X.is_contiguous():
        raise ValueError("X must be contiguous (row-major [tokens, d])")
    return X.numel() // d, _DTYPES[X.dtype]


# ---------------------------------------------------------------- raw calls


def hess_create(d: int) -> int:
    h = ctypes.c_void_p()
    check(_lib.load().hess_create(int(d), ctypes.byref(h)))
    return h.value


def hess_add_batch(h: int, X: torch.Tensor, d: int, stream=None) -> None:
    n, dt = _tokens_view(X, d)
    check(_lib.load().hess_add_batch(h, X.data_ptr() if n else None, n, dt, _stream(stream)))


def hess_flush(h: int, stream=None) -> None:
    check(_lib.load().hess_flush(h, _stream(stream)))


def hess_materialize(h: int, H_out: torch.Tensor, damp_percent: float, stream=None,
                     want_damp: bool = True) -> Optional[float]:
    if H_out.dtype != torch.float32 or not H_out.is_cuda or not H_out.is_contiguous():
        raise ValueError("H_out must be a contiguous float32 CUDA tensor")
    v = ctypes.c_float()
    check(_lib.load().hess_materialize(h, H_out.data_ptr(), float(damp_percent), _stream(stream),
                                       ctypes.byref(v) if want_damp else None))
    return float(v.value) if want_damp else None


def hess_token_count(h: int) -> int:
    return int(_lib.load().hess_token_count(h))


def hess_pending_batches(h: int) -> int:
    return int(_lib.load().hess_pending_batches(h))


def hess_kernel_launches(h: int) -> int:
    return int(_lib.load().hess_kernel_launches(h))


def hess_sync(h: int, stream=None) -> None:
    check(_lib.load().hess_sync(h, _stream(stream)))


def hess_reset(h: int, stream=None) -> None:
    check(_lib.load().hess_reset(h, _stream(stream)))


def hess_set_option(h: int, name: str, value: int) -> None:
    check(_lib.load().hess_set_option(h, _lib.OPTIONS[name], int(value)))


def hess_destroy(h: int) -> None:
    check(_lib.load().hess_destroy(h))


def hess_merge(dst: int, src: int, stream=None) -> None:
    check(_lib.load().hess_merge(dst, src, _stream(stream)))


def hess_clone(src: int, stream=None) -> int:
    h = ctypes.c_void_p()
    check(_lib.load().hess_clone(src, ctypes.byref(h), _stream(stream)))
    return h.value


def hess_state_bytes(h: int) -> int:
    return int(_lib.load().hess_state_bytes(h))


def hess_export_state(h: int, dst: torch.Tensor, stream=None) -> int:
    """Copy the state into `dst` (a contiguous uint8 tensor on the host or the
    device); returns the token count N."""
    n = ctypes.c_int64()
    check(_lib.load().hess_export_state(h, dst.data_ptr(), dst.numel() * dst.element_size(),
                                        _stream(stream), ctypes.byref(n)))
    return n.value


def hess_import_state(h: int, src: torch.Tensor, n_tokens: int, stream=None) -> None:
    check(_lib.load().hess_import_state(h, src.data_ptr(), src.numel() * src.element_size(),
                                        int(n_tokens), _stream(stream)))


def imatrix_create(d: int) -> int:
    h = ctypes.c_void_p()
    check(_lib.load().imatrix_create(int(d), ctypes.byref(h)))
    return h.value


def imatrix_add(h: int, X: torch.Tensor, d: int, stream=None) -> None:
    n, dt = _tokens_view(X, d)
    check(_lib.load().imatrix_add(h, X.data_ptr() if n else None, n, dt, _stream(stream)))


def imatrix_read(h: int, out: torch.Tensor, stream=None) -> None:
    if out.dtype != torch.float32 or not out.is_cuda or not out.is_contiguous():
        raise ValueError("out must be a contiguous float32 CUDA tensor")
    check(_lib.load().imatrix_read(h, out.data_ptr(), _stream(stream)))


def imatrix_token_count(h: int) -> int:
    return int(_lib.load().imatrix_token_count(h))


def imatrix_reset(h: int, stream=None) -> None:
    check(_lib.load().imatrix_reset(h, _stream(stream)))


def imatrix_destroy(h: int) -> None:
    check(_lib.load().imatrix_destroy(h))


def local_hess_create(d: int, block: int = 16) -> int:
    h = ctypes.c_void_p()
    check(_lib.load().local_hess_create(int(d), int(block), ctypes.byref(h)))
    return h.value


def local_hess_add(h: int, X: torch.Tensor, d: int, block: int = 16, stream=None) -> None:
    n, dt = _tokens_view(X, d)
    check(_lib.load().local_hess_add(h, X.data_ptr() if n else None, n, int(d), int(block), dt,
                                     _stream(stream)))


def local_hess_read(h: int, out: torch.Tensor, stream=None) -> None:
    if out.dtype != torch.float32 or not out.is_cuda or not out.is_contiguous():
        raise ValueError("out must be a contiguous float32 CUDA tensor")
    check(_lib.load().local_hess_read(h, out.data_ptr(), _stream(stream)))


def local_hess_token_count(h: int) -> int:
    return int(_lib.load().local_hess_token_count(h))


def local_hess_sync(h: int, stream=None) -> None:
    check(_lib.load().local_hess_sync(h, _stream(stream)))


def local_hess_reset(h: int, stream=None) -> None:
    check(_lib.load().local_hess_reset(h, _stream(stream)))


def local_hess_destroy(h: int) -> None:
    check(_lib.load().local_hess_destroy(h))


# ------------------------------------------------------------------ objects


class Hessian:
    """Accumulator of ``H = (2/N) sum x x^T`` for one layer input of width d.

    One object may be used from several host threads: a re-entrant lock
    makes each library call and the bookkeeping of the batches it borrows
    one step, so a batch that another thread has just queued is never
    released early."""

    def __init__(self, d: int, **options):
        self.d = int(d)
        self._lock = threading.RLock()
        self.handle = hess_create(self.d)
        self._queued = []  # batches the library still borrows, oldest first
        for k, v in options.items():
            hess_set_option(self.handle, k, v)

    def add_batch(self, X: torch.Tensor, stream=None) -> None:
        with self._lock:
            hess_add_batch(self.handle, X, self.d, stream)
            if X.numel():
                self._queued.append(X)
            self._release(stream)

    def _release(self, stream=None) -> None:
        """Drop the references to batches the library has flushed.  The flush
        was enqueued on the stream of the call that triggered it (`stream`,
        else the current stream), so each tensor is marked as in use there:
        the caching allocator then reuses its memory only after that flush
        has read it.  Called with the lock held."""
        keep = hess_pending_batches(self.handle)
        if keep < len(self._queued):
            s = stream if stream is not None else torch.cuda.current_stream()
            for t in self._queued[: len(self._queued) - keep]:
                t.record_stream(s)
            self._queued = self._queued[len(self._queued) - keep:] if keep else []

    def flush(self, stream=None) -> None:
        with self._lock:
            hess_flush(self.handle, stream)
            self._release(stream)

    def materialize(self, damp_percent: float = 0.0, out: Optional[torch.Tensor] = None,
                    stream=None, want_damp: bool = True):
        if out is None:
            out = torch.empty((self.d, self.d), dtype=torch.float32, device="cuda")
        with self._lock:
            damp = hess_materialize(self.handle, out, damp_percent, stream, want_damp)
            self._release(stream)
        return out, damp

    @property
    def n_tokens(self) -> int:
        return hess_token_count(self.handle)

    def sync(self, stream=None) -> None:
        hess_sync(self.handle, stream)

    def reset(self, stream=None) -> None:
        with self._lock:
            hess_reset(self.handle, stream)
            self._queued = []

    def set_option(self, name: str, value: int) -> None:
        hess_set_option(self.handle, name, value)

    def merge(self, other: "Hessian", stream=None) -> None:
        """Add another accumulator's sums and token count into this one."""
        first, second = sorted((self, other), key=id)  # one lock order for every pair
        with first._lock, second._lock:
            hess_merge(self.handle, other.handle, stream)
            self._release(stream)
            other._release(stream)

    def clone(self, stream=None) -> "Hessian":
        """An independent copy of the sums, token count and options."""
        h = Hessian.__new__(Hessian)
        h.d = self.d
        h._lock = threading.RLock()
        h._queued = []
        with self._lock:
            h.handle = hess_clone(self.handle, stream)
            self._release(stream)
        return h

    def export_state(self, device: str = "cpu", stream=None) -> tuple:
        """A checkpoint: (state, N), the state a uint8 tensor on `device` (host
        memory is pinned).  The copy has completed when this returns."""
        buf = torch.empty(hess_state_bytes(self.handle), dtype=torch.uint8, device=device)
        if buf.device.type == "cpu":
            buf = buf.pin_memory()
        with self._lock:
            n = hess_export_state(self.handle, buf, stream)
            hess_sync(self.handle, stream)
            self._release(stream)
        return buf, n

    def import_state(self, state: torch.Tensor, n_tokens: int, stream=None) -> None:
        """Resume from a checkpoint of export_state (queued batches are dropped)."""
        state = state.contiguous()
        with self._lock:
            hess_import_state(self.handle, state, n_tokens, stream)
            self._queued = []
            hess_sync(self.handle, stream)

    def close(self) -> None:
        with self._lock:
            if self.handle:
                hess_destroy(self.handle)
                self.handle = None
                self._queued = []

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class LocalHessian:
    """Per-block 16x16 Hessians (local_hessian) for inputs of width d."""

    def __init__(self, d: int, block: int = 16):
        self.d, self.block = int(d), int(block)
        self.handle = local_hess_create(self.d, self.block)

    def add_batch(self, X: torch.Tensor, stream=None) -> None:
        local_hess_add(self.handle, X, self.d, self.block, stream)

    def read(self, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        if out is None:
            out = torch.empty((self.d // self.block, self.block, self.block), dtype=torch.float32,
                              device="cuda")
        local_hess_read(self.handle, out, stream)
        return out

    @property
    def n_tokens(self) -> int:
        return local_hess_token_count(self.handle)

    def sync(self, stream=None) -> None:
        local_hess_sync(self.handle, stream)

    def reset(self, stream=None) -> None:
        local_hess_reset(self.handle, stream)

    def close(self) -> None:
        if self.handle:
            local_hess_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class IMatrix:
    """imatrix statistic: per-column sums of squares of the activations."""

    def __init__(self, d: int):
        self.d = int(d)
        self.handle = imatrix_create(self.d)

    def add_batch(self, X: torch.Tensor, stream=None) -> None:
        imatrix_add(self.handle, X, self.d, stream)

    def read(self, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        if out is None:
            out = torch.empty(self.d, dtype=torch.float32, device="cuda")
        imatrix_read(self.handle, out, stream)
        return out

    @property
    def n_tokens(self) -> int:
        return imatrix_token_count(self.handle)

    def reset(self, stream=None) -> None:
        imatrix_reset(self.handle, stream)

    def close(self) -> None:
        if self.handle:
            imatrix_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
