"""ctypes loader for ``libgptq_hess.so`` and the prototypes of ``include/*.h``.

Loading never falls back to anything: if the library is missing the caller
gets a RuntimeError naming the build step.
"""

from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgptq_hess.so")

HESS_BF16, HESS_F32 = 0, 1
(HESS_OK, HESS_ERR_INVALID, HESS_ERR_UNSUPPORTED, HESS_ERR_OOM, HESS_ERR_CUDA, HESS_ERR_TIMEOUT,
 HESS_ERR_NOT_PD, HESS_ERR_INTERNAL) = range(8)
STATUS_NAMES = {0: "HESS_OK", 1: "HESS_ERR_INVALID", 2: "HESS_ERR_UNSUPPORTED", 3: "HESS_ERR_OOM",
                4: "HESS_ERR_CUDA", 5: "HESS_ERR_TIMEOUT", 6: "HESS_ERR_NOT_PD", 7: "HESS_ERR_INTERNAL"}
OPTIONS = {"flush_tokens": 1, "max_pending": 2, "chunk_tokens": 3, "wait_timeout_ns": 4,
           "split_k": 5, "grid": 6, "pair_kernel": 7, "fold_every": 8,
           "overlap_launches": 9}

_vp, _i32, _i64, _f64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
_fp = ctypes.POINTER(ctypes.c_float)

# name -> (restype, argtypes); mirrors include/hess.h and include/gptq.h
PROTOTYPES = {
    "hess_create": (_i32, [_i64, ctypes.POINTER(_vp)]),
    "hess_add_batch": (_i32, [_vp, _vp, _i64, _i32, _vp]),
    "hess_flush": (_i32, [_vp, _vp]),
    "hess_materialize": (_i32, [_vp, _vp, _f64, _vp, _fp]),
    "hess_token_count": (_i64, [_vp]),
    "hess_pending_batches": (_i64, [_vp]),
    "hess_kernel_launches": (_i64, [_vp]),
    "hess_dim": (_i64, [_vp]),
    "hess_sync": (_i32, [_vp, _vp]),
    "hess_reset": (_i32, [_vp, _vp]),
    "hess_set_option": (_i32, [_vp, _i32, _i64]),
    "hess_destroy": (_i32, [_vp]),
    "hess_merge": (_i32, [_vp, _vp, _vp]),
    "hess_clone": (_i32, [_vp, ctypes.POINTER(_vp), _vp]),
    "hess_state_bytes": (_i64, [_vp]),
    "hess_export_state": (_i32, [_vp, _vp, _i64, _vp, ctypes.POINTER(_i64)]),
    "hess_import_state": (_i32, [_vp, _vp, _i64, _i64, _vp]),
    "imatrix_create": (_i32, [_i64, ctypes.POINTER(_vp)]),
    "imatrix_add": (_i32, [_vp, _vp, _i64, _i32, _vp]),
    "imatrix_read": (_i32, [_vp, _vp, _vp]),
    "imatrix_token_count": (_i64, [_vp]),
    "imatrix_reset": (_i32, [_vp, _vp]),
    "imatrix_destroy": (_i32, [_vp]),
    "local_hess_create": (_i32, [_i64, _i32, ctypes.POINTER(_vp)]),
    "local_hess_add": (_i32, [_vp, _vp, _i64, _i64, _i32, _i32, _vp]),
    "local_hess_read": (_i32, [_vp, _vp, _vp]),
    "local_hess_token_count": (_i64, [_vp]),
    "local_hess_sync": (_i32, [_vp, _vp]),
    "local_hess_reset": (_i32, [_vp, _vp]),
    "local_hess_destroy": (_i32, [_vp]),
    "local_hess_compute_noalloc": (_i32, [_vp, _i64, _i64, _i32, _i32, _vp, _vp]),
    "gptq_create": (_i32, [_i64, _i64, ctypes.POINTER(_vp)]),
    "gptq_prepare": (_i32, [_vp, _vp, _i64, _f64, _vp, _fp]),
    "gptq_prepare_hess": (_i32, [_vp, _vp, _f64, _vp, _fp]),
    "gptq_read_factor": (_i32, [_vp, _vp, _vp]),
    "gptq_quantize": (_i32, [_vp, _vp, _i32, _i64, _i32, _vp, _vp, _vp, _vp, ctypes.POINTER(_f64)]),
    "gptq_destroy": (_i32, [_vp]),
    "hess_last_error": (ctypes.c_char_p, []),
    "hess_abi_version": (_i32, []),
}


class HessError(RuntimeError):
    """A non-OK status from the library, with its message."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build the CUDA library first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in PROTOTYPES.items():
                fn = getattr(lib, name)
                fn.restype, fn.argtypes = res, args
            _lib = lib
    return _lib


def check(status: int) -> None:
    if status != HESS_OK:
        msg = load().hess_last_error()
        raise HessError(status, msg.decode(errors="replace") if msg else "")
