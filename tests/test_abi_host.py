"""Host-side checks of the C ABI (no GPU needed).

The library must load, export every function ``include/*.h`` declares, and
reject invalid arguments before any CUDA call.
"""

import ctypes
import glob
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hess.h")


@pytest.fixture(scope="module")
def lib():
    from gptq_qqq_calibration_gb300 import build as b
    b.build()
    from gptq_qqq_calibration_gb300 import _lib
    return _lib.load()


def declared_functions():
    text = "\n".join(open(p).read() for p in sorted(glob.glob(os.path.join(ROOT, "include", "*.h"))))
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("hess_create", "hess_add_batch", "hess_materialize", "local_hess_add", "hess_destroy",
              "gptq_create", "gptq_prepare", "gptq_quantize"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from gptq_qqq_calibration_gb300 import _lib
    names = declared_functions()
    assert set(names) == set(_lib.PROTOTYPES), "binding prototypes and header disagree"
    for n in names:
        assert hasattr(lib, n), n


def test_abi_version(lib):
    text = open(HEADER).read()
    v = int(re.search(r"#define HESS_ABI_VERSION (\d+)", text).group(1))
    assert lib.hess_abi_version() == v


def test_invalid_arguments_rejected_before_cuda(lib):
    from gptq_qqq_calibration_gb300._lib import HESS_ERR_INVALID, HESS_ERR_UNSUPPORTED
    h = ctypes.c_void_p()
    assert lib.hess_create(0, ctypes.byref(h)) == HESS_ERR_INVALID
    assert lib.hess_create(-8, ctypes.byref(h)) == HESS_ERR_INVALID
    assert lib.hess_create(12, ctypes.byref(h)) == HESS_ERR_UNSUPPORTED
    assert b"multiple of 8" in lib.hess_last_error()
    assert lib.hess_create(32776, ctypes.byref(h)) == HESS_ERR_UNSUPPORTED  # widest is 32,768
    assert b"exceeds 32768" in lib.hess_last_error()
    assert lib.hess_create(8, None) == HESS_ERR_INVALID
    assert lib.hess_add_batch(None, None, 4, 0, None) == HESS_ERR_INVALID
    assert lib.hess_flush(None, None) == HESS_ERR_INVALID
    assert lib.hess_materialize(None, None, 0.01, None, None) == HESS_ERR_INVALID
    assert lib.hess_set_option(None, 1, 5) == HESS_ERR_INVALID
    assert lib.hess_token_count(None) == -1
    assert lib.hess_destroy(None) == 0
    assert lib.local_hess_create(64, 8, ctypes.byref(h)) == HESS_ERR_UNSUPPORTED
    assert lib.local_hess_create(40, 16, ctypes.byref(h)) == HESS_ERR_UNSUPPORTED
    assert lib.local_hess_add(None, None, 0, 16, 16, 0, None) == HESS_ERR_INVALID
    assert lib.local_hess_destroy(None) == 0
    g = ctypes.c_void_p()
    assert lib.gptq_create(0, 4, ctypes.byref(g)) == HESS_ERR_INVALID
    assert lib.gptq_create(256, -1, ctypes.byref(g)) == HESS_ERR_INVALID
    assert lib.gptq_create(200, 4, ctypes.byref(g)) == HESS_ERR_UNSUPPORTED
    assert b"multiple of 128" in lib.hess_last_error()
    assert lib.gptq_create(256, 4, None) == HESS_ERR_INVALID
    assert lib.gptq_prepare(None, None, 0, 0.01, None, None) == HESS_ERR_INVALID
    assert lib.gptq_prepare_hess(None, None, 0.01, None, None) == HESS_ERR_INVALID
    assert lib.gptq_read_factor(None, None, None) == HESS_ERR_INVALID
    assert lib.gptq_quantize(None, None, 0, 0, 128, None, None, None, None, None) == HESS_ERR_INVALID
    assert lib.gptq_destroy(None) == 0


def test_more_entry_points_reject_bad_arguments_before_cuda(lib):
    """Merge, clone, checkpoint, imatrix and the allocation-free local call
    refuse NULL handles and impossible sizes on the host, before any CUDA
    call (this container has no GPU)."""
    from gptq_qqq_calibration_gb300._lib import HESS_ERR_INVALID, HESS_ERR_UNSUPPORTED
    h = ctypes.c_void_p()
    n = ctypes.c_int64()
    assert lib.hess_merge(None, None, None) == HESS_ERR_INVALID
    assert lib.hess_clone(None, ctypes.byref(h), None) == HESS_ERR_INVALID
    assert lib.hess_clone(None, None, None) == HESS_ERR_INVALID
    assert lib.hess_state_bytes(None) == 0
    assert lib.hess_export_state(None, None, 0, None, ctypes.byref(n)) == HESS_ERR_INVALID
    assert lib.hess_import_state(None, None, 0, 0, None) == HESS_ERR_INVALID
    assert lib.hess_pending_batches(None) == -1
    assert lib.hess_kernel_launches(None) == -1
    assert lib.hess_dim(None) == -1
    assert lib.hess_sync(None, None) == HESS_ERR_INVALID
    assert lib.hess_reset(None, None) == HESS_ERR_INVALID
    assert lib.imatrix_create(0, ctypes.byref(h)) == HESS_ERR_INVALID
    assert lib.imatrix_add(None, None, 4, 0, None) == HESS_ERR_INVALID
    assert lib.imatrix_read(None, None, None) == HESS_ERR_INVALID
    assert lib.imatrix_token_count(None) == -1
    assert lib.imatrix_destroy(None) == 0
    assert lib.local_hess_read(None, None, None) == HESS_ERR_INVALID
    assert lib.local_hess_token_count(None) == -1
    out = ctypes.c_void_p(16)  # never dereferenced: each call fails before any CUDA call
    assert lib.local_hess_compute_noalloc(None, -1, 64, 16, 0, out, None) == HESS_ERR_INVALID
    assert lib.local_hess_compute_noalloc(None, 4, 0, 16, 0, out, None) == HESS_ERR_INVALID
    assert lib.local_hess_compute_noalloc(None, 4, 64, 16, 0, None, None) == HESS_ERR_INVALID
    assert lib.local_hess_compute_noalloc(None, 4, 64, 8, 0, out, None) == HESS_ERR_UNSUPPORTED
    assert lib.local_hess_compute_noalloc(None, 4, 72, 16, 0, out, None) == HESS_ERR_UNSUPPORTED
    assert lib.local_hess_compute_noalloc(None, 4, 64, 16, 1, out, None) == HESS_ERR_UNSUPPORTED
    assert lib.local_hess_compute_noalloc(None, 4, 64, 16, 9, out, None) == HESS_ERR_INVALID
    assert lib.local_hess_compute_noalloc(None, 4, 64, 16, 0, out, None) == HESS_ERR_INVALID  # X NULL
    assert b"X is NULL" in lib.hess_last_error()


def test_status_codes_match_header():
    from gptq_qqq_calibration_gb300 import _lib
    text = open(HEADER).read()
    enum = dict((k, int(v)) for k, v in re.findall(r"(HESS_(?:OK|ERR_\w+))\s*=\s*(\d+)", text))
    assert enum == {v: k for k, v in _lib.STATUS_NAMES.items()}


def test_injected_allocation_failure_reports_oom():
    # In a child process so the environment knob stays local.
    code = (
        "import ctypes, sys; sys.path.insert(0, %r)\n"
        "from gptq_qqq_calibration_gb300 import _lib\n"
        "L = _lib.load(); h = ctypes.c_void_p()\n"
        "assert L.hess_create(256, ctypes.byref(h)) == _lib.HESS_ERR_OOM\n"
        "assert h.value is None\n"
        "assert L.local_hess_create(256, 16, ctypes.byref(h)) == _lib.HESS_ERR_OOM\n"
        "print('ok')\n" % ROOT)
    env = dict(os.environ, HESS_FAULT="alloc")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and "ok" in r.stdout, r.stderr
