"""The allocation-free local-Hessian entry point, through the C ABI.

local_hess_compute_noalloc serves callers that may not allocate device
memory while they run (memory reserved up front by a pooling allocator, or
a runtime that forbids the synchronisation cudaMalloc/cudaFree can cause).
It keeps its fp64 scratch in a fixed array inside the library, so this test
checks three things: two calls in a row each give the same block Hessians
as the handle-based entry points (local_hess_create / add / read, which
allocate) and as the float64 oracle, within the tolerance of the other
local tests, also at the largest width the scratch holds (d = 16,384); a
call leaves the device's free memory unchanged; wider inputs are refused.

This file is collected last so that a run stopping at the first failure
has run every other test before it.
"""

import ctypes

import numpy as np
import pytest
import torch

from helpers import TOL_BF16, block_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from gptq_qqq_calibration_gb300 import build as b
    b.build()
    from gptq_qqq_calibration_gb300 import _lib
    return _lib.load()


def _handle_result(lib, X, d):
    from gptq_qqq_calibration_gb300._lib import HESS_OK
    h = ctypes.c_void_p()
    assert lib.local_hess_create(d, 16, ctypes.byref(h)) == HESS_OK
    s = torch.cuda.current_stream().cuda_stream
    assert lib.local_hess_add(h, X.data_ptr(), X.shape[0], d, 16, 0, s) == HESS_OK
    out = torch.empty((d // 16, 16, 16), dtype=torch.float32, device="cuda")
    assert lib.local_hess_read(h, out.data_ptr(), s) == HESS_OK
    torch.cuda.synchronize()
    assert lib.local_hess_destroy(h) == HESS_OK
    return out.cpu().numpy()


def _noalloc_result(lib, X, d, out):
    from gptq_qqq_calibration_gb300._lib import HESS_OK
    s = torch.cuda.current_stream().cuda_stream
    st = lib.local_hess_compute_noalloc(X.data_ptr(), X.shape[0], d, 16, 0, out.data_ptr(), s)
    assert st == HESS_OK, lib.hess_last_error()
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _oracle(X, d):
    from oracle import LocalGramOracle
    from helpers import host
    o = LocalGramOracle(d)
    o.add_batch(host(X))
    return o.read()


def test_noalloc_matches_handle_path_on_two_calls_in_a_row(lib):
    from gptq_qqq_calibration_gb300.synthetic import make_batch
    d = 1024
    xs = [make_batch(n, d, 900 + k, profile="student_t_every16", profile_seed=9, device="cuda")
          for k, n in enumerate((3000, 517))]
    refs = [_handle_result(lib, X, d) for X in xs]
    out = torch.empty((d // 16, 16, 16), dtype=torch.float32, device="cuda")
    got0 = _noalloc_result(lib, xs[0], d, out)
    free0, _ = torch.cuda.mem_get_info()
    got1 = _noalloc_result(lib, xs[1], d, out)
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, "the no-alloc entry point changed free device memory"
    # the second call must not carry sums over from the first
    assert block_rel_err(got0, refs[0].astype(np.float64)) <= TOL_BF16
    assert block_rel_err(got1, refs[1].astype(np.float64)) <= TOL_BF16
    # and each call equals the float64 oracle of its own batch
    assert block_rel_err(got0, _oracle(xs[0], d)) <= TOL_BF16
    assert block_rel_err(got1, _oracle(xs[1], d)) <= TOL_BF16


def test_noalloc_at_its_width_limit(lib):
    """d = 16,384 fills the whole scratch array (1,024 blocks): two calls in
    a row, each graded against the float64 oracle of its own batch."""
    from gptq_qqq_calibration_gb300.synthetic import make_batch
    d = 16384
    xs = [make_batch(n, d, 950 + k, profile="student_t", profile_seed=10, device="cuda")
          for k, n in enumerate((300, 129))]
    out = torch.empty((d // 16, 16, 16), dtype=torch.float32, device="cuda")
    got0 = _noalloc_result(lib, xs[0], d, out)
    free0, _ = torch.cuda.mem_get_info()
    got1 = _noalloc_result(lib, xs[1], d, out)
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, "the no-alloc entry point changed free device memory"
    assert block_rel_err(got0, _oracle(xs[0], d)) <= TOL_BF16
    assert block_rel_err(got1, _oracle(xs[1], d)) <= TOL_BF16


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    from gptq_qqq_calibration_gb300._lib import HESS_ERR_UNSUPPORTED, HESS_OK
    X = torch.zeros((4, 16400), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((16400 // 16, 16, 16), dtype=torch.float32, device="cuda")
    st = lib.local_hess_compute_noalloc(X.data_ptr(), 4, 16400, 16, 0, out.data_ptr(), None)
    assert st == HESS_ERR_UNSUPPORTED
    assert b"16384" in lib.hess_last_error()
    empty = torch.full((2, 16, 16), 7.0, device="cuda")
    assert lib.local_hess_compute_noalloc(None, 0, 32, 16, 0, empty.data_ptr(), None) == HESS_OK
    torch.cuda.synchronize()
    assert not torch.any(empty)
