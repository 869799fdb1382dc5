"""GPU parity of the CUDA path against the float64 oracle, small sizes (and
the widest layers, on sampled columns).

Every call goes through the C ABI (ctypes binding).  Sizes span several
128x128 tiles, ragged token tails (n not a multiple of 128, n = 1), widths
that are not multiples of the tile (136, 8), empty batches, several fused
flushes, every split-K/chunk setting, and the degenerate N = 0 case.
"""

import ctypes

import numpy as np
import pytest
import torch

from helpers import TOL_BF16, TOL_F32, batches, block_rel_err, host, rel_err
from oracle import GramOracle, LocalGramOracle, column_sum_of_squares, gram_columns

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gptq_qqq_calibration_gb300 import build as b
    b.build()


def _run(d, counts, seed, damp=0.01, profile="normal", dtype=torch.bfloat16, **opts):
    from gptq_qqq_calibration_gb300 import Hessian
    h = Hessian(d, **opts)
    o = GramOracle(d)
    for X in batches(d, counts, seed, profile, dtype=dtype):
        h.add_batch(X)
        o.add_batch(host(X))
    H, dv = h.materialize(damp)
    h.sync()
    Href, dref = o.materialize(damp)
    assert h.n_tokens == o.N
    Hn = H.cpu().numpy()
    h.close()
    return Hn, dv, Href, dref


@pytest.mark.parametrize("pair", [1, 0])
@pytest.mark.parametrize("d,counts", [
    (256, [128, 128, 128, 128]),
    (136, [1, 63, 64, 65, 200]),
    (8, [5, 70]),
    (16, [1]),
    (384, [333, 0, 1, 130]),
    (640, [1000]),
])
def test_bf16_matches_oracle(d, counts, pair):
    H, dv, Href, dref = _run(d, counts, seed=d, pair_kernel=pair)
    assert rel_err(H, Href) <= TOL_BF16
    assert np.array_equal(H, H.T), "H_out must be bit-exactly symmetric"
    assert dv == pytest.approx(dref, rel=TOL_BF16)


@pytest.mark.parametrize("opts", [
    dict(chunk_tokens=128), dict(chunk_tokens=384, split_k=3), dict(split_k=7),
    dict(grid=4), dict(grid=2, chunk_tokens=128), dict(flush_tokens=1),
    dict(max_pending=3, chunk_tokens=4096), dict(split_k=40),
    dict(pair_kernel=0), dict(pair_kernel=0, split_k=3, grid=5),
    dict(pair_kernel=0, grid=1, chunk_tokens=384), dict(pair_kernel=0, flush_tokens=1),
    # single-slab flushes of the low part with the last wave's tiles split in
    # halves (10 tiles on 4 or 3 CTAs), and with every flush folding
    dict(grid=4, flush_tokens=1), dict(grid=3, flush_tokens=1, chunk_tokens=128),
    dict(grid=4, flush_tokens=1, fold_every=1), dict(flush_tokens=1, fold_every=3),
    dict(flush_tokens=1, overlap_launches=0),
])
def test_bf16_schedules(opts):
    H, dv, Href, dref = _run(512, [700, 1, 64, 129, 512, 33], seed=11, **opts)
    assert rel_err(H, Href) <= TOL_BF16
    assert np.array_equal(H, H.T)


@pytest.mark.parametrize("opts", [dict(split_k=1), dict(split_k=7), dict(split_k=40),
                                  dict(split_k=1, pair_kernel=1), dict(split_k=40, pair_kernel=1),
                                  dict(split_k=1, dtype=torch.float32), dict(split_k=40, dtype=torch.float32),
                                  dict(split_k=1, flush_tokens=2000, fold_every=8, ulps=2.5),
                                  dict(split_k=1, flush_tokens=2000, fold_every=2, ulps=2.0),
                                  dict(split_k=1, flush_tokens=2000, fold_every=3, pair_kernel=1, ulps=2.0)])
def test_accumulation_is_exact_on_integer_data(opts):
    """Integer activations in [-64, 64] make every product and every
    tensor-memory chain exact (chain sums stay below 2^24), so the only
    rounding left is in the (hi, lo) accumulator, whose entries grow past
    2^24.  The single-slab read-modify-write of both parts and the
    compensated atomics of split-K launches must both keep the exact integer
    sum: H then equals the oracle's exact sum times 2/N to within one fp32
    ulp (a lost rounding error of an fp32 add would show as an error of
    several ulps).  A flush that updates the low part alone rounds once
    (0.5 ulp of a partial sum: only the diagonal sums pass 2^24 here, and
    they grow monotonically, so at most 0.5 ulp of the total); a later fold
    keeps that error.  With k such flushes the bound is 1 + k/2 ulp: the
    three flushes here are low-part flushes with a fold every 8th flush
    (2.5 ulp), and two of them with a fold every 2nd or 3rd (2 ulp)."""
    from gptq_qqq_calibration_gb300 import Hessian
    opts = dict(opts)
    dtype = opts.pop("dtype", torch.bfloat16)
    ulps = opts.pop("ulps", 1.0)
    opts.setdefault("fold_every", 1)
    opts.setdefault("flush_tokens", 1 << 20)
    d, counts = 384, [6000, 5000, 3000]
    h = Hessian(d, **opts)
    o = GramOracle(d)
    g = torch.Generator(device="cuda").manual_seed(29)
    for n in counts:
        X = torch.randint(-64, 65, (n, d), generator=g, device="cuda").to(dtype)
        h.add_batch(X)
        o.add_batch(host(X))
    H, _ = h.materialize(0.0)
    h.sync()
    H = H.cpu().numpy().astype(np.float64)
    h.close()
    Href, _ = o.materialize(0.0)
    assert np.abs(o.S).max() > 2 ** 24  # the accumulator must round in fp32
    ulp = np.spacing(np.abs(Href).astype(np.float32)).astype(np.float64)
    err = np.abs(H - Href) / ulp
    assert err.max() <= ulps, f"max {err.max():.2f} ulp"


@pytest.mark.parametrize("d,counts", [
    (256, [128, 128, 128, 128]),
    (136, [1, 31, 32, 33, 200]),
    (8, [5, 70]),
    (384, [333, 0, 1, 130]),
    (640, [1000, 77]),
])
def test_f32_matches_oracle(d, counts):
    H, dv, Href, dref = _run(d, counts, seed=d + 7, dtype=torch.float32)
    assert rel_err(H, Href) <= TOL_F32
    assert np.array_equal(H, H.T)
    assert dv == pytest.approx(dref, rel=TOL_F32)


@pytest.mark.parametrize("opts", [dict(chunk_tokens=128), dict(split_k=5), dict(grid=3),
                                  dict(flush_tokens=1), dict(chunk_tokens=2048),
                                  dict(grid=4, flush_tokens=1), dict(grid=3, flush_tokens=1, fold_every=2)])
def test_f32_schedules(opts):
    H, dv, Href, dref = _run(512, [700, 1, 32, 129, 512, 33], seed=17, dtype=torch.float32, **opts)
    assert rel_err(H, Href) <= TOL_F32


def test_f32_loguniform_channels():
    """The fp32 workload's channel profile (per-channel std log-uniform in
    [0.1, 10]) at the fp32 bound."""
    H, _, Href, _ = _run(512, [2000, 999], seed=20, profile="loguniform", dtype=torch.float32)
    assert rel_err(H, Href) <= TOL_F32


def test_f32_outlier_channels_within_bf16_bound():
    """With channels 20x the rest (diagonal 80x the mean) the remaining
    round-toward-zero bias of the 32-token hi*hi chains is ~1.2e-5 of the mean
    diagonal: above the fp32 bound, which no fp32 workload here asks for on
    such data, and well inside the bf16 bound."""
    H, _, Href, _ = _run(768, [2000, 1500, 37], seed=19, profile="outlier", dtype=torch.float32)
    assert rel_err(H, Href) <= TOL_BF16


def test_mixed_dtypes_in_one_handle():
    """bf16 and fp32 batches may alternate; a dtype switch flushes (H is fp32
    either way, Model-Optimizer PR #3002)."""
    from gptq_qqq_calibration_gb300 import Hessian
    d = 384
    h = Hessian(d)
    o = GramOracle(d)
    for k, n in enumerate((300, 17, 1000, 64)):
        dt = torch.bfloat16 if k % 2 == 0 else torch.float32
        X = next(batches(d, [n], 40 + k, dtype=dt))
        h.add_batch(X)
        o.add_batch(host(X))
    H, _ = h.materialize(0.0)
    h.sync()
    assert h.n_tokens == o.N
    assert rel_err(H.cpu().numpy(), o.hessian()) <= TOL_BF16
    h.close()


def test_f32_path_on_upcast_bf16_equals_bf16_path():
    """bf16 -> fp32 is exact, so both kernels see the same numbers."""
    from gptq_qqq_calibration_gb300 import Hessian
    d = 512
    xs = list(batches(d, [900, 33, 1200], 41))
    hb, hf = Hessian(d), Hessian(d)
    for X in xs:
        hb.add_batch(X)
        hf.add_batch(X.float())
    Hb, _ = hb.materialize(0.0)
    Hf, _ = hf.materialize(0.0)
    torch.cuda.synchronize()
    m = float(torch.diagonal(Hf).mean())
    assert float((Hb - Hf).abs().max()) <= TOL_BF16 * m
    hb.close()
    hf.close()


def test_many_small_batches_fused_into_few_flushes():
    rng = np.random.default_rng(5)
    counts = rng.integers(1, 50, size=420)
    H, dv, Href, dref = _run(256, counts, seed=12, damp=0.005)
    assert rel_err(H, Href) <= TOL_BF16


def test_outlier_channels():
    H, dv, Href, dref = _run(768, [2000, 1500, 37], seed=13, profile="outlier")
    assert rel_err(H, Href) <= TOL_BF16


def test_empty_and_zero_tokens():
    from gptq_qqq_calibration_gb300 import Hessian
    h = Hessian(64)
    h.add_batch(torch.empty((0, 64), dtype=torch.bfloat16, device="cuda"))
    assert h.n_tokens == 0
    H, dv = h.materialize(0.01)
    assert dv == 0.0 and not torch.any(H)
    X = torch.randn(10, 64, device="cuda").to(torch.bfloat16)
    h.add_batch(X)
    h.add_batch(torch.empty((0, 64), dtype=torch.bfloat16, device="cuda"))
    assert h.n_tokens == 10
    h.close()


def test_materialize_is_not_destructive_and_reset_clears():
    from gptq_qqq_calibration_gb300 import Hessian
    d = 256
    h = Hessian(d)
    o = GramOracle(d)
    for k, X in enumerate(batches(d, [100, 200, 300], 21)):
        h.add_batch(X)
        o.add_batch(host(X))
        H, dv = h.materialize(0.01)
        Href, dref = o.materialize(0.01)
        assert rel_err(H.cpu().numpy(), Href) <= TOL_BF16
    h.reset()
    assert h.n_tokens == 0
    X = next(batches(d, [77], 22))
    h.add_batch(X)
    o2 = GramOracle(d)
    o2.add_batch(host(X))
    H, _ = h.materialize(0.0)
    assert rel_err(H.cpu().numpy(), o2.hessian()) <= TOL_BF16
    h.close()


def test_batches_from_another_stream():
    from gptq_qqq_calibration_gb300 import Hessian
    d = 256
    h = Hessian(d)
    o = GramOracle(d)
    side = torch.cuda.Stream()
    for k in range(6):
        with torch.cuda.stream(side):
            X = torch.randn(300 + k, d, device="cuda").to(torch.bfloat16)
            h.add_batch(X, stream=side)
        side.synchronize()
        o.add_batch(host(X))
    H, _ = h.materialize(0.0)
    torch.cuda.synchronize()
    assert rel_err(H.cpu().numpy(), o.hessian()) <= TOL_BF16
    h.close()


def test_add_batch_allocates_no_device_memory():
    from gptq_qqq_calibration_gb300 import Hessian
    d = 1024
    h = Hessian(d)
    xs = [torch.randn(2000, d, device="cuda").to(torch.bfloat16) for _ in range(4)]
    out = torch.empty((d, d), device="cuda")
    h.add_batch(xs[0])
    h.materialize(0.0, out=out)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    a0 = torch.cuda.memory_allocated()
    for X in xs:
        h.add_batch(X)
    h.flush()
    h.materialize(0.01, out=out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == a0
    assert free1 == free0
    h.close()


def test_invalid_pointer_alignment_is_rejected():
    from gptq_qqq_calibration_gb300 import _lib
    L = _lib.load()
    from gptq_qqq_calibration_gb300 import hess_create, hess_destroy
    h = hess_create(64)
    buf = torch.zeros(1024, dtype=torch.bfloat16, device="cuda")
    assert L.hess_add_batch(h, buf.data_ptr() + 2, 4, 0, None) == _lib.HESS_ERR_INVALID
    assert L.hess_add_batch(h, buf.data_ptr(), -1, 0, None) == _lib.HESS_ERR_INVALID
    assert L.hess_add_batch(h, buf.data_ptr(), 4, 7, None) == _lib.HESS_ERR_INVALID
    assert L.hess_token_count(h) == 0
    hess_destroy(h)


def test_host_buffers_are_refused_before_any_launch():
    """Every entry point that takes activations or an output buffer refuses
    host memory (pageable or pinned) with INVALID and leaves the handle
    usable: a wrong pointer must not reach a kernel."""
    from gptq_qqq_calibration_gb300 import _lib
    from gptq_qqq_calibration_gb300 import (hess_create, hess_destroy, imatrix_create, local_hess_create)
    L = _lib.load()
    d = 64
    for pinned in (False, True):
        Xh = torch.ones((32, d), dtype=torch.bfloat16)
        Oh = torch.zeros((d, d), dtype=torch.float32)
        if pinned:
            Xh, Oh = Xh.pin_memory(), Oh.pin_memory()
        h = hess_create(d)
        assert L.hess_add_batch(h, Xh.data_ptr(), 32, 0, None) == _lib.HESS_ERR_INVALID
        assert b"host memory" in L.hess_last_error()
        assert L.hess_token_count(h) == 0
        assert L.hess_materialize(h, Oh.data_ptr(), 0.0, None, None) == _lib.HESS_ERR_INVALID
        X = Xh.cuda()
        assert L.hess_add_batch(h, X.data_ptr(), 32, 0, None) == _lib.HESS_OK
        H = torch.empty((d, d), dtype=torch.float32, device="cuda")
        assert L.hess_materialize(h, H.data_ptr(), 0.0, None, None) == _lib.HESS_OK
        torch.cuda.synchronize()
        assert torch.allclose(H, torch.full_like(H, 2.0))  # (2/32) * 32 * 1 * 1
        hess_destroy(h)
        m = imatrix_create(d)
        assert L.imatrix_add(m, Xh.data_ptr(), 32, 0, None) == _lib.HESS_ERR_INVALID
        assert L.imatrix_destroy(m) == _lib.HESS_OK
        lh = local_hess_create(d)
        assert L.local_hess_add(lh, Xh.data_ptr(), 32, d, 16, 0, None) == _lib.HESS_ERR_INVALID
        assert L.local_hess_destroy(lh) == _lib.HESS_OK
        Lo = torch.zeros((d // 16, 16, 16), dtype=torch.float32)
        assert L.local_hess_compute_noalloc(X.data_ptr(), 32, d, 16, 0, Lo.data_ptr(), None) == _lib.HESS_ERR_INVALID
        assert L.local_hess_compute_noalloc(Xh.data_ptr(), 32, d, 16, 0, Lo.cuda().data_ptr(), None) == \
            _lib.HESS_ERR_INVALID


def test_chunk_option_is_whole_pipeline_stages():
    """bf16 chunks are whole 128-token pipeline stages: other lengths are
    rejected before any launch, and the handle stays usable."""
    from gptq_qqq_calibration_gb300 import Hessian, HessError
    from gptq_qqq_calibration_gb300._lib import HESS_ERR_INVALID
    h = Hessian(256)
    for bad in (0, 64, 200, 65536 + 128):
        with pytest.raises(HessError) as ei:
            h.set_option("chunk_tokens", bad)
        assert ei.value.status == HESS_ERR_INVALID
    for good in (128, 384, 65536):
        h.set_option("chunk_tokens", good)
    h.close()


def test_device_wait_limit_reports_timeout_and_handle_recovers():
    """A zero wait limit makes the kernel's first unsatisfied wait give up;
    the kernel drains its copies, frees tensor memory and returns, and the
    host reads HESS_ERR_TIMEOUT.  The handle then works again."""
    from gptq_qqq_calibration_gb300 import Hessian, HessError
    from gptq_qqq_calibration_gb300._lib import HESS_ERR_TIMEOUT
    d = 512
    h = Hessian(d, wait_timeout_ns=0)
    X = torch.randn(4096, d, device="cuda").to(torch.bfloat16)
    h.add_batch(X)
    h.flush()
    with pytest.raises(HessError) as ei:
        h.sync()
    assert ei.value.status == HESS_ERR_TIMEOUT
    h.reset()
    h.set_option("wait_timeout_ns", 2_000_000_000)
    o = GramOracle(d)
    h.add_batch(X)
    o.add_batch(host(X))
    H, _ = h.materialize(0.0)
    h.sync()
    assert rel_err(H.cpu().numpy(), o.hessian()) <= TOL_BF16
    h.close()


# ------------------------------------------------------------------ local


def _run_local(d, counts, seed, profile="normal"):
    from gptq_qqq_calibration_gb300 import LocalHessian
    lh = LocalHessian(d)
    lo = LocalGramOracle(d)
    for X in batches(d, counts, seed, profile):
        lh.add_batch(X)
        lo.add_batch(host(X))
    L = lh.read()
    lh.sync()
    assert lh.n_tokens == lo.N
    Ln = L.cpu().numpy()
    lh.close()
    return Ln, lo.read()


@pytest.mark.parametrize("d,counts", [
    (16, [1, 5]), (272, [63, 64, 65]), (512, [1000]), (4096, [257, 0, 31]), (1040, [2048, 3]),
])
def test_local_matches_oracle(d, counts):
    L, Lref = _run_local(d, counts, seed=d + 1)
    assert block_rel_err(L, Lref) <= TOL_BF16
    assert np.array_equal(L, np.transpose(L, (0, 2, 1)))


def test_local_heavy_tailed_channels():
    L, Lref = _run_local(1024, [4096, 4096], seed=5, profile="student_t_every16")
    assert block_rel_err(L, Lref) <= TOL_BF16


def test_local_blocks_equal_diagonal_blocks_of_full_hessian():
    from gptq_qqq_calibration_gb300 import Hessian, LocalHessian
    d = 512
    h, lh = Hessian(d), LocalHessian(d)
    for X in batches(d, [900, 37], 31):
        h.add_batch(X)
        lh.add_batch(X)
    H, _ = h.materialize(0.0)
    L = lh.read().cpu().numpy()
    H = H.cpu().numpy()
    m = np.mean(np.diagonal(H))
    for b in range(d // 16):
        assert np.abs(L[b] - H[16 * b:16 * b + 16, 16 * b:16 * b + 16]).max() <= 2 * TOL_BF16 * m
    h.close()
    lh.close()


def test_local_zero_and_reset():
    from gptq_qqq_calibration_gb300 import LocalHessian
    lh = LocalHessian(64)
    assert not torch.any(lh.read())
    lh.add_batch(torch.randn(10, 64, device="cuda").to(torch.bfloat16))
    assert lh.n_tokens == 10
    lh.reset()
    assert lh.n_tokens == 0 and not torch.any(lh.read())
    lh.close()


@pytest.mark.parametrize("d,counts,dtype", [
    (16376, [300, 77, 1], torch.bfloat16),
    (12296, [40, 129], torch.float32),
    (32768, [200, 56], torch.bfloat16),
    (32760, [129], torch.float32),
])
def test_wide_ragged_width(d, counts, dtype):
    """The widest layers: 8,256 upper tiles at d = 16,376, with a last tile
    row 120 wide (d is a multiple of 8 but not of 128), and the largest width
    a handle takes, d = 32,768 (32,896 upper tiles, a 4.3 GB accumulator),
    with its ragged neighbour 32,760.  The oracle computes a seeded sample of
    whole columns, the last column included, and the full diagonal (which
    fixes the damping)."""
    from gptq_qqq_calibration_gb300 import Hessian
    cols = np.sort(np.concatenate([np.random.default_rng(7).choice(d - 1, 11, replace=False), [d - 1]]))
    h = Hessian(d)
    S = np.zeros((d, cols.size))
    sq = np.zeros(d)
    N = 0
    for X in batches(d, counts, seed=31, dtype=dtype):
        h.add_batch(X)
        Xh = host(X)
        part, n = gram_columns([Xh], cols)
        S += part
        sq += column_sum_of_squares([Xh])[0]
        N += n
    H, damp = h.materialize(0.01)
    h.sync()
    assert h.n_tokens == N == sum(counts)
    scale = 2.0 / N
    mean_diag = sq.mean() * scale
    ref = S * scale
    ref[cols, np.arange(cols.size)] += 0.01 * mean_diag
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    got = H[:, torch.from_numpy(cols).cuda()].cpu().numpy().astype(np.float64)
    assert np.abs(got - ref).max() / mean_diag <= tol
    diag = torch.diagonal(H).cpu().numpy().astype(np.float64)
    assert np.abs(diag - (sq * scale + 0.01 * mean_diag)).max() / mean_diag <= tol
    assert damp == pytest.approx(0.01 * mean_diag, rel=tol)
    rows = H[torch.from_numpy(cols).cuda(), :].cpu().numpy()
    assert np.array_equal(rows.T, got.astype(np.float32))
    h.close()


def test_one_handle_fed_from_several_host_threads():
    """Calls on one handle are serialised by its mutex: four host threads
    add 80 ragged batches at once, each on its own CUDA stream, through the
    C ABI (ctypes releases the interpreter lock during the call); two others
    poll the token count meanwhile.  The sum must be the oracle's whatever
    the order, and N must count every token once."""
    import threading
    from gptq_qqq_calibration_gb300 import _lib, hess_create, hess_destroy
    L = _lib.load()
    d = 384
    counts = np.random.default_rng(41).integers(1, 700, size=80)
    xs = list(batches(d, counts, seed=42))
    torch.cuda.synchronize()
    o = GramOracle(d)
    for X in xs:
        o.add_batch(host(X))
    h = hess_create(d)
    L.hess_set_option(h, _lib.OPTIONS["flush_tokens"], 3000)  # many flushes while threads race
    streams = [torch.cuda.Stream() for _ in range(4)]
    errors = []
    stop = threading.Event()

    def feed(k):
        for X in xs[k::4]:
            st = L.hess_add_batch(h, X.data_ptr(), X.shape[0], 0, streams[k].cuda_stream)
            if st != _lib.HESS_OK:
                errors.append((k, st, L.hess_last_error()))

    def poll():
        while not stop.is_set():
            if L.hess_token_count(h) < 0:
                errors.append(("count",))

    pollers = [threading.Thread(target=poll) for _ in range(2)]
    feeders = [threading.Thread(target=feed, args=(k,)) for k in range(4)]
    for t in pollers + feeders:
        t.start()
    for t in feeders:
        t.join()
    stop.set()
    for t in pollers:
        t.join()
    assert not errors, errors
    assert L.hess_token_count(h) == int(counts.sum())
    H = torch.empty((d, d), dtype=torch.float32, device="cuda")
    assert L.hess_materialize(h, H.data_ptr(), 0.0, None, None) == _lib.HESS_OK
    assert L.hess_sync(h, None) == _lib.HESS_OK
    torch.cuda.synchronize()
    assert rel_err(H.cpu().numpy(), o.hessian()) <= TOL_BF16
    hess_destroy(h)
