"""GPU tests of the host-side ordering and lifetime rules of the Hessian
handle: what a clone copies while another thread adds, when a borrowed batch
may be reused by the caching allocator, and how a device-side timeout reaches
a caller that does not wait.

The sums are graded against the float64 oracle (GPTQModel PR #2981,
Validation: the accumulated result equals 2/N X^T X over the batches it
counts)."""

import threading

import numpy as np
import pytest
import torch

from helpers import TOL_BF16, batches, host, rel_err
from oracle import GramOracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gptq_qqq_calibration_gb300 import build as b
    b.build()


def test_clone_while_another_thread_adds():
    """A clone holds exactly the batches its token count counts: the flush,
    the copy of the sums and the read of N happen under one hold of the
    source's mutex, while a second host thread keeps adding batches on its
    own stream.  Both threads call the C ABI directly (ctypes releases the
    interpreter lock), so the handle's mutex is the only thing ordering
    them.  Every clone must equal the oracle over the prefix of batches that
    its N names."""
    import ctypes

    from gptq_qqq_calibration_gb300 import _lib, hess_create, hess_destroy
    L = _lib.load()
    d = 256
    counts = np.random.default_rng(31).integers(1, 200, size=800)
    xs = list(batches(d, counts, seed=31))
    torch.cuda.synchronize()
    src = hess_create(d)
    assert L.hess_set_option(src, _lib.OPTIONS["flush_tokens"], 3000) == _lib.HESS_OK
    s_add, s_clone = torch.cuda.Stream(), torch.cuda.Stream()
    clones, errors = [], []
    # Clone j starts once the adder has begun batch 50 j and runs while it
    # adds batches 50 j .. 50 j + 49; the adder then waits for it, so every
    # clone lands at a different point of the stream, in the middle of adds.
    n_clones = 15
    reached = [threading.Event() for _ in range(n_clones)]
    done = [threading.Event() for _ in range(n_clones)]

    def adder():
        for k, X in enumerate(xs):
            j = k // 50
            if k % 50 == 0 and j < n_clones:
                reached[j].set()
            st = L.hess_add_batch(src, X.data_ptr(), X.shape[0], 0, s_add.cuda_stream)
            if st != _lib.HESS_OK:
                errors.append(("add", st, L.hess_last_error()))
            if k % 50 == 49 and j < n_clones:
                done[j].wait(60)

    def cloner():
        for j in range(n_clones):
            reached[j].wait(60)
            out = ctypes.c_void_p()
            st = L.hess_clone(src, ctypes.byref(out), s_clone.cuda_stream)
            if st != _lib.HESS_OK:
                errors.append(("clone", st, L.hess_last_error()))
            else:
                clones.append(out.value)
            done[j].set()

    ta, tc = threading.Thread(target=adder), threading.Thread(target=cloner)
    ta.start()
    tc.start()
    ta.join(120)
    tc.join(120)
    assert not ta.is_alive() and not tc.is_alive()
    assert not errors, errors
    torch.cuda.synchronize()
    prefix = np.concatenate([[0], np.cumsum(counts)])
    assert L.hess_token_count(src) == prefix[-1]
    want = {}
    for c in clones:
        n = L.hess_token_count(c)
        k = int(np.searchsorted(prefix, n))
        assert prefix[k] == n, "a clone's N must end on a batch boundary"
        want.setdefault(k, []).append(c)
    assert len(want) >= 4, f"the clones should see several prefixes of the stream: {sorted(want)}"
    o = GramOracle(d)
    done_k = 0
    H = torch.empty((d, d), dtype=torch.float32, device="cuda")
    for k in sorted(want):
        for X in xs[done_k:k]:
            o.add_batch(host(X))
        done_k = k
        Href = o.hessian()
        for c in want[k]:
            assert L.hess_materialize(c, H.data_ptr(), 0.0, None, None) == _lib.HESS_OK
            assert L.hess_sync(c, None) == _lib.HESS_OK
            if k == 0:
                assert not torch.any(H)
            else:
                assert rel_err(H.cpu().numpy(), Href) <= TOL_BF16, f"clone at {k} batches"
            hess_destroy(c)
    hess_destroy(src)


def test_flushed_batch_is_not_reused_before_its_side_stream_flush_runs():
    """A batch flushed on a side stream stays reserved for that stream.  The
    side stream is held back by a sleep kernel, the caller drops its only
    reference to X, and a new tensor of the same size is allocated and
    filled on the default stream without any synchronisation.  If X's
    memory were handed out before the flush read it, the fill would land
    in the Gram."""
    from gptq_qqq_calibration_gb300 import Hessian
    d, n = 512, 4096
    X = next(batches(d, [n], seed=33))
    Xh = host(X)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    h = Hessian(d)
    with torch.cuda.stream(side):
        torch.cuda._sleep(100_000_000)  # ~50 ms of the side stream
    h.add_batch(X, stream=side)
    h.flush(stream=side)
    del X
    Y = torch.full((n, d), 1000.0, dtype=torch.bfloat16, device="cuda")
    H, _ = h.materialize(0.0, stream=side)
    h.sync(stream=side)
    o = GramOracle(d)
    o.add_batch(Xh)
    assert rel_err(H.cpu().numpy(), o.hessian()) <= TOL_BF16
    del Y
    h.close()


def test_timeout_reaches_a_caller_that_does_not_wait():
    """With a zero wait limit the flush inside materialize gives up.  A
    materialize that asks for no damping value does not wait, but the
    status word follows its work to the host; once the stream has drained,
    the next call on the handle fails with HESS_ERR_TIMEOUT before doing
    anything, and keeps failing until reset.  After reset the handle is
    exact again."""
    from gptq_qqq_calibration_gb300 import Hessian, HessError
    from gptq_qqq_calibration_gb300._lib import HESS_ERR_TIMEOUT
    d = 512
    X = torch.randn(4096, d, device="cuda").to(torch.bfloat16)
    h = Hessian(d, wait_timeout_ns=0)
    h.add_batch(X)
    h.materialize(0.0, want_damp=False)
    torch.cuda.synchronize()
    n_before = h.n_tokens
    for call in (lambda: h.add_batch(X), lambda: h.flush(), lambda: h.materialize(0.0, want_damp=False)):
        with pytest.raises(HessError) as ei:
            call()
        assert ei.value.status == HESS_ERR_TIMEOUT
    assert h.n_tokens == n_before, "a refused add must not count its tokens"
    h.reset()
    h.set_option("wait_timeout_ns", 2_000_000_000)
    o = GramOracle(d)
    h.add_batch(X)
    o.add_batch(host(X))
    H, _ = h.materialize(0.0, want_damp=False)
    torch.cuda.synchronize()
    h.sync()
    assert rel_err(H.cpu().numpy(), o.hessian()) <= TOL_BF16
    h.close()


def test_first_call_on_a_new_host_thread_flushes():
    """A host thread whose first CUDA call is the library's: an add_batch
    that flushes at once (one batch, one stream, so nothing else binds a
    context before the tensor map is encoded).  The library binds the
    device's primary context for its driver calls; the call succeeds and
    the sum is the oracle's."""
    from gptq_qqq_calibration_gb300 import _lib, hess_create, hess_destroy
    L = _lib.load()
    d = 384
    X = next(batches(d, [700], seed=35))
    torch.cuda.synchronize()
    h = hess_create(d)
    assert L.hess_set_option(h, _lib.OPTIONS["flush_tokens"], 1) == _lib.HESS_OK
    res = []

    def worker():
        res.append((L.hess_add_batch(h, X.data_ptr(), X.shape[0], 0, None), L.hess_last_error()))

    t = threading.Thread(target=worker)
    t.start()
    t.join(60)
    assert res and res[0][0] == _lib.HESS_OK, res
    H = torch.empty((d, d), dtype=torch.float32, device="cuda")
    assert L.hess_materialize(h, H.data_ptr(), 0.0, None, None) == _lib.HESS_OK
    assert L.hess_sync(h, None) == _lib.HESS_OK
    o = GramOracle(d)
    o.add_batch(host(X))
    assert rel_err(H.cpu().numpy(), o.hessian()) <= TOL_BF16
    hess_destroy(h)


def test_injected_descriptor_failure_leaves_no_trace(monkeypatch):
    """HESS_FAULT=encode makes the tensor-map encoding of a flush fail (as
    if the driver refused the descriptor).  The add_batch whose flush fails
    returns HESS_ERR_UNSUPPORTED and leaves no trace (its batch neither
    queued nor counted); the batches queued before it stay queued, and an
    explicit flush fails the same way.  Once the fault is gone, the same
    calls sum everything exactly once."""
    from gptq_qqq_calibration_gb300 import Hessian, HessError
    from gptq_qqq_calibration_gb300._lib import HESS_ERR_UNSUPPORTED
    d = 256
    X1, X2 = batches(d, [300, 800], seed=37)
    h = Hessian(d, flush_tokens=1000)
    h.add_batch(X1)
    assert h.n_tokens == 300
    monkeypatch.setenv("HESS_FAULT", "encode")
    with pytest.raises(HessError) as ei:
        h.add_batch(X2)  # 1,100 pending tokens: this call flushes
    assert ei.value.status == HESS_ERR_UNSUPPORTED
    assert h.n_tokens == 300
    from gptq_qqq_calibration_gb300.hessian import hess_pending_batches
    assert hess_pending_batches(h.handle) == 1
    with pytest.raises(HessError) as ei:
        h.flush()
    assert ei.value.status == HESS_ERR_UNSUPPORTED
    monkeypatch.delenv("HESS_FAULT")
    h.add_batch(X2)
    assert h.n_tokens == 1100
    H, _ = h.materialize(0.0)
    h.sync()
    o = GramOracle(d)
    o.add_batch(host(X1))
    o.add_batch(host(X2))
    assert rel_err(H.cpu().numpy(), o.hessian()) <= TOL_BF16
    h.close()
