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
    source's lock, while a second thread keeps adding batches on its own
    stream.  Every clone must equal the oracle over the prefix of batches
    that its N names."""
    from gptq_qqq_calibration_gb300 import Hessian
    d = 256
    counts = np.random.default_rng(31).integers(1, 200, size=800)
    xs = list(batches(d, counts, seed=31))
    torch.cuda.synchronize()
    src = Hessian(d, flush_tokens=3000)
    clones = []
    # Clone j runs while the adder adds batches 50 j .. 50 j + 49; the adder
    # then waits for it, so the clones land at different points of the stream.
    n_clones = 15
    done = [threading.Event() for _ in range(n_clones)]

    def adder():
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            for k, X in enumerate(xs):
                src.add_batch(X, stream=s)
                j = k // 50
                if k % 50 == 49 and j < n_clones:
                    done[j].wait(60)

    def cloner():
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            for j in range(n_clones):
                clones.append(src.clone(stream=s))
                done[j].set()

    ta, tc = threading.Thread(target=adder), threading.Thread(target=cloner)
    ta.start()
    tc.start()
    ta.join(120)
    tc.join(120)
    assert not ta.is_alive() and not tc.is_alive()
    torch.cuda.synchronize()
    prefix = np.concatenate([[0], np.cumsum(counts)])
    assert src.n_tokens == prefix[-1]
    want = {}
    for c in clones:
        k = int(np.searchsorted(prefix, c.n_tokens))
        assert prefix[k] == c.n_tokens, "a clone's N must end on a batch boundary"
        want.setdefault(k, []).append(c)
    assert len(want) >= 4, f"the clones should see several prefixes of the stream: {sorted(want)}"
    o = GramOracle(d)
    done = 0
    for k in sorted(want):
        for X in xs[done:k]:
            o.add_batch(host(X))
        done = k
        Href = o.hessian()
        for c in want[k]:
            H, _ = c.materialize(0.0)
            c.sync()
            if k == 0:
                assert not torch.any(H)
            else:
                assert rel_err(H.cpu().numpy(), Href) <= TOL_BF16, f"clone at {k} batches"
            c.close()
    src.close()


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
