"""GPU tests of the companion statistics: merging partial accumulators,
cloning a Hessian (shared-input dedup), checkpoint and resume, and the
imatrix column sums of squares, each against the float64 oracle."""

import numpy as np
import pytest
import torch

from helpers import TOL_BF16, batches, host, rel_err
from oracle import GramOracle, column_sum_of_squares

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gptq_qqq_calibration_gb300 import build as b
    b.build()


def test_merge_of_partials_equals_one_accumulator():
    """Partials built on two streams and merged give the Hessian of all
    tokens, with N the total token count (GPTQModel PR #2979/#2981)."""
    from gptq_qqq_calibration_gb300 import Hessian
    d = 640
    a, b = Hessian(d), Hessian(d)
    o = GramOracle(d)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    xs = list(batches(d, [700, 33, 1000, 5, 250], 61))
    torch.cuda.synchronize()  # the batches are ready before other streams use them
    for k, X in enumerate(xs):
        o.add_batch(host(X))
        with torch.cuda.stream(s1 if k % 2 == 0 else s2):
            (a if k % 2 == 0 else b).add_batch(X, stream=s1 if k % 2 == 0 else s2)
    torch.cuda.synchronize()
    na, nb = a.n_tokens, b.n_tokens
    a.merge(b)
    assert a.n_tokens == na + nb == o.N
    assert b.n_tokens == nb  # src unchanged
    H, damp = a.materialize(0.01)
    a.sync()
    Href, dref = o.materialize(0.01)
    assert rel_err(H.cpu().numpy(), Href) <= TOL_BF16
    assert damp == pytest.approx(dref, rel=TOL_BF16)
    a.close()
    b.close()


def test_merge_rejects_mismatches():
    from gptq_qqq_calibration_gb300 import Hessian, HessError
    a, b = Hessian(64), Hessian(128)
    with pytest.raises(HessError):
        a.merge(b)
    with pytest.raises(HessError):
        a.merge(a)
    a.close()
    b.close()


def test_clone_is_an_independent_copy():
    """A follower's Hessian is a private copy: later batches on the leader do
    not reach it (GPTQModel PR #3052, adopt_hessian_from)."""
    from gptq_qqq_calibration_gb300 import Hessian
    d = 384
    leader = Hessian(d, chunk_tokens=512)
    o = GramOracle(d)
    for X in batches(d, [300, 77], 62):
        leader.add_batch(X)
        o.add_batch(host(X))
    follower = leader.clone()
    assert follower.n_tokens == leader.n_tokens == o.N
    Hf0, _ = follower.materialize(0.0)
    Hf0 = Hf0.cpu().numpy()
    for X in batches(d, [500], 63):
        leader.add_batch(X)
    Hf1, _ = follower.materialize(0.0)
    torch.cuda.synchronize()
    assert np.array_equal(Hf0, Hf1.cpu().numpy())
    assert rel_err(Hf0, o.hessian()) <= TOL_BF16
    assert leader.n_tokens == o.N + 500 and follower.n_tokens == o.N
    # the follower keeps accumulating on its own
    Y = next(batches(d, [64], 64))
    follower.add_batch(Y)
    o.add_batch(host(Y))
    H2, _ = follower.materialize(0.0)
    follower.sync()
    assert rel_err(H2.cpu().numpy(), o.hessian()) <= TOL_BF16
    leader.close()
    follower.close()


@pytest.mark.parametrize("where", ["cpu", "cuda"])
def test_checkpoint_resume_equals_an_uninterrupted_run(where):
    """A run exported after part A and resumed in a fresh handle gives, after
    part B, exactly the H of one handle that ran A then B with the same
    flushes; and both match the oracle."""
    from gptq_qqq_calibration_gb300 import Hessian
    d = 384
    a_counts, b_counts = [700, 129, 1], [513, 64]
    xa = list(batches(d, a_counts, 31, "outlier"))
    xb = list(batches(d, b_counts, 32, "outlier"))
    ref = Hessian(d)
    for X in xa:
        ref.add_batch(X)
    ref.flush()
    for X in xb:
        ref.add_batch(X)
    H_ref, _ = ref.materialize(0.01)

    first = Hessian(d)
    for X in xa:
        first.add_batch(X)
    state, n = first.export_state(device=where)
    first.close()
    assert n == sum(a_counts)
    resumed = Hessian(d)
    resumed.add_batch(xb[0])  # dropped by the import
    resumed.import_state(state, n)
    assert resumed.n_tokens == n
    for X in xb:
        resumed.add_batch(X)
    H, _ = resumed.materialize(0.01)
    torch.cuda.synchronize()
    assert torch.equal(H, H_ref)
    o = GramOracle(d)
    for X in xa + xb:
        o.add_batch(host(X))
    Href, _ = o.materialize(0.01)
    assert rel_err(H.cpu().numpy(), Href) <= TOL_BF16
    ref.close()
    resumed.close()


def test_import_rejects_a_state_of_another_width():
    from gptq_qqq_calibration_gb300 import Hessian, HessError
    from gptq_qqq_calibration_gb300._lib import HESS_ERR_INVALID
    small, big = Hessian(256), Hessian(384)
    state, n = small.export_state()
    with pytest.raises(HessError) as ei:
        big.import_state(state, n)
    assert ei.value.status == HESS_ERR_INVALID
    with pytest.raises(HessError):
        small.import_state(state, -1)
    small.close()
    big.close()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("d,counts", [(8, [1, 3]), (4096, [32768, 17]), (1032, [999, 0, 64])])
def test_imatrix_column_sum_of_squares(d, counts, dtype):
    from gptq_qqq_calibration_gb300 import IMatrix
    im = IMatrix(d)
    xs = list(batches(d, counts, 65, profile="loguniform", dtype=dtype))
    for X in xs:
        im.add_batch(X)
    got = im.read().cpu().numpy().astype(np.float64)
    ref, N = column_sum_of_squares([host(X) for X in xs])
    assert im.n_tokens == N
    assert np.max(np.abs(got - ref) / ref) <= 2e-7
    im.reset()
    assert im.n_tokens == 0 and not torch.any(im.read())
    im.close()


def test_imatrix_matches_hessian_diagonal():
    """The column sums of squares are N/2 times the Hessian's diagonal."""
    from gptq_qqq_calibration_gb300 import Hessian, IMatrix
    d = 512
    h, im = Hessian(d), IMatrix(d)
    for X in batches(d, [1000, 3], 66):
        h.add_batch(X)
        im.add_batch(X)
    H, _ = h.materialize(0.0)
    diag = torch.diagonal(H).double().cpu().numpy()
    sq = im.read().double().cpu().numpy()
    np.testing.assert_allclose(diag * h.n_tokens / 2.0, sq, rtol=1e-5)
    h.close()
    im.close()
