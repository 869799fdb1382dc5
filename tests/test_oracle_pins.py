"""Pins for the float64 oracle: facts fixed by the pages and by mathematics.

Each check here is independent of the oracle's own code path: exact rational
arithmetic, the worked example printed in GPTQModel PR #3052's review,
closed forms written as explicit loops, and invariants of the definition
``H = (2/N) sum_t x_t x_t^T`` (GPTQModel PR #2979 Summary, PR #2981
Validation) with damping ``damp_percent * mean(diag H)`` (GPTQModel wiki
"QQQ", Concepts, step 3).  ``test_pins_catch_planted_mistakes`` plants a
mistake in copies of the oracle and checks that some pin fails for each.
"""

import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import GramOracle, LocalGramOracle, column_sum_of_squares, gram_columns
from gptq_qqq_calibration_gb300.synthetic import make_batch, to_float64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
U64 = 2.0 ** -53


def _rand_bf16(n, d, seed, scale=1.0):
    return to_float64(make_batch(n, d, seed, dtype=torch.bfloat16) * 1) * scale


def _rand_f32(n, d, seed):
    return to_float64(make_batch(n, d, seed, dtype=torch.float32))


def _exact_gram(batches, d):
    S = [[Fraction(0)] * d for _ in range(d)]
    N = 0
    for X in batches:
        for row in X:
            fr = [Fraction(float(v)) for v in row]
            for i in range(d):
                for j in range(d):
                    S[i][j] += fr[i] * fr[j]
            N += 1
    return S, N


# ---------------------------------------------------------------------------
# pin functions, parameterised by the oracle classes so that planted mistakes
# can be run through the same checks


def pin_exact_rational(Oracle, seed=0):
    """Brute force with exact rationals on tiny inputs (bf16 and fp32)."""
    for maker in (_rand_bf16, _rand_f32):
        for d, sizes in ((1, (1,)), (3, (5, 2)), (8, (7, 0, 9, 16))):
            batches = [maker(n, d, seed * 97 + 13 * k + d) for k, n in enumerate(sizes)]
            o = Oracle(d)
            for X in batches:
                o.add_batch(X)
            S_ex, N_ex = _exact_gram(batches, d)
            assert o.N == N_ex
            H = o.hessian()
            for i in range(d):
                for j in range(d):
                    exact = S_ex[i][j] * Fraction(2, N_ex)
                    mag = sum(abs(Fraction(float(X[t, i])) * Fraction(float(X[t, j])))
                              for X in batches for t in range(X.shape[0])) * Fraction(2, N_ex)
                    bound = float(mag) * (N_ex + 2) * U64 * 2 + 1e-300
                    assert abs(Fraction(float(H[i, j])) - exact) <= Fraction(bound), (i, j)


def pin_worked_example(Oracle):
    """GPTQModel PR #3052 review, finding P2: fp16 1.0009765625, one token."""
    with open(os.path.join(GOLDEN, "staging_worked_example.json")) as f:
        g = json.load(f)
    x16 = torch.tensor([[g["input_fp16"]]], dtype=torch.float16)
    assert float(x16) == g["input_fp16"]  # representable in fp16
    o32 = Oracle(1)
    o32.add_batch(to_float64(x16.to(torch.float32)))
    assert o32.N == g["n_tokens"]
    h32 = np.float32(o32.hessian()[0, 0])  # H is stored fp32
    assert float(h32) == g["H_fp32_staging"]
    o16 = Oracle(1)
    o16.add_batch(to_float64(x16.to(torch.bfloat16)))
    assert float(np.float32(o16.hessian()[0, 0])) == g["H_bf16_staging"]


def pin_diag_sum_of_squares(Oracle):
    """diag(H)_i = (2/N) sum_t x_{t,i}^2, as a plain loop."""
    d = 5
    batches = [_rand_f32(n, d, 40 + n) for n in (3, 11, 1)]
    o = Oracle(d)
    for X in batches:
        o.add_batch(X)
    N = sum(X.shape[0] for X in batches)
    for i in range(d):
        s = 0.0
        for X in batches:
            for t in range(X.shape[0]):
                s += X[t, i] * X[t, i]
        assert o.hessian()[i, i] == pytest.approx(2.0 * s / N, rel=1e-14)


def pin_offdiag_loop(Oracle):
    """H_ij = (2/N) sum_t x_{t,i} x_{t,j} for i != j, as a plain loop."""
    d = 4
    X = _rand_f32(9, d, 77)
    o = Oracle(d)
    o.add_batch(X[:4])
    o.add_batch(X[4:])
    for i in range(d):
        for j in range(d):
            s = sum(X[t, i] * X[t, j] for t in range(9))
            assert o.hessian()[i, j] == pytest.approx(2.0 * s / 9, rel=1e-13, abs=1e-15)


def pin_damping(Oracle):
    """Damping adds damp * mean(diag H) to the diagonal only (QQQ wiki)."""
    d = 6
    X = _rand_f32(20, d, 5) * np.arange(1, d + 1)
    o = Oracle(d)
    o.add_batch(X)
    H = o.hessian()
    Hd, damp = o.materialize(0.01)
    # mean of the scaled diagonal, written out as a loop
    m = sum(2.0 * sum(X[t, i] ** 2 for t in range(20)) / 20 for i in range(d)) / d
    assert damp == pytest.approx(0.01 * m, rel=1e-13)
    off = ~np.eye(d, dtype=bool)
    assert np.array_equal(Hd[off], H[off])
    assert np.allclose(np.diagonal(Hd) - np.diagonal(H), damp, rtol=1e-12, atol=0)


def pin_empty_batch(Oracle):
    """An empty batch changes neither H nor N (PR #2981, Validation)."""
    d = 4
    o = Oracle(d)
    X = _rand_bf16(6, d, 3)
    o.add_batch(X)
    H0, N0 = o.hessian().copy(), o.N
    o.add_batch(np.zeros((0, d)))
    assert o.N == N0
    assert np.array_equal(o.hessian(), H0)
    e = Oracle(d)
    e.add_batch(np.zeros((0, d)))
    assert e.N == 0 and not e.hessian().any()


def pin_multibatch_equals_concat(Oracle):
    """Several batches give the closed form over their concatenation."""
    d = 16
    batches = [_rand_bf16(n, d, 200 + n) for n in (1, 17, 64, 3)]
    o = Oracle(d)
    for X in batches:
        o.add_batch(X)
    Xc = np.concatenate(batches)
    ref = (2.0 / Xc.shape[0]) * np.einsum("ti,tj->ij", Xc, Xc)
    assert o.N == Xc.shape[0]
    np.testing.assert_allclose(o.hessian(), ref, rtol=1e-13, atol=1e-13)


def pin_duplicate_and_permute(Oracle):
    """Duplicating every batch leaves H unchanged; token order is irrelevant;
    permuting features permutes H."""
    d = 12
    X = _rand_bf16(40, d, 9)
    a = Oracle(d)
    a.add_batch(X)
    b = Oracle(d)
    b.add_batch(X)
    b.add_batch(X)
    assert b.N == 2 * a.N
    np.testing.assert_allclose(b.hessian(), a.hessian(), rtol=1e-15, atol=0)
    rng = np.random.default_rng(1)
    c = Oracle(d)
    c.add_batch(X[rng.permutation(40)])
    np.testing.assert_allclose(c.hessian(), a.hessian(), rtol=1e-14, atol=1e-14)
    p = rng.permutation(d)
    e = Oracle(d)
    e.add_batch(X[:, p])
    np.testing.assert_allclose(e.hessian(), a.hessian()[np.ix_(p, p)], rtol=1e-14, atol=1e-14)


def pin_symmetric_psd(Oracle):
    d = 32
    o = Oracle(d)
    o.add_batch(_rand_f32(50, d, 8))
    H = o.hessian()
    np.testing.assert_allclose(H, H.T, rtol=1e-15, atol=0)
    w = np.linalg.eigvalsh(H)
    assert w.min() >= -64 * U64 * np.abs(w).max() * d


def pin_statistics(Oracle):
    """Unit-variance inputs give diag(H) near 2 (Model-Optimizer PR #3002,
    Testing: "the diagonal is about 2")."""
    d = 64
    o = Oracle(d)
    o.add_batch(_rand_f32(4096, d, 11))
    diag = np.diagonal(o.hessian())
    assert abs(diag.mean() - 2.0) < 0.03
    off = o.hessian()[~np.eye(d, dtype=bool)]
    assert np.abs(off).max() < 6 * 2 / np.sqrt(4096)


def pin_local_exact(LocalOracle):
    """Local 16x16 blocks by exact rationals, scaled by 2/N."""
    d, blk = 32, 16
    batches = [_rand_bf16(n, d, 500 + n) for n in (3, 0, 5)]
    lo = LocalOracle(d, blk)
    for X in batches:
        lo.add_batch(X)
    N = 8
    assert lo.N == N
    L = lo.read()
    for b in range(d // blk):
        for i in range(blk):
            for j in range(blk):
                ex = Fraction(0)
                for X in batches:
                    for t in range(X.shape[0]):
                        ex += Fraction(float(X[t, b * blk + i])) * Fraction(float(X[t, b * blk + j]))
                ex *= Fraction(2, N)
                assert abs(Fraction(float(L[b, i, j])) - ex) <= abs(ex) * Fraction(2 ** -50) + Fraction(1, 2 ** 1000)


def pin_local_vs_full(LocalOracle, Oracle):
    """Block b of the local Hessian is the b-th 16x16 diagonal block of H."""
    d = 64
    X = _rand_bf16(33, d, 21)
    lo = LocalOracle(d, 16)
    lo.add_batch(X)
    o = Oracle(d)
    o.add_batch(X)
    H = o.hessian()
    for b in range(4):
        np.testing.assert_allclose(lo.read()[b], H[16 * b:16 * b + 16, 16 * b:16 * b + 16], rtol=1e-14, atol=1e-14)


ALL_PINS = [
    pin_exact_rational, pin_worked_example, pin_diag_sum_of_squares, pin_offdiag_loop,
    pin_damping, pin_empty_batch, pin_multibatch_equals_concat, pin_duplicate_and_permute,
    pin_symmetric_psd, pin_statistics,
]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_gram_oracle_pin(pin):
    pin(GramOracle)


def test_local_oracle_exact():
    pin_local_exact(LocalGramOracle)


def test_local_oracle_matches_full_diagonal_blocks():
    pin_local_vs_full(LocalGramOracle, GramOracle)


def test_column_helpers_match_full_gram():
    d = 24
    batches = [_rand_bf16(n, d, 70 + n) for n in (5, 0, 31)]
    o = GramOracle(d)
    for X in batches:
        o.add_batch(X)
    cols = [0, 7, 23]
    S, N = gram_columns(batches, cols)
    assert N == o.N
    np.testing.assert_allclose(S, o.S[:, cols], rtol=1e-14, atol=1e-14)
    sq, N2 = column_sum_of_squares(batches)
    assert N2 == o.N
    np.testing.assert_allclose(sq, np.diagonal(o.S), rtol=1e-14)


# ---------------------------------------------------------------------------
# planted mistakes: each mutant must fail at least one pin


class _CountsBatches(GramOracle):
    def add_batch(self, X):
        X = np.asarray(X, dtype=np.float64).reshape(-1, self.d)
        if X.shape[0] == 0:
            return
        self.S += X.T @ X
        self.N += 1


class _DropsTwo(GramOracle):
    def hessian(self):
        return self.S / self.N if self.N else np.zeros_like(self.S)


class _DampsUnscaled(GramOracle):
    def materialize(self, damp_percent):
        H = self.hessian().copy()
        damp = damp_percent * float(np.mean(np.diagonal(self.S)))
        H[np.diag_indices(self.d)] += damp
        return H, damp


class _DampsEverything(GramOracle):
    def materialize(self, damp_percent):
        H = self.hessian()
        damp = damp_percent * float(np.mean(np.diagonal(H)))
        return H + damp, damp


class _WrongIndex(GramOracle):
    def add_batch(self, X):
        X = np.asarray(X, dtype=np.float64).reshape(-1, self.d)
        if X.shape[0] == 0:
            return
        self.S += X.T @ np.roll(X, 1, axis=1)
        self.N += X.shape[0]


class _CountsEmpty(GramOracle):
    def add_batch(self, X):
        X = np.asarray(X, dtype=np.float64).reshape(-1, self.d)
        if X.shape[0] == 0:
            self.N += 1
            return
        super().add_batch(X)


class _SignFlip(GramOracle):
    def add_batch(self, X):
        X = np.asarray(X, dtype=np.float64).reshape(-1, self.d)
        if X.shape[0] == 0:
            return
        self.S += X.T @ X - 2 * np.triu(X.T @ X, 1)
        self.N += X.shape[0]


class _MeanOverAll(GramOracle):
    def materialize(self, damp_percent):
        H = self.hessian().copy()
        damp = damp_percent * float(np.mean(H))
        H[np.diag_indices(self.d)] += damp
        return H, damp


MUTANTS = [_CountsBatches, _DropsTwo, _DampsUnscaled, _DampsEverything, _WrongIndex,
           _CountsEmpty, _SignFlip, _MeanOverAll]


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda c: c.__name__)
def test_pins_catch_planted_mistakes(mutant):
    failed = []
    for pin in ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"{mutant.__name__} passed every pin"


class _LocalNoScale(LocalGramOracle):
    def read(self):
        return self.S.copy()


class _LocalShifted(LocalGramOracle):
    def add_batch(self, X):
        X = np.asarray(X, dtype=np.float64).reshape(-1, self.d)
        if X.shape[0] == 0:
            return
        for b in range(self.nb):
            Xb = X[:, b * self.block:(b + 1) * self.block]
            Xn = X[:, ((b + 1) % self.nb) * self.block:((b + 1) % self.nb + 1) * self.block]
            self.S[b] += Xb.T @ Xn
        self.N += X.shape[0]


@pytest.mark.parametrize("mutant", [_LocalNoScale, _LocalShifted], ids=lambda c: c.__name__)
def test_local_pins_catch_planted_mistakes(mutant):
    with pytest.raises(AssertionError):
        pin_local_exact(mutant)
        pin_local_vs_full(mutant, GramOracle)
