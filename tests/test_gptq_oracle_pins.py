"""Pins for the quantization-pass oracle (GPTQModel wiki "QQQ", Concepts:
dead columns, damping, upper Cholesky of the inverse, blockwise error
propagation).

* Loss identity: with Delta = W - Wq (dead columns zeroed), the summed loss
  sum err_i^2 / 2 equals 1/2 Delta H_damped Delta^T exactly, because
  Delta = err U and H_damped = U^-1 U^-T.  Any wrong factor, propagation
  coefficient, sign or skipped trailing update breaks it.
* Identity and diagonal Hessians leave nothing to propagate: the result is
  round-to-nearest with the defined scalar quantizer, written here as loops.
* U is upper triangular with a positive diagonal and U^T U H = I.
* Damping and dead columns against explicit loops.
* Planted mistakes in copies of the oracle fail these pins.
"""

import numpy as np
import pytest

from oracle import gptq_oracle as go


def _problem(d=256, rows=24, seed=0, dead=()):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((4 * d, d)) * np.exp(rng.uniform(-1, 1, d))
    H = 2.0 / X.shape[0] * X.T @ X
    for i in dead:
        H[i, :] = 0.0
        H[:, i] = 0.0
    W = rng.standard_normal((rows, d)) * 0.05
    return H, W


def _rtn(W, group_size):
    rows, d = W.shape
    out = np.zeros_like(W)
    for r in range(rows):
        if group_size == -1:
            m = max(abs(v) for v in W[r])
            s = (m if m > 0 else 1.0) / 7.0
            for j in range(d):
                out[r, j] = s * min(7, max(-8, round(W[r, j] / s)))
        else:
            for g in range(0, d, group_size):
                m = max(abs(v) for v in W[r, g:g + group_size])
                s = 2.0 * (m if m > 0 else 1.0) / 15.0
                for j in range(g, g + group_size):
                    out[r, j] = s * (min(15, max(0, round(W[r, j] / s) + 8)) - 8)
    return out


def pin_loss_identity(quantize):
    for group in (128, -1):
        H, W = _problem(seed=3)
        res = quantize(H, W, 0.01, group)
        Hd = H.copy()
        Hd[np.diag_indices(H.shape[0])] += res["damp"]
        Delta = W - res["Wq"]
        quad = 0.5 * np.einsum("ri,ij,rj->", Delta, Hd, Delta)
        assert res["loss"] == pytest.approx(quad, rel=1e-9)


def pin_identity_hessian_is_rtn(quantize):
    for group in (128, -1):
        d = 256
        W = np.random.default_rng(5).standard_normal((6, d))
        res = quantize(np.eye(d) * 3.0, W, 0.01, group)
        np.testing.assert_allclose(res["Wq"], _rtn(W, group), rtol=0, atol=1e-12)
        res = quantize(np.diag(np.linspace(0.5, 4.0, d)), W, 0.01, group)
        np.testing.assert_allclose(res["Wq"], _rtn(W, group), rtol=0, atol=1e-12)


def pin_factor(quantize):
    H, W = _problem(seed=4)
    res = quantize(H, W, 0.02, 128)
    U = res["U"]
    d = H.shape[0]
    assert np.allclose(np.tril(U, -1), 0.0)
    assert np.all(np.diagonal(U) > 0)
    Hd = H.copy()
    Hd[np.diag_indices(d)] += res["damp"]
    np.testing.assert_allclose(U.T @ U @ Hd, np.eye(d), atol=1e-8)


def pin_damp_and_dead(quantize):
    H, W = _problem(seed=6, dead=(3, 200))
    res = quantize(H, W, 0.05, 128)
    d = H.shape[0]
    diag = [1.0 if H[i, i] == 0 else H[i, i] for i in range(d)]
    assert res["damp"] == pytest.approx(0.05 * sum(diag) / d, rel=1e-12)
    assert not res["Wq"][:, 3].any() and not res["Wq"][:, 200].any()
    assert res["dead"][3] and res["dead"][200] and res["dead"].sum() == 2


def _coupled_problem():
    """A factor with one off-diagonal entry, U = I + a e_0 e_128^T (a = -4), so
    that only column 0's error reaches a later column (column 128, the first
    of the second 128-column group/block), and H_damped = U^-1 U^-T with no
    damping.  One row with four nonzero weights."""
    d, a = 256, -4.0
    Uinv = np.eye(d)
    Uinv[0, 128] = -a
    H = Uinv @ Uinv.T  # H[0,0] = 17, H[0,128] = H[128,0] = 4, else identity
    W = np.zeros((1, d))
    w0, w1, w128, w129 = 0.27, 0.5, 0.6, 0.23
    W[0, [0, 1, 128, 129]] = w0, w1, w128, w129
    return H, W, a, (w0, w1, w128, w129)


def pin_scale_timing_on_a_coupled_example(quantize):
    """The scale readings of "Whole-row and grouped weight quantization"
    (GPTQModel wiki "QQQ") on a case worked by hand.  Column 0's error
    err0 = w0 - q0 (U_00 = 1) changes column 128 to w128 - a err0 before the
    second block starts, and that raises the row's and the second group's
    largest magnitude.
      * grouped: the second group's scale comes from the updated column
        (2 max(|w128 - a err0|, |w129|) / 15), not from the original W;
      * whole-row: the one scale max|w| / 7 is taken before any column is
        quantized and kept for every block (it is not re-taken from the
        updated row)."""
    H, W, a, (w0, w1, w128, w129) = _coupled_problem()

    def rnd(x):  # round half to even, as the pages' torch.round
        return float(np.rint(x))

    # grouped, group 128: centered 4-bit codes c = clamp(round(w/s) + 8, 0, 15) - 8
    def code_g(w, s):
        return min(15.0, max(0.0, rnd(w / s) + 8.0)) - 8.0
    s0 = 2.0 * max(abs(w0), abs(w1)) / 15.0
    q0 = s0 * code_g(w0, s0)
    w128u = w128 - a * (w0 - q0)
    s1 = 2.0 * max(abs(w128u), abs(w129)) / 15.0
    res = quantize(H, W, 0.0, 128)
    assert res["scales"][0, 0] == pytest.approx(s0, rel=1e-12)
    assert res["scales"][0, 1] == pytest.approx(s1, rel=1e-12)
    want = {0: q0, 1: s0 * code_g(w1, s0), 128: s1 * code_g(w128u, s1), 129: s1 * code_g(w129, s1)}
    for j, v in want.items():
        assert res["Wq"][0, j] == pytest.approx(v, abs=1e-12), j

    # whole row: signed 4-bit codes c = clamp(round(w/s), -8, 7), one scale
    def code_r(w, s):
        return min(7.0, max(-8.0, rnd(w / s)))
    s = max(abs(w0), abs(w1), abs(w128), abs(w129)) / 7.0
    q0 = s * code_r(w0, s)
    w128u = w128 - a * (w0 - q0)
    res = quantize(H, W, 0.0, -1)
    assert res["scales"][0, 0] == pytest.approx(s, rel=1e-12)
    want = {0: q0, 1: s * code_r(w1, s), 128: s * code_r(w128u, s), 129: s * code_r(w129, s)}
    for j, v in want.items():
        assert res["Wq"][0, j] == pytest.approx(v, abs=1e-12), j


ALL = [pin_loss_identity, pin_identity_hessian_is_rtn, pin_factor, pin_damp_and_dead,
       pin_scale_timing_on_a_coupled_example]


@pytest.mark.parametrize("pin", ALL, ids=lambda f: f.__name__)
def test_gptq_oracle_pin(pin):
    pin(go.gptq_quantize)


def test_gptq_beats_round_to_nearest():
    """Error compensation lowers the Hessian-weighted error (the point of
    the quadratic objective)."""
    H, W = _problem(seed=8, rows=32)
    res = go.gptq_quantize(H, W, 0.01, 128)
    Hd = H + res["damp"] * np.eye(H.shape[0])
    D = W - _rtn(W, 128)
    assert res["loss"] < 0.5 * np.einsum("ri,ij,rj->", D, Hd, D)


# ---------------------------------------------------------- planted mistakes

def _mutant(kind):
    def q(H, W, damp, group, dtype=np.float64, U=None):
        H = np.array(H, dtype=np.float64)
        W = np.array(W, dtype=np.float64)
        d = H.shape[0]
        dead = np.diagonal(H) == 0
        if kind != "damp_before_dead":
            H[dead, dead] = 1.0
        damp_v = damp * float(np.mean(np.diagonal(H)))
        H[np.diag_indices(d)] += damp_v
        if kind == "damp_before_dead":
            H[dead, dead] = 1.0
        W[:, dead] = 0.0
        U = go.upper_cholesky_of_inverse(H)
        if kind == "lower_factor":
            U = np.linalg.cholesky(np.linalg.inv(H))
        grouped = group == 128
        rows = W.shape[0]
        W_orig = W.copy()
        scales = np.zeros((rows, d // 128 if grouped else 1))
        if not grouped:
            scales[:, 0] = go._scale(np.max(np.abs(W), axis=1), 7.0)
        Wq = np.zeros_like(W)
        loss = 0.0
        for b0 in range(0, d, 128):
            b1 = b0 + 128
            Err = np.zeros((rows, 128))
            if grouped:
                src = W_orig if kind == "group_scale_from_original" else W
                scales[:, b0 // 128] = go._scale(np.max(np.abs(src[:, b0:b1]), axis=1), 7.5)
            elif kind == "row_scale_per_block":
                scales[:, 0] = go._scale(np.max(np.abs(W), axis=1), 7.0)
            s = scales[:, b0 // 128 if grouped else 0]
            for i in range(b0, b1):
                w = W[:, i]
                wq, _ = go.quantize_column(w, s, grouped)
                Wq[:, i] = wq
                dii = U[i, i]
                err = (w - wq) / (1.0 if kind == "no_divide" else dii)
                loss += float(np.sum(((w - wq) / dii) ** 2) / 2.0)
                sign = -1.0 if kind == "sign" else 1.0
                W[:, i + 1:b1] -= sign * np.outer(err, U[i, i + 1:b1])
                Err[:, i - b0] = err
            if b1 < d and kind != "no_trailing":
                W[:, b1:] -= Err @ U[b0:b1, b1:]
        return {"Wq": Wq, "scales": scales, "damp": damp_v, "loss": loss, "U": U, "dead": dead}
    return q


@pytest.mark.parametrize("kind", ["no_divide", "lower_factor", "sign", "no_trailing", "damp_before_dead",
                                  "group_scale_from_original", "row_scale_per_block"])
def test_pins_catch_planted_mistakes(kind):
    failed = 0
    for pin in ALL:
        try:
            pin(_mutant(kind))
        except (AssertionError, np.linalg.LinAlgError):
            failed += 1
    assert failed, kind


def test_codes_and_average_loss():
    """Wq = scale * code with codes in [-8, 7]; the average loss divides the
    summed loss by the token count."""
    H, W = _problem(seed=9)
    for group in (128, -1):
        res = go.gptq_quantize(H, W, 0.01, group, n_tokens=1000)
        s = np.repeat(res["scales"], 128, axis=1) if group == 128 else res["scales"]
        np.testing.assert_array_equal(res["Wq"], s * res["codes"])
        assert res["codes"].min() >= -8 and res["codes"].max() <= 7
        assert res["avg_loss"] == res["loss"] / 1000
        # Wpre is what each column held when quantized: the code is its
        # rounded quotient by the scale
        q = np.clip(np.rint(res["Wpre"] / s), -8, 7)
        np.testing.assert_array_equal(q, res["codes"])
