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


ALL = [pin_loss_identity, pin_identity_hessian_is_rtn, pin_factor, pin_damp_and_dead]


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
        scales = np.zeros((rows, d // 128 if grouped else 1))
        if not grouped:
            scales[:, 0] = go._scale(np.max(np.abs(W), axis=1), 7.0)
        Wq = np.zeros_like(W)
        loss = 0.0
        for b0 in range(0, d, 128):
            b1 = b0 + 128
            Err = np.zeros((rows, 128))
            if grouped:
                scales[:, b0 // 128] = go._scale(np.max(np.abs(W[:, b0:b1]), axis=1), 7.5)
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


@pytest.mark.parametrize("kind", ["no_divide", "lower_factor", "sign", "no_trailing", "damp_before_dead"])
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
