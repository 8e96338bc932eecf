"""Pins of the oracle's backward (``kda_backward``) against central finite differences of
the forward oracle in fp64: the directional derivative of
L = sum(d_out * out) + sum(d_final_state * final_state) along a random direction of each
input equals the gradient's inner product with that direction.  The finite differences
use only ``kda_forward``, so they are independent of the backward's own arithmetic."""
import numpy as np
import pytest

from oracle import kda_backward, kda_forward

NAMES = ("q", "k", "v", "g", "beta_logits", "a_log", "dt_bias", "initial_state")
GRAD = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta_logits": "dbeta_logits",
        "a_log": "da_log", "dt_bias": "ddt_bias", "initial_state": "dinitial_state"}


def case(seed, B=2, T=9, H=2, dk=5, dv=3):
    r = np.random.default_rng(700 + seed)
    x = {"q": r.normal(size=(B, T, H, dk)), "k": r.normal(size=(B, T, H, dk)),
         "v": r.normal(size=(B, T, H, dv)), "g": r.normal(size=(B, T, H, dk)),
         "beta_logits": r.normal(size=(B, T, H)), "a_log": r.uniform(-1, 1, size=H),
         "dt_bias": r.normal(size=(dk, H)) * 0.3, "initial_state": r.normal(size=(B, H, dk, dv))}
    cot = {"d_out": r.normal(size=(B, T, H, dv)), "d_final_state": r.normal(size=(B, H, dk, dv))}
    return x, cot


def loss(x, cot, scale, lb, order, with_final=True):
    out, fs = kda_forward(x["q"], x["k"], x["v"], x["g"], x["beta_logits"], x["a_log"],
                          x["dt_bias"], scale, lb, x["initial_state"], order)
    val = np.sum(cot["d_out"] * out)
    if with_final:
        val += np.sum(cot["d_final_state"] * fs)
    return val


def grads(x, cot, scale, lb, order, with_final=True):
    return kda_backward(x["q"], x["k"], x["v"], x["g"], x["beta_logits"], x["a_log"],
                        x["dt_bias"], cot["d_out"], cot["d_final_state"] if with_final else None,
                        scale, lb, x["initial_state"], order)


def directional(x, cot, name, direction, scale, lb, order, with_final, h=1e-5):
    xp = dict(x); xm = dict(x)
    xp[name] = x[name] + h * direction
    xm[name] = x[name] - h * direction
    return (loss(xp, cot, scale, lb, order, with_final) -
            loss(xm, cot, scale, lb, order, with_final)) / (2 * h)


@pytest.mark.parametrize("with_final", [True, False])
@pytest.mark.parametrize("order", ["decay_first", "literal"])
def test_directional_derivatives_match_finite_differences(order, with_final):
    x, cot = case(1)
    scale, lb = 0.6, -2.5
    gr = grads(x, cot, scale, lb, order, with_final)
    r = np.random.default_rng(5)
    for name in NAMES:
        direction = r.normal(size=np.shape(x[name]))
        fd = directional(x, cot, name, direction, scale, lb, order, with_final)
        an = float(np.sum(gr[GRAD[name]] * direction))
        assert an == pytest.approx(fd, rel=1e-6, abs=1e-8), (name, an, fd)


def test_every_coordinate_on_a_tiny_case():
    """Coordinate by coordinate (a full gradient check) on B = 1, T = 4, H = 1, dk = 3,
    dv = 2, strong decay (lower_bound -5)."""
    x, cot = case(2, B=1, T=4, H=1, dk=3, dv=2)
    gr = grads(x, cot, 1.0, -5.0, "decay_first")
    for name in NAMES:
        flat = np.zeros(np.size(x[name]))
        for i in range(flat.size):
            e = np.zeros_like(flat)
            e[i] = 1.0
            flat[i] = directional(x, cot, name, e.reshape(np.shape(x[name])), 1.0, -5.0,
                                  "decay_first", True)
        np.testing.assert_allclose(np.ravel(gr[GRAD[name]]), flat, rtol=1e-6, atol=1e-8,
                                   err_msg=name)


def test_zero_cotangent_gives_zero_gradients():
    x, cot = case(3)
    cot = {n: np.zeros_like(c) for n, c in cot.items()}
    gr = grads(x, cot, 0.5, -1.0, "decay_first")
    for n, val in gr.items():
        assert np.all(val == 0.0), n


def test_value_gradient_closed_form_single_token():
    """One token from a zero state: out = beta (k^ . q^) v, so d out / d v = beta (k^ . q^)
    on the diagonal: dv = beta (k^ . q^) d_out."""
    r = np.random.default_rng(9)
    B, H, dk, dv = 2, 3, 4, 5
    q, k = r.normal(size=(B, 1, H, dk)), r.normal(size=(B, 1, H, dk))
    v, g = r.normal(size=(B, 1, H, dv)), r.normal(size=(B, 1, H, dk))
    bl = r.normal(size=(B, 1, H))
    d_out = r.normal(size=(B, 1, H, dv))
    gr = kda_backward(q, k, v, g, bl, np.zeros(H), np.zeros((dk, H)), d_out, None, 1.0, -1.0)
    qn = q / np.sqrt((q ** 2).sum(-1, keepdims=True) + 1e-6)
    kn = k / np.sqrt((k ** 2).sum(-1, keepdims=True) + 1e-6)
    beta = 1 / (1 + np.exp(-bl))
    np.testing.assert_allclose(gr["dv"], beta[..., None] * (qn * kn).sum(-1, keepdims=True) * d_out,
                               rtol=1e-12, atol=1e-12)
