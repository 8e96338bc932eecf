"""Pins of the oracle's ``kda_attention`` (the ejkernel kernel_delta_attention call:
per-head log-decay, beta as given, optional L2 norm) against facts fixed by the page and
by hand arithmetic, not by re-running the oracle's own formula."""
import numpy as np
import pytest

from oracle import kda_attention, kda_forward


def _rng(seed):
    return np.random.default_rng(1000 + seed)


def test_scalar_recurrence_by_hand_decay_first_and_literal():
    """dk = dv = 1, no normalisation, scale 1: S0 = 2, k = 1, v = 3, beta = 0.5,
    e^decay = 0.5, q = 1.
    decay first: S' = 1, u = 0.5 (3 - 1) = 1, S1 = 1 + 1 = 2, o = 2.
    literal:     u = 0.5 (3 - 2) = 0.5, S1 = 0.5 * 2 + 0.5 = 1.5, o = 1.5."""
    one = np.ones((1, 1, 1, 1))
    args = dict(query=one, key=one, value=3 * one, beta=0.5 * np.ones((1, 1, 1)),
                decay=np.log(0.5) * np.ones((1, 1, 1)), initial_state=2 * np.ones((1, 1, 1, 1)),
                softmax_scale=1.0, use_qk_l2norm=False)
    o, S = kda_attention(**args)
    assert o.item() == pytest.approx(2.0) and S.item() == pytest.approx(2.0)
    o, S = kda_attention(**args, order="literal")
    assert o.item() == pytest.approx(1.5) and S.item() == pytest.approx(1.5)


def test_scalar_two_tokens_by_hand():
    """dk = dv = 1, no decay, beta = 1, k = 1: each token overwrites the memory with v_t,
    so o_t = v_t * q_t * scale (scale 2 here)."""
    q = np.array([1.0, -3.0]).reshape(1, 2, 1, 1)
    v = np.array([5.0, 7.0]).reshape(1, 2, 1, 1)
    o, S = kda_attention(q, np.ones((1, 2, 1, 1)), v, np.ones((1, 2, 1)), None,
                         7.0 * np.ones((1, 1, 1, 1)), 2.0, use_qk_l2norm=False)
    np.testing.assert_allclose(o.ravel(), [10.0, -42.0])
    assert S.item() == pytest.approx(7.0)


@pytest.mark.parametrize("norm", [True, False])
def test_one_token_closed_form(norm):
    """From a zero memory one token gives o = beta (k^ . q^) v (q^ carrying the scale)."""
    r = _rng(1)
    B, H, dk, dv = 2, 3, 8, 5
    q, k = r.normal(size=(B, 1, H, dk)), r.normal(size=(B, 1, H, dk))
    v, beta = r.normal(size=(B, 1, H, dv)), r.uniform(size=(B, 1, H))
    o, S = kda_attention(q, k, v, beta, r.normal(size=(B, 1, H)) * 0.1, None, 0.7, norm)
    if norm:
        qn = q / np.sqrt((q ** 2).sum(-1, keepdims=True) + 1e-6)
        kn = k / np.sqrt((k ** 2).sum(-1, keepdims=True) + 1e-6)
    else:
        qn, kn = q, k
    expect = beta[..., None] * (kn * 0.7 * qn).sum(-1, keepdims=True) * v
    np.testing.assert_allclose(o, expect, rtol=1e-12, atol=1e-12)
    # the memory is the rank-1 write beta k^ v^T
    np.testing.assert_allclose(S, beta[:, 0, :, None, None] * kn[:, 0, :, :, None] * v[:, 0, :, None, :],
                               rtol=1e-12, atol=1e-12)


def test_pure_decay_closed_form():
    """beta = 0: the memory only decays, S_T = exp(sum of decays) S0 per head, and every
    output reads the decayed initial memory."""
    r = _rng(2)
    B, T, H, dk, dv = 2, 6, 2, 4, 3
    S0 = r.normal(size=(B, H, dk, dv))
    d = -r.uniform(0, 0.5, size=(B, T, H))
    q = r.normal(size=(B, T, H, dk))
    o, S = kda_attention(q, r.normal(size=(B, T, H, dk)), r.normal(size=(B, T, H, dv)),
                         np.zeros((B, T, H)), d, S0, 1.0, use_qk_l2norm=False)
    cum = np.cumsum(d, axis=1)  # [B, T, H]
    np.testing.assert_allclose(S, np.exp(cum[:, -1])[..., None, None] * S0, rtol=1e-12)
    expect = np.exp(cum)[..., None] * np.einsum("bhij,bthi->bthj", S0, q)
    np.testing.assert_allclose(o, expect, rtol=1e-12, atol=1e-12)


def test_orthonormal_keys_exact_retrieval():
    """No decay, beta = 1, orthonormal keys, zero start: writing v_i under key e_i and
    reading with q = e_j (scale 1) returns v_j once it has been written."""
    dk, dv, T = 4, 3, 4
    keys = np.eye(dk)[None, :, None, :]             # [1, T, 1, dk]
    v = _rng(3).normal(size=(1, T, 1, dv))
    q = keys.copy()
    o, S = kda_attention(q, keys, v, np.ones((1, T, 1)), None, None, 1.0, use_qk_l2norm=True)
    np.testing.assert_allclose(o[0, :, 0], v[0, :, 0] / (1 + 1e-6), rtol=1e-9)
    np.testing.assert_allclose(S[0, 0], v[0, :, 0] / np.sqrt(1 + 1e-6), rtol=1e-9)  # row i = k^_i v_i


def test_norm_off_equals_norm_on_for_unit_inputs():
    r = _rng(4)
    q = r.normal(size=(1, 5, 2, 8))
    k = r.normal(size=(1, 5, 2, 8))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    args = (q, k, r.normal(size=(1, 5, 2, 3)), r.uniform(size=(1, 5, 2)), -r.uniform(size=(1, 5, 2)))
    o1, S1 = kda_attention(*args, use_qk_l2norm=True)
    o2, S2 = kda_attention(*args, use_qk_l2norm=False)
    np.testing.assert_allclose(o1, o2, rtol=1e-5)
    np.testing.assert_allclose(S1, S2, rtol=1e-5)


def test_default_scale_and_agreement_with_the_gated_form():
    """softmax_scale None is dk^-0.5; and a per-head decay d equals the kda_tkg gate form
    with raw gates chosen so that lower_bound * sigmoid(exp(a_log) (g + dt_bias)) = d on
    every channel, beta logits = logit(beta)."""
    r = _rng(5)
    B, T, H, dk, dv = 1, 7, 2, 16, 4
    q, k = r.normal(size=(B, T, H, dk)), r.normal(size=(B, T, H, dk))
    v = r.normal(size=(B, T, H, dv))
    beta = r.uniform(0.05, 0.95, size=(B, T, H))
    d = -r.uniform(0.01, 2.0, size=(B, T, H))
    lb, a_log = -3.0, np.array([0.2, -0.4])
    dt_bias = r.normal(size=(dk, H)) * 0.1
    p = d / lb                                          # sigmoid(z) = d / lb
    z = np.log(p / (1 - p))
    g = z[..., None] / np.exp(a_log)[None, None, :, None] - dt_bias.T[None, None]
    o1, S1 = kda_attention(q, k, v, beta, d, None, None)
    o2, S2 = kda_forward(q, k, v, g, np.log(beta / (1 - beta)), a_log, dt_bias, dk ** -0.5, lb)
    np.testing.assert_allclose(o1, o2, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(S1, S2, rtol=1e-9, atol=1e-12)
