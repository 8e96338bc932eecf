"""Pins for the fp64 oracle: facts the pages and the mathematics fix, none of them a
retyping of the oracle's own formulas.

Every pin is chosen so that a plausible slip in the oracle (a dropped decay, a wrong
sign in the delta term, the output read before the update, a transposed memory, a
missing normalisation or sigmoid, a shifted cumulative gate, the wrong decay/delta
order) fails at least one of them.  Page references: ``kernel_delta_attention`` =
ejkernel module page (its "core recurrence" and parameter list); ``kda_tkg`` = NKI "KDA
TKG Kernel API Reference" parameter list.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import (activate_gate, kda_decode_step, kda_forward, kda_forward_varlen,
                    l2_normalize, sigmoid)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
INF = np.inf


def _logit(p):
    return math.log(p / (1.0 - p))


def _gate_inputs_for(p, a_log, dt_bias):
    """Raw g such that the activated gate's sigmoid equals ``p`` exactly:
    g = -dt_bias + logit(p) / exp(a_log).  ``p`` is ``[..., H, dk]``."""
    p = np.asarray(p, dtype=np.float64)
    lg = np.log(p / (1.0 - p))
    return -np.asarray(dt_bias).T + lg / np.exp(np.asarray(a_log))[:, None]


# --------------------------------------------------------------------------- prologue

def test_sigmoid_special_values():
    assert sigmoid(0.0) == 0.5
    assert abs(sigmoid(math.log(3.0)) - 0.75) < 1e-15
    assert sigmoid(-INF) == 0.0 and sigmoid(INF) == 1.0
    x = np.linspace(-30, 30, 61)
    np.testing.assert_allclose(sigmoid(-x), 1.0 - sigmoid(x), atol=1e-15)


def test_gate_midpoint_and_three_quarters():
    """kda_tkg: gamma = lower_bound * sigmoid(exp(a_log) * (g + dt_bias)).
    g = -dt_bias puts the sigmoid at 1/2 whatever a_log is; a_log = log(log 3) with
    g + dt_bias = 1 puts it at 3/4 (a missing exp on a_log would give ~0.52)."""
    rng = np.random.default_rng(0)
    H, dk = 3, 5
    a_log = rng.uniform(-1, 1, H)
    dt_bias = rng.normal(0, 0.1, (dk, H))
    for lb in (-5.0, -1.3, 0.0):
        gam = activate_gate(-dt_bias.T[None], a_log, dt_bias, lb)
        np.testing.assert_allclose(gam, lb / 2, atol=1e-15)
        a2 = np.full(H, math.log(math.log(3.0)))
        gam = activate_gate((1.0 - dt_bias.T)[None], a2, dt_bias, lb)
        np.testing.assert_allclose(gam, 0.75 * lb, atol=1e-14)


def test_gate_limits_and_range():
    """lower_bound in [-5, 0] (kda_tkg): gamma in [lower_bound, 0], so exp(gamma) in (0, 1]."""
    H, dk = 2, 4
    a_log = np.zeros(H)
    dt_bias = np.zeros((dk, H))
    big = np.full((1, H, dk), 1e4)
    np.testing.assert_allclose(activate_gate(big, a_log, dt_bias, -5.0), -5.0)
    np.testing.assert_allclose(activate_gate(-big, a_log, dt_bias, -5.0), 0.0, atol=1e-300)
    rng = np.random.default_rng(1)
    g = rng.normal(0, 3, (64, H, dk))
    gam = activate_gate(g, rng.uniform(-1, 1, H), rng.normal(0, .1, (dk, H)), -5.0)
    assert np.all(gam <= 0) and np.all(gam >= -5.0)


def test_l2_normalize_unit_norm_and_direction():
    rng = np.random.default_rng(2)
    x = rng.normal(size=(7, 16)) * 1e3
    y = l2_normalize(x)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), 1.0, atol=1e-12)
    np.testing.assert_allclose(y * np.linalg.norm(x, axis=-1, keepdims=True), x, rtol=1e-12)


# ------------------------------------------------------------------- the recurrence

def _zero_gate_params(H, dk):
    return np.zeros(H), np.zeros((dk, H))


def test_one_token_closed_form():
    """From S0 = 0 a single token gives S1 = beta k^ v^T and o1 = beta (k^ . q^) v, with
    q^ carrying the scale (kda_tkg scale parameter).  dk != dv catches transposes."""
    rng = np.random.default_rng(3)
    B, H, dk, dv = 2, 2, 3, 5
    q = rng.normal(size=(B, 1, H, dk)) * 50
    k = rng.normal(size=(B, 1, H, dk)) * 50
    v = rng.normal(size=(B, 1, H, dv))
    bl = np.full((B, 1, H), math.log(3.0))  # beta = 3/4
    a_log, dt_bias = _zero_gate_params(H, dk)
    g = rng.normal(size=(B, 1, H, dk))
    scale = 0.37
    out, S = kda_forward(q, k, v, g, bl, a_log, dt_bias, scale, -4.0)
    kh = k[:, 0] / np.linalg.norm(k[:, 0], axis=-1, keepdims=True)
    qh = scale * q[:, 0] / np.linalg.norm(q[:, 0], axis=-1, keepdims=True)
    S1 = 0.75 * kh[..., :, None] * v[:, 0][..., None, :]
    np.testing.assert_allclose(S, S1, atol=1e-9)
    o1 = 0.75 * np.sum(kh * qh, -1)[..., None] * v[:, 0]
    np.testing.assert_allclose(out[:, 0], o1, atol=1e-9)


def test_pure_decay_when_beta_is_zero():
    """beta = 0 (logit -inf): each token only multiplies row i of S by exp(gamma_i), so
    S_t = diag(exp(lower_bound * sum_{s<=t} p_s)) S0 with gate sigmoids p chosen exactly."""
    rng = np.random.default_rng(4)
    B, T, H, dk, dv = 1, 6, 2, 4, 3
    lb = -2.0
    a_log = rng.uniform(-1, 1, H)
    dt_bias = rng.normal(0, 0.1, (dk, H))
    p = rng.uniform(0.05, 0.95, (B, T, H, dk))
    g = _gate_inputs_for(p, a_log, dt_bias)
    S0 = rng.normal(size=(B, H, dk, dv))
    q = rng.normal(size=(B, T, H, dk))
    out, S = kda_forward(q, rng.normal(size=(B, T, H, dk)), rng.normal(size=(B, T, H, dv)),
                         g, np.full((B, T, H), -INF), a_log, dt_bias, 1.0, lb, S0)
    G = lb * np.cumsum(p, axis=1)  # [B, T, H, dk]
    for t in range(T):
        St = np.exp(G[:, t])[..., :, None] * S0
        qh = q[:, t] / np.sqrt(np.sum(q[:, t] ** 2, -1, keepdims=True) + 1e-6)
        np.testing.assert_allclose(out[:, t], np.einsum("bhij,bhi->bhj", St, qh), atol=1e-12)
    np.testing.assert_allclose(S, np.exp(G[:, -1])[..., :, None] * S0, atol=1e-12)


def test_orthonormal_keys_are_retrieved_exactly():
    """No decay (lower_bound = 0), beta = 1: writing (k_i, v_i) for orthonormal keys and
    then reading with q = k_i (beta = 0 on the reading tokens, scale 1) returns v_i."""
    rng = np.random.default_rng(5)
    H, dk, dv, n = 1, 8, 5, 6
    Qm, _ = np.linalg.qr(rng.normal(size=(dk, dk)))
    keys = Qm[:, :n].T * 1e4  # large norms make the 1e-6 epsilon invisible
    vals = rng.normal(size=(n, dv))
    T = 2 * n
    k = np.concatenate([keys, keys])[None, :, None, :]
    v = np.concatenate([vals, np.zeros_like(vals)])[None, :, None, :]
    q = k.copy()
    bl = np.concatenate([np.full(n, INF), np.full(n, -INF)])[None, :, None]
    a_log, dt_bias = _zero_gate_params(H, dk)
    g = rng.normal(size=(1, T, H, dk))
    out, S = kda_forward(q, k, v, g, bl, a_log, dt_bias, 1.0, 0.0)
    np.testing.assert_allclose(out[0, n:, 0], vals, atol=1e-12)
    kh = keys / np.linalg.norm(keys, axis=1, keepdims=True)
    np.testing.assert_allclose(S[0, 0], kh.T @ vals, atol=1e-12)


def test_delta_rule_overwrites_instead_of_adding():
    """beta = 1: writing (k, v1) then (k, v2) leaves S^T k^ = v2 (an additive memory would
    give v1 + v2).  beta = 1/2 (logit 0) twice with the same pair gives (3/4) v."""
    rng = np.random.default_rng(6)
    H, dk, dv = 1, 4, 3
    kk = rng.normal(size=dk) * 1e4
    v1, v2 = rng.normal(size=dv), rng.normal(size=dv)
    k = np.stack([kk, kk])[None, :, None]
    a_log, dt_bias = _zero_gate_params(H, dk)
    g = np.zeros((1, 2, H, dk))
    kh = kk / np.linalg.norm(kk)
    _, S = kda_forward(k, k, np.stack([v1, v2])[None, :, None], g,
                       np.full((1, 2, H), INF), a_log, dt_bias, 1.0, 0.0)
    np.testing.assert_allclose(S[0, 0].T @ kh, v2, atol=1e-12)
    _, S = kda_forward(k, k, np.stack([v1, v1])[None, :, None], g,
                       np.zeros((1, 2, H)), a_log, dt_bias, 1.0, 0.0)
    np.testing.assert_allclose(S[0, 0].T @ kh, 0.75 * v1, atol=1e-12)


@pytest.mark.parametrize("order", ["decay_first", "literal"])
def test_decay_and_delta_order(order):
    """S0 = k^ v0^T, a uniform gate gamma = lower_bound / 2, beta = 1 and key k:
    decay first gives S1 = k^ v^T (the write sees the decayed memory); the literal
    reading gives S1 = e^gamma k^ v0^T + k^ (v - v0)^T."""
    rng = np.random.default_rng(7)
    H, dk, dv = 1, 5, 4
    kk = rng.normal(size=dk) * 1e4
    kh = kk / np.linalg.norm(kk)
    v0, v = rng.normal(size=dv), rng.normal(size=dv)
    lb = -3.0
    a_log = np.array([0.3])
    dt_bias = rng.normal(0, .1, (dk, H))
    g = -dt_bias.T[None, None]  # sigmoid(0) = 1/2 -> gamma = lb / 2 in every channel
    S0 = (kh[:, None] * v0[None, :])[None, None]
    _, S = kda_forward(kk[None, None, None], kk[None, None, None], v[None, None, None], g,
                       np.full((1, 1, 1), INF), a_log, dt_bias, 1.0, lb, S0, order=order)
    c = math.exp(lb / 2)
    if order == "decay_first":
        want = kh[:, None] * v[None, :]
    else:
        want = c * kh[:, None] * v0[None, :] + kh[:, None] * (v - v0)[None, :]
    np.testing.assert_allclose(S[0, 0], want, atol=1e-12)


def test_orders_agree_without_gate():
    rng = np.random.default_rng(8)
    d = dict(q=rng.normal(size=(1, 9, 2, 4)), k=rng.normal(size=(1, 9, 2, 4)),
             v=rng.normal(size=(1, 9, 2, 3)), g=rng.normal(size=(1, 9, 2, 4)),
             beta_logits=rng.normal(size=(1, 9, 2)), a_log=rng.uniform(-1, 1, 2),
             dt_bias=rng.normal(0, .1, (4, 2)), initial_state=rng.normal(size=(1, 2, 4, 3)))
    a = kda_forward(**d, scale=0.5, lower_bound=0.0, order="decay_first")
    b = kda_forward(**d, scale=0.5, lower_bound=0.0, order="literal")
    np.testing.assert_allclose(a[0], b[0], atol=1e-13)
    np.testing.assert_allclose(a[1], b[1], atol=1e-13)


def test_scalar_memory_matches_geometric_series():
    """dk = dv = 1 with constant inputs: s_t = a s_{t-1} + b with
    a = e^gamma (1 - beta kappa), b = beta k^ v, kappa = k^2 / (k^2 + eps);
    so s_T = a^T s0 + b (1 - a^T) / (1 - a) and o_t = s_t q^."""
    T, eps = 25, 1e-6
    kv, qv, vv, s0, lb, scale = -0.8, 1.7, 2.3, 0.4, -1.0, 0.9
    p, beta = 0.3, 0.6
    a_log = np.array([0.2])
    dt_bias = np.array([[0.05]])
    g = _gate_inputs_for(np.full((1, T, 1, 1), p), a_log, dt_bias)
    out, S = kda_forward(np.full((1, T, 1, 1), qv), np.full((1, T, 1, 1), kv),
                         np.full((1, T, 1, 1), vv), g, np.full((1, T, 1), _logit(beta)),
                         a_log, dt_bias, scale, lb, np.full((1, 1, 1, 1), s0))
    kh = kv / math.sqrt(kv * kv + eps)
    qh = scale * qv / math.sqrt(qv * qv + eps)
    a = math.exp(lb * p) * (1 - beta * kh * kh)
    b = beta * kh * vv
    for t in range(1, T + 1):
        st = a ** t * s0 + b * (1 - a ** t) / (1 - a)
        assert abs(out[0, t - 1, 0, 0] - st * qh) < 1e-12
    assert abs(S[0, 0, 0, 0] - (a ** T * s0 + b * (1 - a ** T) / (1 - a))) < 1e-12


# -------------------------------------------------------------- structural invariants

def _random_problem(rng, B=2, T=23, H=3, dk=6, dv=5, lb=-5.0, init=True):
    return dict(q=rng.normal(size=(B, T, H, dk)), k=rng.normal(size=(B, T, H, dk)),
                v=rng.normal(size=(B, T, H, dv)), g=rng.normal(size=(B, T, H, dk)),
                beta_logits=rng.normal(size=(B, T, H)), a_log=rng.uniform(-1, 1, H),
                dt_bias=rng.normal(0, 0.1, (dk, H)), lower_bound=lb,
                initial_state=rng.normal(0, 0.5, (B, H, dk, dv)) if init else None)


def test_split_sequence_equals_one_pass():
    """State passthrough (kernel_delta_attention: initial_state / return_state)."""
    rng = np.random.default_rng(9)
    d = _random_problem(rng, T=37, lb=-0.7)
    out, S = kda_forward(**d, scale=0.3)
    d1 = {n: (x[:, :20] if n in "q k v g beta_logits".split() else x) for n, x in d.items()}
    d2 = {n: (x[:, 20:] if n in "q k v g beta_logits".split() else x) for n, x in d.items()}
    o1, s1 = kda_forward(**d1, scale=0.3)
    d2["initial_state"] = s1
    o2, s2 = kda_forward(**d2, scale=0.3)
    np.testing.assert_allclose(np.concatenate([o1, o2], 1), out, atol=1e-12)
    np.testing.assert_allclose(s2, S, atol=1e-12)


def test_decode_step_equals_last_scan_step():
    """kda_tkg advances the recurrence by one token in its own layouts (q/k/g
    [B, dk, H], v [B, H, dv], beta [B, 1, H]); it must equal the scan's last token."""
    rng = np.random.default_rng(10)
    d = _random_problem(rng, B=3, T=5, H=2, dk=6, dv=4)
    out, S = kda_forward(**d, scale=0.25)
    dp = {n: (x[:, :4] if n in "q k v g beta_logits".split() else x) for n, x in d.items()}
    _, S4 = kda_forward(**dp, scale=0.25)
    t = 4
    o, Sn = kda_decode_step(np.swapaxes(d["q"][:, t], 1, 2), np.swapaxes(d["k"][:, t], 1, 2),
                            d["v"][:, t], np.swapaxes(d["g"][:, t], 1, 2),
                            d["beta_logits"][:, t][:, None, :], d["a_log"][None, :],
                            d["dt_bias"], 0.25, d["lower_bound"], S4)
    np.testing.assert_allclose(o, out[:, t], atol=1e-12)
    np.testing.assert_allclose(Sn, S, atol=1e-12)


def test_memory_never_grows_without_writes():
    """kda_tkg lower_bound: exp(gamma) in (0, 1], so with beta = 0 no entry of S grows."""
    rng = np.random.default_rng(11)
    d = _random_problem(rng, T=1, lb=-5.0)
    S = d["initial_state"]
    for _ in range(10):
        d["initial_state"] = S
        d["g"] = rng.normal(size=d["g"].shape) * 3
        d["beta_logits"] = np.full(d["beta_logits"].shape, -INF)
        _, Sn = kda_forward(**d, scale=1.0)
        assert np.all(np.abs(Sn) <= np.abs(S) + 1e-15)
        S = Sn


def test_spectral_norm_bound():
    """(I - beta k^ k^T) D has operator norm <= 1 for beta in [0, 1] and D <= I, hence
    ||S_t||_2 <= ||S_{t-1}||_2 + beta_t ||v_t||_2 at every token."""
    rng = np.random.default_rng(12)
    d = _random_problem(rng, B=1, T=1, H=1, dk=7, dv=4)
    S = d["initial_state"]
    for _ in range(30):
        d.update(initial_state=S, q=rng.normal(size=d["q"].shape),
                 k=rng.normal(size=d["k"].shape), v=rng.normal(size=d["v"].shape) * 3,
                 g=rng.normal(size=d["g"].shape), beta_logits=rng.normal(size=(1, 1, 1)) * 3)
        _, Sn = kda_forward(**d, scale=1.0)
        beta = 1 / (1 + math.exp(-d["beta_logits"][0, 0, 0]))
        assert (np.linalg.norm(Sn[0, 0], 2)
                <= np.linalg.norm(S[0, 0], 2) + beta * np.linalg.norm(d["v"]) + 1e-12)
        S = Sn


def test_normalisation_and_linearity_invariances():
    """q and k are L2-normalised (kernel_delta_attention use_qk_l2norm; kda_tkg q/k raw):
    positive rescaling of q or k changes nothing; the map (v, S0) -> (out, S) is linear;
    out is linear in scale."""
    rng = np.random.default_rng(13)
    d = _random_problem(rng, lb=-1.0)
    d["q"] *= 1e3
    d["k"] *= 1e3
    out, S = kda_forward(**d, scale=0.4)
    c = rng.uniform(0.5, 4.0, size=d["q"].shape[:-1] + (1,))
    for name in ("q", "k"):
        dd = dict(d)
        dd[name] = d[name] * c
        o2, s2 = kda_forward(**dd, scale=0.4)
        np.testing.assert_allclose(o2, out, atol=1e-10)
        np.testing.assert_allclose(s2, S, atol=1e-10)
    dd = dict(d, v=d["v"] * 2.5, initial_state=d["initial_state"] * 2.5)
    o2, s2 = kda_forward(**dd, scale=0.4)
    np.testing.assert_allclose(o2, 2.5 * out, atol=1e-11)
    np.testing.assert_allclose(s2, 2.5 * S, atol=1e-11)
    o3, _ = kda_forward(**d, scale=0.8)
    np.testing.assert_allclose(o3, 2 * out, atol=1e-11)


def test_default_scale_is_inverse_sqrt_head_dim():
    rng = np.random.default_rng(14)
    d = _random_problem(rng, dk=16)
    a, _ = kda_forward(**d)
    b, _ = kda_forward(**d, scale=0.25)
    np.testing.assert_allclose(a, b, atol=1e-14)


def test_varlen_equals_separate_sequences_and_handles_empty_ones():
    """recurrent page cu_seqlens convention: each packed sequence runs from its own
    initial state; an empty sequence returns its initial state untouched."""
    rng = np.random.default_rng(15)
    H, dk, dv = 2, 4, 3
    lens = [5, 0, 11, 1]
    cu = np.concatenate([[0], np.cumsum(lens)])
    tot = cu[-1]
    d = dict(q=rng.normal(size=(tot, H, dk)), k=rng.normal(size=(tot, H, dk)),
             v=rng.normal(size=(tot, H, dv)), g=rng.normal(size=(tot, H, dk)),
             beta_logits=rng.normal(size=(tot, H)))
    a_log, dt_bias = rng.uniform(-1, 1, H), rng.normal(0, .1, (dk, H))
    S0 = rng.normal(size=(len(lens), H, dk, dv))
    out, fin = kda_forward_varlen(**d, a_log=a_log, dt_bias=dt_bias, cu_seqlens=cu,
                                  scale=0.5, lower_bound=-2.0, initial_state=S0)
    for n, L in enumerate(lens):
        a, b = cu[n], cu[n + 1]
        o, s = kda_forward(*(d[x][None, a:b] for x in "q k v g beta_logits".split()),
                           a_log, dt_bias, 0.5, -2.0, S0[n:n + 1])
        np.testing.assert_allclose(out[a:b], o[0], atol=1e-13)
        np.testing.assert_allclose(fin[n], s[0], atol=1e-13)
    np.testing.assert_array_equal(fin[1], S0[1])


# ------------------------------------------------------------------ the chunked form

@pytest.mark.parametrize("lb", [-5.0, -0.05])
@pytest.mark.parametrize("C", [1, 2, 16, 64, 100])
def test_chunked_form_equals_scan_fp64(C, lb):
    """The chunk algebra the kernels use (tests/chunk_form.py) is an exact
    re-association of the scan: fp64 agreement to ~1e-10 for every chunk size,
    a ragged last chunk (T = 100) and both a steep and a slow gate."""
    from chunk_form import chunk_core
    rng = np.random.default_rng(16)
    d = _random_problem(rng, B=1, T=100, H=1, dk=8, dv=6, lb=lb)
    out, S = kda_forward(**d, scale=0.3)
    gam = activate_gate(d["g"], d["a_log"], d["dt_bias"], lb)[0, :, 0]
    o, s = chunk_core(0.3 * l2_normalize(d["q"][0, :, 0]), l2_normalize(d["k"][0, :, 0]),
                      d["v"][0, :, 0], gam, sigmoid(d["beta_logits"][0, :, 0]),
                      d["initial_state"][0, 0], C)
    np.testing.assert_allclose(o, out[0, :, 0], atol=1e-10)
    np.testing.assert_allclose(s, S[0, 0], atol=1e-10)


def test_chunked_form_stays_finite_in_fp32_at_steepest_gate():
    """lower_bound = -5 with saturated gates is the worst case for the factorised
    exponentials: every factor must stay finite in fp32 and the result close to fp64."""
    from chunk_form import chunk_core
    rng = np.random.default_rng(17)
    T, dk, dv = 128, 32, 16
    d = _random_problem(rng, B=1, T=T, H=1, dk=dk, dv=dv, lb=-5.0)
    d["g"] = np.full_like(d["g"], 50.0)  # sigmoid -> 1: gamma = -5 everywhere
    out, S = kda_forward(**d, scale=dk ** -0.5)
    gam = activate_gate(d["g"], d["a_log"], d["dt_bias"], -5.0)[0, :, 0]
    o, s = chunk_core(dk ** -0.5 * l2_normalize(d["q"][0, :, 0]), l2_normalize(d["k"][0, :, 0]),
                      d["v"][0, :, 0], gam, sigmoid(d["beta_logits"][0, :, 0]),
                      d["initial_state"][0, 0], 64, dtype=np.float32)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(s))
    np.testing.assert_allclose(o, out[0, :, 0], atol=2e-5)
    np.testing.assert_allclose(s, S[0, 0], atol=2e-5)


# ------------------------------------------------------------------------ golden files

def test_page_one_example_shapes():
    """The kernel_delta_attention page's example: B=2, T=64, H=8, head_dim=32 gives an
    output of shape (2, 64, 8, 32), a state of (2, 8, 32, 32) and a next-token call
    on the returned state gives (2, 1, 8, 32)."""
    with open(os.path.join(GOLDEN, "p1_example_shapes.json")) as f:
        gold = json.load(f)
    B, T, H, D = (gold["inputs"][x] for x in ("batch", "seq_len", "num_heads", "head_dim"))
    rng = np.random.default_rng(18)
    d = _random_problem(rng, B=B, T=T, H=H, dk=D, dv=D, init=False)
    out, S = kda_forward(**d)
    assert list(out.shape) == gold["output_shape"]
    assert list(S.shape) == gold["state_shape"]
    d1 = _random_problem(rng, B=B, T=1, H=H, dk=D, dv=D, init=False)
    d1["initial_state"] = S
    o1, _ = kda_forward(**d1)
    assert list(o1.shape) == gold["next_token_output_shape"]


def test_regression_fixture():
    """Guards the oracle against silent change; the fixture is written by
    tests/golden/make_golden.py from the oracle itself."""
    from golden.make_golden import tiny_case
    with open(os.path.join(GOLDEN, "tiny_regression.json")) as f:
        gold = json.load(f)
    out, S = kda_forward(**tiny_case())
    np.testing.assert_allclose(out, np.array(gold["out"]), atol=1e-12)
    np.testing.assert_allclose(S, np.array(gold["final_state"]), atol=1e-12)
