"""Pins of the oracle's ``recurrent_attention`` (gated linear recurrence, the reading of the
ejkernel recurrent page) against closed forms computed without its loop: causal linear
attention as masked matrix products, and a brute-force double sum with the gate
exponentials taken directly over each token pair."""
import numpy as np
import pytest

from oracle import recurrent_attention


def rnd(seed, *shape):
    return np.random.default_rng(1200 + seed).normal(size=shape)


def brute(q, k, v, a, bgate, scale, h0):
    """o_t[j] = sum_{s<=t} sum_c q_t[c] k_s[c] v_s[j] exp(sum_{r=s+1..t} a_r[c] + bgate_r[j])
             + sum_c q_t[c] h0[c][j] exp(sum_{r<=t} a_r[c] + bgate_r[j])   (one head)."""
    T, D = q.shape
    out = np.zeros((T, D))
    for t in range(T):
        for s in range(t + 1):
            dec = np.exp(a[s + 1:t + 1].sum(0)[:, None] + bgate[s + 1:t + 1].sum(0)[None, :])
            out[t] += np.einsum("c,c,j,cj->j", scale * q[t], k[s], v[s], dec)
        dec0 = np.exp(a[:t + 1].sum(0)[:, None] + bgate[:t + 1].sum(0)[None, :])
        out[t] += np.einsum("c,cj->j", scale * q[t], h0 * dec0)
    return out


def test_ungated_is_causal_linear_attention():
    B, T, H, D = 2, 7, 3, 4
    q, k, v = rnd(1, B, T, H, D), rnd(2, B, T, H, D), rnd(3, B, T, H, D)
    o, S = recurrent_attention(q, k, v, softmax_scale=0.5)
    mask = np.tril(np.ones((T, T)))
    for b in range(B):
        for h in range(H):
            A = (q[b, :, h] @ k[b, :, h].T) * mask * 0.5
            np.testing.assert_allclose(o[b, :, h], A @ v[b, :, h], rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(S[b, h], k[b, :, h].T @ v[b, :, h], rtol=1e-12, atol=1e-12)


def test_all_gates_against_brute_force():
    B, T, Hq, D = 1, 6, 2, 3
    q, k, v = rnd(4, B, T, Hq, D), rnd(5, B, T, Hq, D), rnd(6, B, T, Hq, D)
    g, gk, gv = -np.abs(rnd(7, B, T, Hq, D)) * 0.3, -np.abs(rnd(8, B, T, Hq, D)) * 0.2, \
        -np.abs(rnd(9, B, T, Hq, D)) * 0.25
    gg = -np.abs(rnd(10, B, Hq)) * 0.1
    h0 = rnd(11, B, Hq, D, D)
    o, S = recurrent_attention(q, k, v, g, gg, gk, gv, 0.8, h0)
    for h in range(Hq):
        a = g[0, :, h] + gk[0, :, h] + gg[0, h]
        np.testing.assert_allclose(o[0, :, h], brute(q[0, :, h], k[0, :, h], v[0, :, h], a,
                                                     gv[0, :, h], 0.8, h0[0, h]),
                                   rtol=1e-11, atol=1e-12)


def test_default_scale_and_initial_state_decay():
    """One head, k = 0 (no writes), constant g_gamma: o_t = scale e^{gamma t} h0^T q_t with
    scale = D^-0.5."""
    B, T, H, D = 1, 5, 1, 4
    q = rnd(12, B, T, H, D)
    h0 = rnd(13, B, H, D, D)
    o, S = recurrent_attention(q, np.zeros((B, T, H, D)), rnd(14, B, T, H, D),
                               g_gamma=np.full((B, H), -0.3), initial_state=h0)
    for t in range(T):
        np.testing.assert_allclose(o[0, t, 0], D ** -0.5 * np.exp(-0.3 * (t + 1)) * h0[0, 0].T @ q[0, t, 0],
                                   rtol=1e-12)
    np.testing.assert_allclose(S[0, 0], np.exp(-0.3 * T) * h0[0, 0], rtol=1e-12)


def test_reverse_equals_time_flipped_forward():
    B, T, H, D = 2, 6, 2, 3
    args = [rnd(15 + i, B, T, H, D) for i in range(3)]
    gk = -np.abs(rnd(18, B, T, H, D)) * 0.2
    o_r, S_r = recurrent_attention(*args, gk=gk, reverse=True)
    flip = [x[:, ::-1] for x in args]
    o_f, S_f = recurrent_attention(*flip, gk=gk[:, ::-1])
    np.testing.assert_allclose(o_r, o_f[:, ::-1], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S_r, S_f, rtol=1e-12, atol=1e-12)


def test_grouped_kv_heads_equal_repeated_heads():
    B, T, Hq, Hkv, D = 1, 5, 4, 2, 3
    q, k, v = rnd(19, B, T, Hq, D), rnd(20, B, T, Hkv, D), rnd(21, B, T, Hkv, D)
    o1, S1 = recurrent_attention(q, k, v)
    o2, S2 = recurrent_attention(q, np.repeat(k, 2, axis=2), np.repeat(v, 2, axis=2))
    np.testing.assert_allclose(o1, o2, rtol=1e-12)
    np.testing.assert_allclose(S1, S2, rtol=1e-12)
    # head 1 of the queries reads kv head 0: it matches a single-head run against kv head 0
    o3, _ = recurrent_attention(q[:, :, 1:2], k[:, :, 0:1], v[:, :, 0:1])
    np.testing.assert_allclose(o1[:, :, 1:2], o3, rtol=1e-12)


def test_packed_sequences_equal_separate_calls():
    lens = [3, 0, 5]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, H, D = int(cu[-1]), 2, 3
    q, k, v = rnd(22, 1, T, H, D), rnd(23, 1, T, H, D), rnd(24, 1, T, H, D)
    gv = -np.abs(rnd(25, 1, T, H, D)) * 0.1
    h0 = rnd(26, 3, H, D, D)
    o, S = recurrent_attention(q, k, v, gv=gv, initial_state=h0, cu_seqlens=cu)
    for n in range(3):
        a, b = cu[n], cu[n + 1]
        on, Sn = recurrent_attention(q[:, a:b], k[:, a:b], v[:, a:b], gv=gv[:, a:b],
                                     initial_state=h0[n:n + 1])
        np.testing.assert_allclose(o[:, a:b], on, rtol=1e-12)
        np.testing.assert_allclose(S[n], Sn[0], rtol=1e-12)
