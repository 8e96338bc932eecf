"""The oracle's process pool (oracle/pool.py) returns what the oracle returns when called
directly: it only cuts the problem into independent (sequence, head) groups."""
import numpy as np
import pytest

from gated_delta_rule_55_gb300 import synth
from oracle import kda_decode_step, kda_forward, kda_forward_varlen, pool


@pytest.fixture(scope="module")
def ex():
    with pool.Pool(workers=3) as e:
        yield e


def test_forward_groups_equal_one_call(ex):
    d = synth.chunk_inputs(2, 23, 5, 16, 8, seed=3, state_std=0.1)
    args = (d["q"], d["k"], d["v"], d["g"], d["beta_logits"], d["a_log"], d["dt_bias"], 0.3,
            -2.0, d["initial_state"])
    o1, s1 = kda_forward(*args)
    o2, s2 = pool.forward(ex, *args, workers=3)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(s2, s1, rtol=0, atol=1e-12)


def test_forward_varlen_groups_equal_one_call(ex):
    d = synth.varlen_inputs([7, 0, 30, 1], 3, 16, 16, seed=4, state_std=0.1)
    args = (d["q"], d["k"], d["v"], d["g"], d["beta_logits"], d["a_log"], d["dt_bias"],
            d["cu_seqlens"], 0.25, -1.0, d["initial_state"])
    o1, s1 = kda_forward_varlen(*args)
    o2, s2 = pool.forward_varlen(ex, *args, workers=3)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(s2, s1, rtol=0, atol=1e-12)


def test_decode_chain_equals_consecutive_steps(ex):
    B, H, dk, dv = 3, 4, 16, 8
    a_log, dt_bias = synth.gate_params(H, dk, 5)
    S = synth.decode_state(B, H, dk, dv, 5)
    toks = [synth.decode_token_inputs(B, H, dk, dv, 5, step) for step in range(4)]
    outs, S_ref = [], S
    for t in toks:
        o, S_ref = kda_decode_step(**t, a_log=a_log, dt_bias=dt_bias, scale=0.25,
                                   lower_bound=-3.0, S=S_ref)
        outs.append(o)
    o2, s2 = pool.decode_chain(ex, toks, a_log, dt_bias, 0.25, -3.0, S, workers=3)
    np.testing.assert_allclose(o2, np.stack(outs), rtol=0, atol=1e-12)
    np.testing.assert_allclose(s2, S_ref, rtol=0, atol=1e-12)


def test_recurrent_groups_equal_one_call(ex):
    from oracle import recurrent_attention
    r = np.random.default_rng(9)
    B, T, Hq, Hkv, D = 2, 13, 6, 3, 8
    q = r.normal(size=(B, T, Hq, D))
    k = r.normal(size=(B, T, Hkv, D))
    v = r.normal(size=(B, T, Hkv, D))
    gk = -r.uniform(0, 0.5, size=(B, T, Hq, D))
    gam = -r.uniform(0, 0.2, size=(B, Hq))
    s0 = r.normal(size=(B, Hq, D, D))
    o1, s1 = recurrent_attention(q, k, v, None, gam, gk, None, 0.4, s0)
    o2, s2 = pool.recurrent(ex, q, k, v, None, gam, gk, None, 0.4, s0, workers=3)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(s2, s1, rtol=0, atol=1e-12)
