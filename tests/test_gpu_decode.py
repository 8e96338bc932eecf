"""Parity of kda_decode_step (the fused single-token decode kernel) with the fp64 oracle,
through the C ABI, in the kda_tkg layouts.  fp32 path: max |gpu - oracle| <= 1e-4."""
import math

import numpy as np
import pytest
import torch

from gated_delta_rule_55_gb300 import kda_decode_step, synth
from gpu_helpers import F32_ATOL, ensure_built, max_abs, oracle_pool, to_dev
from oracle import kda_decode_step as oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _run(tok, a_log, dt_bias, S, scale, lb):
    B, H, dv = tok["v"].shape
    dk = tok["q"].shape[1]
    out = torch.full((B, H, dv), float("nan"), device="cuda")
    Sd = to_dev(S) if isinstance(S, np.ndarray) else S
    kda_decode_step(to_dev(tok["q"]), to_dev(tok["k"]), to_dev(tok["v"]), to_dev(tok["g"]),
                    to_dev(tok["beta_logits"]), to_dev(a_log), to_dev(dt_bias), scale, lb, out,
                    Sd, B, H, dk, dv)
    torch.cuda.synchronize()
    return out.cpu().numpy(), Sd


@pytest.mark.parametrize("dk,dv", [(128, 128), (128, 64), (64, 128), (32, 32), (64, 32)])
@pytest.mark.parametrize("lb", [-5.0, -0.3, 0.0])
def test_decode_small_shapes(dk, dv, lb):
    B, H = 3, 5
    tok = synth.decode_token_inputs(B, H, dk, dv, seed=100 + dk + dv)
    a_log, dt_bias = synth.gate_params(H, dk, 101)
    S = synth.decode_state(B, H, dk, dv, 102, std=0.5)
    scale = dk ** -0.5
    out, Sd = _run(tok, a_log, dt_bias, S, scale, lb)
    o_ref, S_ref = oracle_decode(**tok, a_log=a_log, dt_bias=dt_bias, scale=scale,
                                 lower_bound=lb, S=S)
    assert max_abs(out, o_ref) <= F32_ATOL
    assert max_abs(Sd.cpu().numpy(), S_ref) <= F32_ATOL


def test_decode_extreme_gates_and_betas():
    """Saturated sigmoids (logits +-30) for both the gate and beta."""
    B, H, dk, dv = 2, 3, 128, 128
    tok = synth.decode_token_inputs(B, H, dk, dv, seed=7)
    tok["g"] = np.sign(tok["g"]) * 30.0
    tok["beta_logits"] = np.sign(tok["beta_logits"]) * 30.0
    a_log, dt_bias = synth.gate_params(H, dk, 8)
    S = synth.decode_state(B, H, dk, dv, 9, std=1.0)
    out, Sd = _run(tok, a_log, dt_bias, S, 0.1, -5.0)
    o_ref, S_ref = oracle_decode(**tok, a_log=a_log, dt_bias=dt_bias, scale=0.1,
                                 lower_bound=-5.0, S=S)
    assert max_abs(out, o_ref) <= F32_ATOL
    assert max_abs(Sd.cpu().numpy(), S_ref) <= F32_ATOL


def test_decode_workload_B64_full_compare():
    """The B=64, H=32, dk=dv=128 decode workload, every output and state entry."""
    w = synth.DECODE_B64
    d = synth.workload_inputs(w)
    tok = {n: d[n] for n in ("q", "k", "v", "g", "beta_logits")}
    out, Sd = _run(tok, d["a_log"], d["dt_bias"], d["S"], w.q_scale, w.lower_bound)
    o_ref, S_ref = oracle_decode(**tok, a_log=d["a_log"], dt_bias=d["dt_bias"],
                                 scale=w.q_scale, lower_bound=w.lower_bound, S=d["S"])
    assert max_abs(out, o_ref) <= F32_ATOL
    assert max_abs(Sd.cpu().numpy(), S_ref) <= F32_ATOL


def test_decode_workload_B512_32_chained_steps_full():
    """B=512, H=32, 128x128 state (1.07 GB) advanced by 32 consecutive calls with the state
    passed through in place: every output of every step and every final-state entry of all
    16,384 (b, h) pairs against 32 chained oracle steps (run over head ranges in a pool of
    host processes)."""
    from oracle import pool
    w = synth.DECODE_B512
    B, H, dk, dv = w.B, w.H, w.dk, w.dv
    a_log, dt_bias = synth.gate_params(H, dk, w.seed)
    S0 = synth.decode_state(B, H, dk, dv, w.seed, w.state_std)
    toks = [synth.decode_token_inputs(B, H, dk, dv, w.seed, step) for step in range(w.steps)]
    oracle_pool()  # start the workers before the device work
    Sd = to_dev(S0)
    outs = []
    for tok in toks:
        out, Sd = _run(tok, a_log, dt_bias, Sd, w.q_scale, w.lower_bound)
        outs.append(out)
    S_gpu = Sd.cpu().numpy()
    del Sd
    o_ref, S_ref = pool.decode_chain(oracle_pool(), toks, a_log, dt_bias, w.q_scale,
                                     w.lower_bound, S0)
    worst_o = max(max_abs(o, r) for o, r in zip(outs, o_ref))
    assert worst_o <= F32_ATOL, worst_o
    assert max_abs(S_gpu, S_ref) <= F32_ATOL


def test_decode_batch_zero_is_a_no_op():
    tok = synth.decode_token_inputs(1, 2, 32, 32, seed=1)
    a_log, dt_bias = synth.gate_params(2, 32, 1)
    out = torch.zeros(1, 2, 32, device="cuda")
    S = torch.zeros(1, 2, 32, 32, device="cuda")
    kda_decode_step(to_dev(tok["q"]), to_dev(tok["k"]), to_dev(tok["v"]), to_dev(tok["g"]),
                    to_dev(tok["beta_logits"]), to_dev(a_log), to_dev(dt_bias), 0.2, -1.0,
                    out, S, 0, 2, 32, 32)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0 and math.isfinite(out.sum().item())
