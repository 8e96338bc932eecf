"""Parity of kda_chunk_bwd (gradients of the chunked forward) with the oracle backward,
which is itself pinned to finite differences of the forward oracle.

fp32 q/k/v: max |gpu - oracle| <= 1e-4 * max(1, max |oracle|) per gradient tensor; bf16:
max |gpu - oracle| / max |oracle| <= 2e-2 per tensor, the oracle fed the same bf16-rounded
q, k, v and d_out."""
import numpy as np
import pytest
import torch

import gated_delta_rule_55_gb300 as kda
from gated_delta_rule_55_gb300 import synth
from gpu_helpers import (BF16_REL, bf16_round, bwd_err, ensure_built, max_abs, param_grad_scales,
                         rel_err, to_dev, workspace)
from oracle import kda_backward

pytestmark = pytest.mark.gpu

GRADS = ("dq", "dk", "dv", "dg", "dbeta_logits", "da_log", "ddt_bias", "dinitial_state")


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _run(d, cot, B, T, H, dk, dv, scale, lb, bf16, want_state=True):
    io = torch.bfloat16 if bf16 else torch.float32
    q, k, v = (to_dev(d[n], io) for n in ("q", "k", "v"))
    g, bl, al, db = (to_dev(d[n]) for n in ("g", "beta_logits", "a_log", "dt_bias"))
    dout = to_dev(cot["d_out"], io)
    dfin = to_dev(cot.get("d_final_state"))
    out = {"dq": torch.full((B, T, H, dk), float("nan"), device="cuda", dtype=io),
           "dk": torch.full((B, T, H, dk), float("nan"), device="cuda", dtype=io),
           "dv": torch.full((B, T, H, dv), float("nan"), device="cuda", dtype=io),
           "dg": torch.full((B, T, H, dk), float("nan"), device="cuda"),
           "dbeta_logits": torch.full((B, T, H), float("nan"), device="cuda"),
           "da_log": torch.full((H,), float("nan"), device="cuda"),
           "ddt_bias": torch.full((dk, H), float("nan"), device="cuda"),
           "dinitial_state": torch.full((B, H, dk, dv), float("nan"), device="cuda")}
    w = workspace(kda.kda_chunk_bwd_workspace_size(B, T, H, dk, dv,
                                                   kda.KDA_BF16 if bf16 else kda.KDA_F32))
    kda.kda_chunk_bwd(q, k, v, g, bl, al, db, scale, lb, to_dev(d.get("initial_state")), dout,
                      dfin, out["dq"], out["dk"], out["dv"], out["dg"], out["dbeta_logits"],
                      out["da_log"], out["ddt_bias"],
                      out["dinitial_state"] if want_state else None, B, T, H, dk, dv,
                      workspace=w)
    torch.cuda.synchronize()
    return {n: t.float().cpu().numpy() for n, t in out.items()}


def _oracle(d, cot, scale, lb, bf16):
    o = dict(d)
    c = dict(cot)
    if bf16:
        for n in ("q", "k", "v"):
            o[n] = bf16_round(d[n])
        c["d_out"] = bf16_round(cot["d_out"])
    return kda_backward(o["q"], o["k"], o["v"], o["g"], o["beta_logits"], o["a_log"],
                        o["dt_bias"], c["d_out"], c.get("d_final_state"), scale, lb,
                        o.get("initial_state"))


def _check(gpu, ref, bf16, names=GRADS, d=None):
    scales = param_grad_scales(ref["dg"], d["g"], d["dt_bias"]) if bf16 else {}
    for n in names:
        if bf16:
            e = bwd_err(n, gpu[n], ref[n], scales)
            assert e <= BF16_REL, (n, e)
        else:
            tol = 1e-4 * max(1.0, float(np.max(np.abs(ref[n]))))
            assert max_abs(gpu[n], ref[n]) <= tol, (n, max_abs(gpu[n], ref[n]), tol)


def _case(B, T, H, dk, dv, seed, state=True, final=True):
    d = synth.chunk_inputs(B, T, H, dk, dv, seed, 0.1 if state else None)
    r = np.random.default_rng(900 + seed)
    cot = {"d_out": r.normal(size=(B, T, H, dv))}
    if final:
        cot["d_final_state"] = r.normal(size=(B, H, dk, dv))
    return d, cot


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("T", [1, 64, 150])
def test_gradients_dk128(T, bf16):
    B, H, dk, dv = 2, 2, 128, 128
    d, cot = _case(B, T, H, dk, dv, T)
    gpu = _run(d, cot, B, T, H, dk, dv, 0.1, -2.0, bf16)
    _check(gpu, _oracle(d, cot, 0.1, -2.0, bf16), bf16, d=d)


@pytest.mark.parametrize("dk,dv", [(64, 32), (32, 64), (128, 32)])
def test_gradients_small_head_dims(dk, dv):
    B, T, H = 2, 90, 3
    d, cot = _case(B, T, H, dk, dv, dk + dv, state=False, final=False)
    gpu = _run(d, cot, B, T, H, dk, dv, 0.3, -0.5, False, want_state=True)
    _check(gpu, _oracle(d, cot, 0.3, -0.5, False), False)


def test_strong_decay_and_no_final_cotangent():
    B, T, H, dk, dv = 1, 130, 2, 128, 64
    d, cot = _case(B, T, H, dk, dv, 7, state=True, final=False)
    gpu = _run(d, cot, B, T, H, dk, dv, 0.09, -5.0, False)
    _check(gpu, _oracle(d, cot, 0.09, -5.0, False), False)


# ---- tensor-core chunk path (bf16, dk = dv = 128): chunk-boundary, decay and state cases


@pytest.mark.parametrize("B,T,H,lb,state,final", [
    (1, 64, 1, -2.0, True, True),     # one full chunk
    (2, 300, 2, -2.0, True, True),    # five chunks, ragged tail of 44 tokens
    (1, 200, 3, -5.0, False, False),  # strongest decay the ABI admits, no states
    (2, 129, 2, 0.0, True, True),     # no decay (lower_bound 0), one-token tail
    (1, 1, 2, -1.0, True, True),      # a single token
    (1, 1024, 1, -1.0, True, True),   # sixteen chunks: the state adjoint over many steps
])
def test_chunked_bf16_gradients(B, T, H, lb, state, final):
    d, cot = _case(B, T, H, 128, 128, 40 + T + H, state=state, final=final)
    gpu = _run(d, cot, B, T, H, 128, 128, 128 ** -0.5, lb, True)
    _check(gpu, _oracle(d, cot, 128 ** -0.5, lb, True), True, d=d)
    assert kda.kda_device_error(1) == 0


def test_chunked_bf16_gradients_without_initial_state_output():
    B, T, H = 2, 100, 2
    d, cot = _case(B, T, H, 128, 128, 77)
    gpu = _run(d, cot, B, T, H, 128, 128, 0.1, -2.0, True, want_state=False)
    _check(gpu, _oracle(d, cot, 0.1, -2.0, True), True, names=GRADS[:-1], d=d)


def test_chunked_bf16_multi_record_ctas_odd_head_count():
    """More (chunk, head) records (16 x 23 = 368) than the prep's persistent CTAs, an odd head
    count (the record walk's head carry) and a partial last chunk, with an initial state and
    a final-state cotangent; three heads compared with the oracle run on each alone (heads
    are independent, the parameter gradients of a head included)."""
    B, T, H = 1, 1000, 23
    d, cot = _case(B, T, H, 128, 128, 61, state=True, final=True)
    lb, scale = -3.0, 128 ** -0.5
    gpu = _run(d, cot, B, T, H, 128, 128, scale, lb, True)
    for h in (0, 11, 22):
        sl = {n: d[n][:, :, h:h + 1] for n in ("q", "k", "v", "g", "beta_logits")}
        sl["a_log"] = d["a_log"][h:h + 1]
        sl["dt_bias"] = d["dt_bias"][:, h:h + 1]
        sl["initial_state"] = d["initial_state"][:, h:h + 1]
        csl = {"d_out": cot["d_out"][:, :, h:h + 1],
               "d_final_state": cot["d_final_state"][:, h:h + 1]}
        ref = _oracle(sl, csl, scale, lb, True)
        got = {n: gpu[n][:, :, h:h + 1] for n in ("dq", "dk", "dv", "dg", "dbeta_logits")}
        got["dinitial_state"] = gpu["dinitial_state"][:, h:h + 1]
        got["da_log"] = gpu["da_log"][h:h + 1]
        got["ddt_bias"] = gpu["ddt_bias"][:, h:h + 1]
        _check(got, ref, True, d=sl)
    assert kda.kda_device_error(1) == 0


def test_chunked_bf16_prefill_workload_sampled_head():
    """The prefill workload's full size (B 4, T 4096, H 32) through the chunked backward,
    every per-token gradient of one sampled (sequence, head) compared with the oracle run on
    that slice alone (sequences and heads are independent; da_log and ddt_bias sum over all
    of them and are checked at the smaller sizes above)."""
    w = synth.PREFILL_B4
    B, T, H, dk, dv = w.B, w.T, w.H, w.dk, w.dv
    d = synth.workload_inputs(w)
    r = np.random.default_rng(11)
    cot = {"d_out": r.standard_normal((B, T, H, dv), dtype=np.float32)}
    gpu = _run(d, cot, B, T, H, dk, dv, w.q_scale, w.lower_bound, True, want_state=True)
    b, h = 2, 19
    sl = {n: d[n][b:b + 1, :, h:h + 1] for n in ("q", "k", "v", "g", "beta_logits")}
    sl["a_log"] = d["a_log"][h:h + 1]
    sl["dt_bias"] = d["dt_bias"][:, h:h + 1]
    sl["initial_state"] = None
    csl = {"d_out": cot["d_out"][b:b + 1, :, h:h + 1]}
    ref = _oracle(sl, csl, w.q_scale, w.lower_bound, True)
    for n in ("dq", "dk", "dv", "dg", "dbeta_logits"):
        got = gpu[n][b:b + 1, :, h:h + 1]
        assert rel_err(got, ref[n]) <= BF16_REL, (n, rel_err(got, ref[n]))
    got = gpu["dinitial_state"][b:b + 1, h:h + 1]
    assert rel_err(got, ref["dinitial_state"]) <= BF16_REL
