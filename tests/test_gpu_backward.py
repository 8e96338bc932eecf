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
from gpu_helpers import BF16_REL, bf16_round, ensure_built, max_abs, rel_err, to_dev, workspace
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
    w = workspace(kda.kda_chunk_bwd_workspace_size(B, T, H, dk, dv))
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


def _check(gpu, ref, bf16, names=GRADS):
    for n in names:
        if bf16:
            assert rel_err(gpu[n], ref[n]) <= BF16_REL, (n, rel_err(gpu[n], ref[n]))
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
    _check(gpu, _oracle(d, cot, 0.1, -2.0, bf16), bf16)


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
