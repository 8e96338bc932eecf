"""The training pair: kda_chunk_fwd_train (the forward, keeping the backward's records in the
workspace) and kda_chunk_bwd_saved (the backward reading them).

The forward is compared with the oracle's forward and with kda_chunk_fwd_ws (bf16: max-norm
relative error <= 2e-2 against the oracle fed the same bf16-rounded q, k, v); the saved
backward with kda_chunk_bwd on the same inputs (both run the same reverse kernels on
identical records: equal gradients, da_log / ddt_bias up to the order of their atomic sums)
and with the oracle backward."""
import numpy as np
import pytest
import torch

import gated_delta_rule_55_gb300 as kda
from gated_delta_rule_55_gb300 import synth
from gpu_helpers import (BF16_REL, bf16_round, bwd_err, ensure_built, param_grad_scales, rel_err,
                         run_chunk, to_dev, workspace)
from oracle import kda_backward, kda_forward

pytestmark = pytest.mark.gpu

GRADS = ("dq", "dk", "dv", "dg", "dbeta_logits", "da_log", "ddt_bias", "dinitial_state")


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _grads(B, T, H):
    io = torch.bfloat16
    return {"dq": torch.full((B, T, H, 128), float("nan"), device="cuda", dtype=io),
            "dk": torch.full((B, T, H, 128), float("nan"), device="cuda", dtype=io),
            "dv": torch.full((B, T, H, 128), float("nan"), device="cuda", dtype=io),
            "dg": torch.full((B, T, H, 128), float("nan"), device="cuda"),
            "dbeta_logits": torch.full((B, T, H), float("nan"), device="cuda"),
            "da_log": torch.full((H,), float("nan"), device="cuda"),
            "ddt_bias": torch.full((128, H), float("nan"), device="cuda"),
            "dinitial_state": torch.full((B, H, 128, 128), float("nan"), device="cuda")}


def _train_pair(d, cot, B, T, H, scale, lb):
    io = torch.bfloat16
    q, k, v = (to_dev(d[n], io) for n in ("q", "k", "v"))
    g, bl, al, db = (to_dev(d[n]) for n in ("g", "beta_logits", "a_log", "dt_bias"))
    s0 = to_dev(d.get("initial_state"))
    out = torch.full((B, T, H, 128), float("nan"), device="cuda", dtype=io)
    s1 = torch.full((B, H, 128, 128), float("nan"), device="cuda")
    w = workspace(kda.kda_chunk_bwd_workspace_size(B, T, H, 128, 128, kda.KDA_BF16))
    kda.kda_chunk_fwd_train(q, k, v, g, bl, al, db, scale, lb, s0, out, s1, B, T, H, 128, 128,
                            workspace=w)
    dout = to_dev(cot["d_out"], io)
    dfin = to_dev(cot.get("d_final_state"))
    saved, fresh = _grads(B, T, H), _grads(B, T, H)
    kda.kda_chunk_bwd_saved(q, k, v, g, bl, al, db, scale, lb, s0, dout, dfin, saved["dq"],
                            saved["dk"], saved["dv"], saved["dg"], saved["dbeta_logits"],
                            saved["da_log"], saved["ddt_bias"], saved["dinitial_state"], B, T,
                            H, 128, 128, workspace=w)
    w2 = workspace(kda.kda_chunk_bwd_workspace_size(B, T, H, 128, 128, kda.KDA_BF16))
    kda.kda_chunk_bwd(q, k, v, g, bl, al, db, scale, lb, s0, dout, dfin, fresh["dq"],
                      fresh["dk"], fresh["dv"], fresh["dg"], fresh["dbeta_logits"],
                      fresh["da_log"], fresh["ddt_bias"], fresh["dinitial_state"], B, T, H, 128,
                      128, workspace=w2)
    torch.cuda.synchronize()
    np_ = lambda t: t.float().cpu().numpy()  # noqa: E731
    return (np_(out), np_(s1), {n: np_(t) for n, t in saved.items()},
            {n: np_(t) for n, t in fresh.items()})


@pytest.mark.parametrize("B,T,H,lb,final", [
    (1, 64, 2, -2.0, True),
    (2, 300, 2, -5.0, True),
    (1, 130, 3, -1.0, False),
])
def test_train_forward_and_saved_backward(B, T, H, lb, final):
    d = synth.chunk_inputs(B, T, H, 128, 128, 60 + T, 0.1)
    r = np.random.default_rng(960 + T)
    cot = {"d_out": r.normal(size=(B, T, H, 128))}
    if final:
        cot["d_final_state"] = r.normal(size=(B, H, 128, 128))
    scale = 128 ** -0.5
    out, s1, saved, fresh = _train_pair(d, cot, B, T, H, scale, lb)

    o = dict(d)
    for n in ("q", "k", "v"):
        o[n] = bf16_round(d[n])
    ref_out, ref_S = kda_forward(o["q"], o["k"], o["v"], o["g"], o["beta_logits"], o["a_log"],
                                 o["dt_bias"], scale, lb, o["initial_state"])
    assert rel_err(out, ref_out) <= BF16_REL
    assert rel_err(s1, ref_S) <= BF16_REL
    ws_out, ws_S = run_chunk(d, B, T, H, 128, 128, scale, lb, 64, True, ws=True)
    assert rel_err(out, ws_out) <= 1e-2
    assert rel_err(s1, ws_S) <= 1e-5

    for n in GRADS:
        if n in ("da_log", "ddt_bias"):
            assert rel_err(saved[n], fresh[n]) <= 1e-5, n
        else:
            assert np.array_equal(saved[n], fresh[n]), n
    c = dict(cot)
    c["d_out"] = bf16_round(cot["d_out"])
    ref = kda_backward(o["q"], o["k"], o["v"], o["g"], o["beta_logits"], o["a_log"],
                       o["dt_bias"], c["d_out"], c.get("d_final_state"), scale, lb,
                       o["initial_state"])
    scales = param_grad_scales(ref["dg"], d["g"], d["dt_bias"])
    for n in GRADS:
        e = bwd_err(n, saved[n], ref[n], scales)
        assert e <= BF16_REL, (n, e)
    assert kda.kda_device_error(1) == 0
