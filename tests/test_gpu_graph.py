"""The C-ABI calls recorded in a CUDA graph.

Every entry point enqueues its launches (and the backward's two memsets) on the caller's
stream with no host synchronisation, allocation or device-to-host read, so a stream capture
records the whole call and a replay recomputes it from whatever the input buffers hold then.
Each test runs a call eagerly, captures the same call on the same buffers, replays it, and
requires the replay to reproduce the eager results bit for bit (the eager results are the
ones the parity tests compare with the oracle); the backward's two parameter gradients are
sums of atomic adds whose order varies, so they are compared to 1e-5 of their magnitude.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_55_gb300 as kda
from gated_delta_rule_55_gb300 import synth
from gpu_helpers import ensure_built, to_dev, workspace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    kda.kda_device_error(reset=True)
    yield
    assert kda.kda_device_error(reset=True) == 0, "a bounded wait gave up"


def _capture(fn):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def _same(a, b, what):
    a, b = a.cpu(), b.cpu()
    assert torch.equal(a.view(torch.uint8) if a.dtype == torch.bfloat16 else a,
                       b.view(torch.uint8) if b.dtype == torch.bfloat16 else b), what


def _prefill(B, T, H, seed):
    d = synth.chunk_inputs(B, T, H, 128, 128, seed, 0.1)
    x = {n: to_dev(d[n], torch.bfloat16) for n in ("q", "k", "v")}
    for n in ("g", "beta_logits", "a_log", "dt_bias", "initial_state"):
        x[n] = to_dev(d[n])
    x["out"] = torch.empty(B, T, H, 128, device="cuda", dtype=torch.bfloat16)
    x["final_state"] = torch.empty(B, H, 128, 128, device="cuda")
    return x


def _fwd_args(x):
    return (x["q"], x["k"], x["v"], x["g"], x["beta_logits"], x["a_log"], x["dt_bias"],
            128 ** -0.5, -5.0, x["initial_state"], x["out"], x["final_state"])


def test_chunk_fwd_ws_replay_and_new_inputs():
    B, T, H = 2, 300, 3
    x = _prefill(B, T, H, 41)
    w = workspace(kda.kda_chunk_fwd_workspace_size(B, T, H, 128, 128, 64))

    def call():
        kda.kda_chunk_fwd_ws(*_fwd_args(x), B, T, H, 128, 128, 64, workspace=w)

    call()
    torch.cuda.synchronize()
    out0, s0 = x["out"].clone(), x["final_state"].clone()
    g = _capture(call)
    x["out"].fill_(float("nan"))
    x["final_state"].fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    _same(x["out"], out0, "out")
    _same(x["final_state"], s0, "final_state")
    # new values in the same buffers: the replay follows them
    d2 = synth.chunk_inputs(B, T, H, 128, 128, 42, 0.1)
    x["q"].copy_(to_dev(d2["q"], torch.bfloat16))
    x["g"].copy_(to_dev(d2["g"]))
    g.replay()
    torch.cuda.synchronize()
    out_g, s_g = x["out"].clone(), x["final_state"].clone()
    call()
    torch.cuda.synchronize()
    _same(out_g, x["out"], "out after new inputs")
    _same(s_g, x["final_state"], "final_state after new inputs")
    assert not torch.equal(out_g.cpu(), out0.cpu())


def test_chunk_fwd_noalloc_replay():
    B, T, H = 1, 200, 2
    x = _prefill(B, T, H, 43)

    def call():
        kda.kda_chunk_fwd_noalloc(*_fwd_args(x), B, T, H, 128, 128, 64)

    call()  # the first call looks up the scratch array, before any capture
    torch.cuda.synchronize()
    out0, s0 = x["out"].clone(), x["final_state"].clone()
    g = _capture(call)
    x["out"].fill_(float("nan"))
    x["final_state"].fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    _same(x["out"], out0, "out")
    _same(x["final_state"], s0, "final_state")


def test_varlen_split_chains_replay():
    # the longest sequence (41 chunks) is split: plan, prep, scan and fix-up launches
    lengths = [64 * 40 + 5, 300, 64 * 20, 1]
    H = 4
    d = synth.varlen_inputs(lengths, H, 128, 128, 44)
    total, N = int(sum(lengths)), len(lengths)
    x = {n: to_dev(d[n], torch.bfloat16) for n in ("q", "k", "v")}
    for n in ("g", "beta_logits", "a_log", "dt_bias", "initial_state"):
        x[n] = to_dev(d[n])
    cu = torch.from_numpy(d["cu_seqlens"].astype(np.int32)).cuda()
    out = torch.empty(total, H, 128, device="cuda", dtype=torch.bfloat16)
    s1 = torch.empty(N, H, 128, 128, device="cuda")
    w = workspace(kda.kda_chunk_fwd_varlen_workspace_size(N, total, H, 128, 128, 64))

    def call():
        kda.kda_chunk_fwd_varlen_ws(x["q"], x["k"], x["v"], x["g"], x["beta_logits"],
                                    x["a_log"], x["dt_bias"], 128 ** -0.5, -5.0, cu, N, total,
                                    x["initial_state"], out, s1, H, 128, 128, 64, workspace=w)

    call()
    torch.cuda.synchronize()
    out0, s0 = out.clone(), s1.clone()
    g = _capture(call)
    out.fill_(float("nan"))
    s1.fill_(float("nan"))
    w.fill_(0xFF)  # the replay rebuilds the plan and every record
    g.replay()
    torch.cuda.synchronize()
    _same(out, out0, "out")
    _same(s1, s0, "final_state")


def test_decode_steps_replay():
    B, H, steps = 8, 4, 4
    S0 = to_dev(synth.decode_state(B, H, 128, 128, 45))
    a_log, dt_bias = (to_dev(t) for t in synth.gate_params(H, 128, 45))
    toks = [{n: to_dev(t) for n, t in synth.decode_token_inputs(B, H, 128, 128, 45, s).items()}
            for s in range(steps)]
    outs = [torch.empty(B, H, 128, device="cuda") for _ in range(steps)]
    S = S0.clone()

    def call():
        for s in range(steps):
            t = toks[s]
            kda.kda_decode_step(t["q"], t["k"], t["v"], t["g"], t["beta_logits"], a_log,
                                dt_bias, 128 ** -0.5, -5.0, outs[s], S, B, H, 128, 128)

    call()
    torch.cuda.synchronize()
    ref_S, ref_o = S.clone(), [o.clone() for o in outs]
    g = _capture(call)
    S.copy_(S0)
    for o in outs:
        o.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    _same(S, ref_S, "state after the chained steps")
    for s in range(steps):
        _same(outs[s], ref_o[s], f"out of step {s}")


def test_chunk_bwd_replay():
    B, T, H = 1, 200, 2
    x = _prefill(B, T, H, 46)
    r = np.random.default_rng(46)
    d_out = torch.from_numpy(r.standard_normal((B, T, H, 128), dtype=np.float32)).to(
        "cuda", torch.bfloat16)
    d_fin = torch.from_numpy(r.standard_normal((B, H, 128, 128), dtype=np.float32) * 0.1).cuda()
    grads = {
        "dq": torch.empty(B, T, H, 128, device="cuda", dtype=torch.bfloat16),
        "dk": torch.empty(B, T, H, 128, device="cuda", dtype=torch.bfloat16),
        "dv": torch.empty(B, T, H, 128, device="cuda", dtype=torch.bfloat16),
        "dg": torch.empty(B, T, H, 128, device="cuda"),
        "dbeta_logits": torch.empty(B, T, H, device="cuda"),
        "da_log": torch.empty(H, device="cuda"),
        "ddt_bias": torch.empty(128, H, device="cuda"),
        "d_initial_state": torch.empty(B, H, 128, 128, device="cuda"),
    }
    w = workspace(kda.kda_chunk_bwd_workspace_size(B, T, H, 128, 128))

    def call():
        kda.kda_chunk_bwd(x["q"], x["k"], x["v"], x["g"], x["beta_logits"], x["a_log"],
                          x["dt_bias"], 128 ** -0.5, -5.0, x["initial_state"], d_out, d_fin,
                          grads["dq"], grads["dk"], grads["dv"], grads["dg"],
                          grads["dbeta_logits"], grads["da_log"], grads["ddt_bias"],
                          grads["d_initial_state"], B, T, H, 128, 128, workspace=w)

    call()
    torch.cuda.synchronize()
    ref = {n: t.clone() for n, t in grads.items()}
    g = _capture(call)
    for t in grads.values():
        t.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    for n, t in grads.items():
        if n in ("da_log", "ddt_bias"):  # atomic sums: order-dependent rounding
            a, b = t.cpu().double(), ref[n].cpu().double()
            assert torch.all(torch.isfinite(a))
            assert float((a - b).abs().max()) <= 1e-5 * max(float(b.abs().max()), 1e-30), n
        else:
            _same(t, ref[n], n)


def test_recurrent_attention_chunked_replay():
    B, T, Hq, Hkv, D = 1, 200, 4, 2, 128
    r = np.random.default_rng(47)
    q = torch.from_numpy(r.standard_normal((B, T, Hq, D), dtype=np.float32)).to(
        "cuda", torch.bfloat16)
    k = torch.from_numpy(r.standard_normal((B, T, Hkv, D), dtype=np.float32) / np.sqrt(D)).to(
        "cuda", torch.bfloat16)
    v = torch.from_numpy(r.standard_normal((B, T, Hkv, D), dtype=np.float32)).to(
        "cuda", torch.bfloat16)
    gk = torch.from_numpy(-0.05 * r.random((B, T, Hq, D), dtype=np.float32)).cuda()  # [B,T,Hq,D]
    gv = torch.from_numpy(-0.05 * r.random((B, T, Hq, D), dtype=np.float32)).cuda()
    out = torch.empty(B, T, Hq, D, device="cuda", dtype=torch.bfloat16)
    fs = torch.empty(B, Hq, D, D, device="cuda")
    nbytes = kda.kda_recurrent_attention_fwd_workspace_size(B, T, Hq, Hkv, D, value_gate=True)
    assert nbytes > 0
    w = workspace(nbytes)

    def call():
        kda.kda_recurrent_attention_fwd_ws(q, k, v, out, B, T, Hq, Hkv, D, gk=gk, gv=gv,
                                           final_state=fs, workspace=w)

    call()
    torch.cuda.synchronize()
    out0, fs0 = out.clone(), fs.clone()
    g = _capture(call)
    out.fill_(float("nan"))
    fs.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    _same(out, out0, "out")
    _same(fs, fs0, "final_state")
