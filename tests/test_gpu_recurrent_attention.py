"""Parity of kda_recurrent_attention_fwd (the recurrent page's gated linear recurrence)
with the fp64 oracle ``recurrent_attention``.

fp32: max |gpu - oracle| <= 1e-4 * max(1, max |oracle|) per tensor; bf16: max |gpu - oracle|
/ max |oracle| <= 2e-2 per tensor, the oracle fed the same bf16-rounded q, k, v."""
import numpy as np
import pytest
import torch

import gated_delta_rule_55_gb300 as kda
from gpu_helpers import BF16_REL, bf16_round, ensure_built, max_abs, rel_err, to_dev
from oracle import recurrent_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _inputs(B, T, Hq, Hkv, D, seed, gates, state, nseq=None):
    r = np.random.default_rng(1500 + seed)
    d = {"q": r.normal(size=(B, T, Hq, D)), "k": r.normal(size=(B, T, Hkv, D)) * D ** -0.5,
         "v": r.normal(size=(B, T, Hkv, D))}
    for n in ("g", "gk", "gv"):
        d[n] = -r.uniform(0.0, 0.3, size=(B, T, Hq, D)) if n in gates else None
    d["g_gamma"] = -r.uniform(0.0, 0.2, size=(B, Hq)) if "g_gamma" in gates else None
    d["s0"] = r.normal(size=(nseq or B, Hq, D, D)) * 0.1 if state else None
    return d


def _run(d, B, T, Hq, Hkv, D, scale, reverse, bf16, cu=None):
    io = torch.bfloat16 if bf16 else torch.float32
    q, k, v = (to_dev(d[n], io) for n in ("q", "k", "v"))
    nseq = B if cu is None else len(cu) - 1
    out = torch.full((B, T, Hq, D), float("nan"), device="cuda", dtype=io)
    s1 = torch.full((nseq, Hq, D, D), float("nan"), device="cuda")
    cu_t = None if cu is None else torch.from_numpy(np.asarray(cu, np.int32)).cuda()
    kda.kda_recurrent_attention_fwd(q, k, v, out, B, T, Hq, Hkv, D, g=to_dev(d["g"]),
                                    g_gamma=to_dev(d["g_gamma"]), gk=to_dev(d["gk"]),
                                    gv=to_dev(d["gv"]), softmax_scale=scale,
                                    initial_state=to_dev(d["s0"]), final_state=s1,
                                    cu_seqlens=cu_t, N=0 if cu is None else nseq,
                                    reverse=reverse)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), s1.cpu().numpy()


def _check(d, out, S, scale, reverse, bf16, cu=None):
    o = dict(d)
    if bf16:
        for n in ("q", "k", "v"):
            o[n] = bf16_round(d[n])
    ro, rs = recurrent_attention(o["q"], o["k"], o["v"], o["g"], o["g_gamma"], o["gk"], o["gv"],
                                 scale, o["s0"], reverse, cu)
    for gpu, ref in ((out, ro), (S, rs)):
        if bf16:
            assert rel_err(gpu, ref) <= BF16_REL, rel_err(gpu, ref)
        else:
            tol = 1e-4 * max(1.0, float(np.max(np.abs(ref))))
            assert max_abs(gpu, ref) <= tol, (max_abs(gpu, ref), tol)


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("reverse", [False, True])
@pytest.mark.parametrize("gates", [(), ("g", "gk", "gv", "g_gamma"), ("gk",), ("gv", "g_gamma")])
def test_gates_reverse_dtypes(gates, reverse, bf16):
    B, T, Hq, Hkv, D = 2, 70, 4, 2, 64
    d = _inputs(B, T, Hq, Hkv, D, len(gates), gates, True)
    out, S = _run(d, B, T, Hq, Hkv, D, 0.2, reverse, bf16)
    _check(d, out, S, 0.2, reverse, bf16)


@pytest.mark.parametrize("D", [32, 128])
def test_head_dims_default_scale_mha(D):
    B, T, H = 1, 45, 3
    d = _inputs(B, T, H, H, D, D, ("gk", "gv"), False)
    out, S = _run(d, B, T, H, H, D, None, False, False)
    _check(d, out, S, None, False, False)


@pytest.mark.parametrize("reverse", [False, True])
def test_packed_sequences(reverse):
    lens = [17, 0, 1, 40, 9]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T, Hq, Hkv, D = int(cu[-1]), 2, 1, 32
    d = _inputs(1, T, Hq, Hkv, D, 7, ("g", "gv"), True, nseq=len(lens))
    out, S = _run(d, 1, T, Hq, Hkv, D, 0.5, reverse, False, cu=cu)
    _check(d, out, S, 0.5, reverse, False, cu=cu)
    # the empty sequence keeps its (fp32) initial state exactly
    np.testing.assert_array_equal(S[1], d["s0"][1].astype(np.float32))
