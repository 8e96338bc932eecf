"""Parity of kda_attention_fwd (the kernel_delta_attention call: per-head log-decay, beta
as given, use_qk_l2norm, use_chunked, order) with the fp64 oracle ``kda_attention``.

fp32 q/k/v: max |gpu - oracle| <= 1e-4; bf16: max |gpu - oracle| / max |oracle| <= 2e-2,
the oracle fed the same bf16-rounded values.  Keys and queries for the runs without L2
normalisation are drawn with norm about 1 (unnormalised N(0, 1) keys make the delta rule
itself diverge: |k|^2 ~ dk)."""
import numpy as np
import pytest
import torch

import gated_delta_rule_55_gb300 as kda
from gpu_helpers import BF16_REL, F32_ATOL, bf16_round, ensure_built, max_abs, rel_err, to_dev
from oracle import kda_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _inputs(B, T, H, dk, dv, seed, norm, decay, state):
    r = np.random.default_rng(500 + seed)
    s = 1.0 if norm else dk ** -0.5
    d = {"q": r.normal(size=(B, T, H, dk)) * s, "k": r.normal(size=(B, T, H, dk)) * s,
         "v": r.normal(size=(B, T, H, dv)), "beta": r.uniform(0.0, 1.0, size=(B, T, H))}
    d["decay"] = None if decay is None else (
        -r.uniform(0.0, 1.5, size=(B, T, H)) if decay == "neg" else
        r.normal(size=(B, T, H)) * -0.01)  # the page's example: N(0, 1) * -0.01
    d["s0"] = r.normal(size=(B, H, dk, dv)) * 0.1 if state else None
    return d


def _run(d, B, T, H, dk, dv, scale, norm, chunked, order, bf16, chunk=64):
    io = torch.bfloat16 if bf16 else torch.float32
    q, k, v = (to_dev(d[n], io) for n in ("q", "k", "v"))
    out = torch.full((B, T, H, dv), float("nan"), device="cuda", dtype=io)
    s1 = torch.full((B, H, dk, dv), float("nan"), device="cuda")
    kda.kda_attention_fwd(q, k, v, to_dev(d["beta"]), to_dev(d["decay"]), to_dev(d["s0"]), out,
                          s1, B, T, H, dk, dv, softmax_scale=scale, chunk=chunk,
                          use_qk_l2norm=norm, use_chunked=chunked, order=order)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), s1.cpu().numpy()


def _check(d, out, S, scale, norm, order, bf16):
    o = dict(d)
    if bf16:
        for n in ("q", "k", "v"):
            o[n] = bf16_round(d[n])
    ref_o, ref_S = kda_attention(o["q"], o["k"], o["v"], o["beta"], o["decay"], o["s0"], scale,
                                 norm, order)
    if bf16:
        assert rel_err(out, ref_o) <= BF16_REL, rel_err(out, ref_o)
        assert rel_err(S, ref_S) <= BF16_REL, rel_err(S, ref_S)
    else:
        assert max_abs(out, ref_o) <= F32_ATOL, max_abs(out, ref_o)
        assert max_abs(S, ref_S) <= F32_ATOL, max_abs(S, ref_S)


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("order", ["decay_first", "literal"])
@pytest.mark.parametrize("norm", [True, False])
@pytest.mark.parametrize("chunked", [True, False])
def test_variants(chunked, norm, order, bf16):
    B, T, H, dk, dv = 2, 77, 2, 128, 64
    d = _inputs(B, T, H, dk, dv, 1, norm, "neg", True)
    out, S = _run(d, B, T, H, dk, dv, 0.3, norm, chunked, order, bf16)
    _check(d, out, S, 0.3, norm, order, bf16)


@pytest.mark.parametrize("chunked", [True, False])
@pytest.mark.parametrize("decay", [None, "page"])
def test_default_decay_and_scale(decay, chunked):
    """decay None (full retention) and the page's example decays (small, either sign);
    softmax_scale None -> dk^-0.5."""
    B, T, H, dk, dv = 1, 64, 3, 64, 32
    d = _inputs(B, T, H, dk, dv, 2, True, decay, False)
    out, S = _run(d, B, T, H, dk, dv, None, True, chunked, "decay_first", False, chunk=16)
    _check(d, out, S, None, True, "decay_first", False)


@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 32)])
def test_head_dims_recurrent_and_chunked_agree_with_oracle(dk, dv):
    B, T, H = 2, 40, 2
    d = _inputs(B, T, H, dk, dv, dk + dv, True, "neg", True)
    for chunked in (True, False):
        out, S = _run(d, B, T, H, dk, dv, 0.2, True, chunked, "decay_first", False)
        _check(d, out, S, 0.2, True, "decay_first", False)


def test_empty_sequence_passes_state_through():
    d = _inputs(2, 1, 2, 32, 32, 3, True, None, True)
    s0 = to_dev(d["s0"])
    for chunked in (True, False):
        s1 = torch.full_like(s0, float("nan"))
        dummy = torch.zeros(16, device="cuda")
        kda.kda_attention_fwd(dummy, dummy, dummy, dummy, None, s0, dummy, s1, 2, 0, 2, 32, 32,
                              use_chunked=chunked)
        torch.cuda.synchronize()
        assert torch.equal(s1, s0)


def test_recurrent_longer_sequence_bf16():
    """A longer scan (T = 700) through the recurrent kernel, bf16."""
    B, T, H, dk, dv = 1, 700, 2, 128, 128
    d = _inputs(B, T, H, dk, dv, 4, True, "neg", True)
    out, S = _run(d, B, T, H, dk, dv, 0.1, True, False, "decay_first", True)
    _check(d, out, S, 0.1, True, "decay_first", True)
