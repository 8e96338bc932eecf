"""Parity of kda_recurrent_attention_fwd_ws -- the recurrent page's gated linear recurrence
in its chunked form on the tensor cores (bf16, D = 128, key-axis gates g / gk / g_gamma and
the value-axis gate gv, forward and reverse order) -- with the fp64 oracle ``recurrent_attention``: every
combination of the key-axis gates (none, one, several) with and without gv, grouped key /
value heads, packed sequences with empty and ragged members, gates from mild to the edge of
the supported range [-5, 1], and the benchmark's full workloads (gk; gk + gv) compared
element by element.  Bar: max |gpu - oracle| / max |oracle| <= 2e-2 per tensor, the oracle
fed the same bf16-rounded q, k, v.  Reverse order (the chunks walked from each sequence's
end) is checked the same way."""
import os

import numpy as np
import pytest
import torch

import gated_delta_rule_55_gb300 as kda
from gpu_helpers import (bf16_round, bf16_round32, check_full, check_rel, ensure_built, oracle_pool,
                         to_dev, workspace)
from oracle import recurrent_attention

pytestmark = pytest.mark.gpu
D = 128


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    kda.kda_device_error(reset=True)
    yield
    assert kda.kda_device_error(reset=True) == 0, "a bounded wait gave up"


def _inputs(B, T, Hq, Hkv, seed, gates, state, nseq=None, lo=-0.3, hi=0.0):
    r = np.random.default_rng(2500 + seed)
    d = {"q": r.normal(size=(B, T, Hq, D)), "k": r.normal(size=(B, T, Hkv, D)) * D ** -0.5,
         "v": r.normal(size=(B, T, Hkv, D))}
    for n in ("g", "gk", "gv"):
        d[n] = r.uniform(lo, hi, size=(B, T, Hq, D)) if n in gates else None
    d["g_gamma"] = -r.uniform(0.0, 0.2, size=(B, Hq)) if "g_gamma" in gates else None
    d["s0"] = r.normal(size=(nseq or B, Hq, D, D)) * 0.1 if state else None
    return d


def _run(d, B, T, Hq, Hkv, scale, cu=None, ws=True, reverse=False):
    q, k, v = (to_dev(d[n], torch.bfloat16) for n in ("q", "k", "v"))
    nseq = B if cu is None else len(cu) - 1
    out = torch.full((B, T, Hq, D), float("nan"), device="cuda", dtype=torch.bfloat16)
    s1 = torch.full((nseq, Hq, D, D), float("nan"), device="cuda")
    cu_t = None if cu is None else torch.from_numpy(np.asarray(cu, np.int32)).cuda()
    kw = dict(g=to_dev(d["g"]), g_gamma=to_dev(d["g_gamma"]), gk=to_dev(d["gk"]),
              gv=to_dev(d["gv"]), softmax_scale=scale, initial_state=to_dev(d["s0"]),
              final_state=s1, cu_seqlens=cu_t, N=0 if cu is None else nseq, reverse=reverse)
    if ws:
        nb = kda.kda_recurrent_attention_fwd_workspace_size(
            B, T, Hq, Hkv, D, N=0 if cu is None else nseq, packed=cu is not None,
            value_gate=d["gv"] is not None, reverse=reverse)
        kda.kda_recurrent_attention_fwd_ws(q, k, v, out, B, T, Hq, Hkv, D, workspace=workspace(nb),
                                           **kw)
    else:
        kda.kda_recurrent_attention_fwd(q, k, v, out, B, T, Hq, Hkv, D, **kw)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), s1.cpu().numpy()


def _check(d, out, S, scale, cu=None):
    o = dict(d)
    for n in ("q", "k", "v"):
        o[n] = bf16_round(d[n])
    ro, rs = recurrent_attention(o["q"], o["k"], o["v"], o["g"], o["g_gamma"], o["gk"], o["gv"],
                                 scale, o["s0"], False, cu)
    check_rel(None, "out", out, ro)
    check_rel(None, "final_state", S, rs)


@pytest.mark.parametrize("gates", [(), ("gk",), ("g",), ("g", "gk"), ("gk", "g_gamma"),
                                   ("g_gamma",), ("g", "gk", "g_gamma"), ("gv",), ("gk", "gv"),
                                   ("g", "gv", "g_gamma"), ("g", "gk", "gv", "g_gamma")])
def test_gate_combinations(gates):
    B, T, Hq, Hkv = 2, 200, 4, 2
    d = _inputs(B, T, Hq, Hkv, len(gates), gates, True)
    out, S = _run(d, B, T, Hq, Hkv, None)
    _check(d, out, S, None)


@pytest.mark.parametrize("gates", [("gk",), ("gk", "gv"), ("gv",)])
@pytest.mark.parametrize("lo,hi", [(-5.0, 0.0), (-1.0, 0.05), (-0.05, 0.0)])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 300])
def test_gate_ranges_and_lengths(T, lo, hi, gates):
    B, Hq, Hkv = 1, 2, 1
    d = _inputs(B, T, Hq, Hkv, T, gates, T % 2 == 0, lo=lo, hi=hi)
    out, S = _run(d, B, T, Hq, Hkv, 0.2)
    _check(d, out, S, 0.2)


@pytest.mark.parametrize("gates", [("gk", "g_gamma"), ("gk", "gv", "g_gamma")])
def test_packed_sequences(gates):
    lens = [130, 0, 1, 64, 200, 63]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T, Hq, Hkv = int(cu[-1]), 4, 4
    d = _inputs(1, T, Hq, Hkv, 7, gates, True, nseq=len(lens))
    out, S = _run(d, 1, T, Hq, Hkv, 0.1, cu=cu)
    _check(d, out, S, 0.1, cu)
    # the empty sequence keeps its state (the fp32 copy the device received)
    np.testing.assert_array_equal(S[1], d["s0"][1].astype(np.float32))


@pytest.mark.parametrize("gates", [("gk",), ("gk", "gv")])
def test_many_records_odd_head_count(gates):
    """More (chunk, head) records than the prep's persistent CTAs, an odd query-head count
    in groups of 3 per key / value head."""
    B, T, Hq, Hkv = 2, 1000, 21, 7
    d = _inputs(B, T, Hq, Hkv, 8, gates, True)
    out, S = _run(d, B, T, Hq, Hkv, None)
    _check(d, out, S, None)


def _check_rev(d, out, S, scale, cu=None):
    o = dict(d)
    for n in ("q", "k", "v"):
        o[n] = bf16_round(d[n])
    ro, rs = recurrent_attention(o["q"], o["k"], o["v"], o["g"], o["g_gamma"], o["gk"], o["gv"],
                                 scale, o["s0"], True, cu)
    check_rel(None, "out", out, ro)
    check_rel(None, "final_state", S, rs)


@pytest.mark.parametrize("gates", [(), ("gk",), ("gv",), ("gk", "gv"), ("g", "gk", "g_gamma"),
                                   ("g", "gk", "gv", "g_gamma")])
@pytest.mark.parametrize("T", [1, 63, 64, 90, 200])
def test_reverse_order(gates, T):
    B, Hq, Hkv = 2, 4, 2
    d = _inputs(B, T, Hq, Hkv, 11 + T, gates, True)
    out, S = _run(d, B, T, Hq, Hkv, 0.3, reverse=True)
    _check_rev(d, out, S, 0.3)


@pytest.mark.parametrize("gates", [("gk", "g_gamma"), ("gk", "gv")])
def test_reverse_packed_sequences(gates):
    lens = [130, 0, 1, 64, 200, 63]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T, Hq, Hkv = int(cu[-1]), 4, 2
    d = _inputs(1, T, Hq, Hkv, 17, gates, True, nseq=len(lens))
    out, S = _run(d, 1, T, Hq, Hkv, 0.1, cu=cu, reverse=True)
    _check_rev(d, out, S, 0.1, cu)


def test_reverse_gate_edge_many_records():
    """Gates at the edge of the range, more records than the prep's persistent CTAs."""
    B, T, Hq, Hkv = 2, 1000, 6, 3
    d = _inputs(B, T, Hq, Hkv, 19, ("gk", "gv"), True, lo=-5.0, hi=0.0)
    out, S = _run(d, B, T, Hq, Hkv, None, reverse=True)
    _check_rev(d, out, S, None)


@pytest.mark.parametrize("value_gate", [False, True])
def test_benchmark_workload_full(value_gate):
    """The benchmark's workloads (B=4, T=4096, Hq=32, Hkv=8, D=128, bf16, gk ~ -0.05 U(0, 1),
    and gv ~ -0.05 U(0, 1) for the second, zero initial state): every element of all 128
    (b, h) pairs."""
    B, T, Hq, Hkv = 4, 4096, 32, 8
    r = np.random.default_rng(77)
    d = {"q": r.standard_normal((B, T, Hq, D), dtype=np.float32),
         "k": r.standard_normal((B, T, Hkv, D), dtype=np.float32) * np.float32(D ** -0.5),
         "v": r.standard_normal((B, T, Hkv, D), dtype=np.float32),
         "gk": (-0.05 * r.random((B, T, Hq, D), dtype=np.float32)),
         "g": None, "gv": None, "g_gamma": None, "s0": None}
    if value_gate:
        d["gv"] = -0.05 * r.random((B, T, Hq, D), dtype=np.float32)
    out, S = _run(d, B, T, Hq, Hkv, None)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(S))
    from oracle import pool
    ro, rs = pool.recurrent(oracle_pool(), *(bf16_round32(d[n]) for n in ("q", "k", "v")),
                            None, None, d["gk"], d["gv"], None, None)
    check_full("recurrent B4 T4096 Hq32 Hkv8, gk" + (" + gv" if value_gate else "") +
               ", kda_recurrent_attention_fwd_ws", out, ro, S, rs)


def test_reverse_value_gate_long_sequences():
    """Reverse order with both gates over 128-chunk sequences (B=2, T=8192, Hq=8, Hkv=2,
    initial states), every element against the oracle."""
    B, T, Hq, Hkv = 2, 8192, 8, 2
    d = _inputs(B, T, Hq, Hkv, 23, ("gk", "gv"), True, lo=-0.1, hi=0.0)
    out, S = _run(d, B, T, Hq, Hkv, None, reverse=True)
    from oracle import pool
    ro, rs = pool.recurrent(oracle_pool(), *(bf16_round(d[n]) for n in ("q", "k", "v")),
                            None, None, d["gk"], d["gv"], None, d["s0"], reverse=True)
    check_rel(None, "out", out, ro)
    check_rel(None, "final_state", S, rs)


def test_random_configurations():
    """Seeded random calls: every subset of the gates (g, gk, gv, g_gamma), either order,
    grouped heads (1 to 3 query heads per key / value head), fixed-length or packed inputs
    (empty, one-token and ragged sequences among them), with and without an initial state,
    gate ranges from mild to the edge of the call's contract (the summed key-axis gate and
    the value-axis gate each in [-5, 1]).  The case count is KDA_RANDOM_CASES
    (default 6), so that a longer sweep runs the same code."""
    rng = np.random.default_rng(4242)
    names = ("g", "gk", "gv", "g_gamma")
    for case in range(int(os.environ.get("KDA_RANDOM_CASES", "6"))):
        gates = tuple(n for n in names if rng.random() < 0.5)
        Hkv = int(rng.integers(1, 4))
        Hq = Hkv * int(rng.integers(1, 4))
        rev = bool(rng.integers(0, 2))
        state = bool(rng.integers(0, 2))
        lo, hi = [(-0.3, 0.0), (-5.0, 0.0), (-1.0, 0.05)][int(rng.integers(0, 3))]
        if "g" in gates and "gk" in gates:
            # the summed key-axis gate g + gk + g_gamma stays in [-5, 1] (g_gamma >= -0.2)
            lo = max(lo, -2.4)
        scale = [None, 0.1, 0.3][int(rng.integers(0, 3))]
        if rng.random() < 0.5:
            lens = [int(x) for x in rng.integers(0, 300, int(rng.integers(1, 6)))]
            if case % 2 == 0:
                lens[int(rng.integers(0, len(lens)))] = int(rng.integers(0, 2))
            if sum(lens) == 0:
                lens[0] = 29
            cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
            B, T, nseq = 1, int(cu[-1]), len(lens)
        else:
            cu, B, T, nseq = None, int(rng.integers(1, 3)), int(rng.integers(1, 400)), None
        d = _inputs(B, T, Hq, Hkv, 900 + case, gates, state, nseq=nseq, lo=lo, hi=hi)
        out, S = _run(d, B, T, Hq, Hkv, scale, cu=cu, reverse=rev)
        o = dict(d)
        for n in ("q", "k", "v"):
            o[n] = bf16_round(d[n])
        ro, rs = recurrent_attention(o["q"], o["k"], o["v"], o["g"], o["g_gamma"], o["gk"],
                                     o["gv"], scale, o["s0"], rev, cu)
        label = (f"random_rec[{case}: gates={'+'.join(gates) or 'none'} Hq={Hq} Hkv={Hkv} "
                 f"rev={int(rev)} packed={int(cu is not None)} T={T}]")
        check_rel(label, "out", out, ro)
        check_rel(label, "final_state", S, rs)


def test_gate_outside_the_range_is_reported():
    """Gates outside the chunked path's range (the summed key-axis gate and the value-axis
    gate each in [-5, 1]): the call completes and records bit 5 of kda_device_error; inside
    the range nothing is recorded."""
    B, T, Hq, Hkv = 1, 100, 2, 1
    kda.kda_device_error(reset=True)
    d = _inputs(B, T, Hq, Hkv, 31, ("gk",), False, lo=-4.0, hi=-4.0)  # inside
    _run(d, B, T, Hq, Hkv, None)
    assert kda.kda_device_error(reset=True) == 0
    d = _inputs(B, T, Hq, Hkv, 31, ("g", "gk"), False, lo=-4.0, hi=-4.0)  # sum -8
    _run(d, B, T, Hq, Hkv, None)
    assert kda.kda_device_error(reset=True) == 32
    d = _inputs(B, T, Hq, Hkv, 32, ("gv",), False, lo=1.5, hi=1.5)  # value gate above 1
    _run(d, B, T, Hq, Hkv, None, reverse=True)
    assert kda.kda_device_error(reset=True) == 32
