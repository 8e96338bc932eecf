"""Parity of kda_chunk_fwd / kda_chunk_fwd_varlen with the fp64 oracle, through the C ABI.

fp32 q/k/v: max |gpu - oracle| <= 1e-4.  bf16 q/k/v: max |gpu - oracle| / max |oracle|
<= 2e-2 per tensor (out and final state), the oracle fed the same bf16-rounded values.
Sizes span several chunks and a ragged last chunk; the full-size workloads are compared
element by element over every (sequence, head) pair, the oracle running over the pairs in a
pool of host processes.
"""
import numpy as np
import pytest
import torch

from gated_delta_rule_55_gb300 import kda_chunk_fwd, synth
from gpu_helpers import (BF16_REL, F32_ATOL, check_full, check_rel, ensure_built, max_abs, oracle_inputs,
                         rel_err, run_chunk, run_varlen, to_dev, workload_reference)
from oracle import kda_forward, kda_forward_varlen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _check(gpu_out, gpu_state, ref_out, ref_state, bf16):
    if bf16:
        check_rel(None, "out", gpu_out, ref_out)
        if gpu_state is not None:
            check_rel(None, "final_state", gpu_state, ref_state)
    else:
        assert max_abs(gpu_out, ref_out) <= F32_ATOL, max_abs(gpu_out, ref_out)
        if gpu_state is not None:
            assert max_abs(gpu_state, ref_state) <= F32_ATOL, max_abs(gpu_state, ref_state)


def _case(B, T, H, dk, dv, lb, chunk, bf16, seed, state_std=0.1, scale=None):
    d = synth.chunk_inputs(B, T, H, dk, dv, seed, state_std)
    scale = dk ** -0.5 if scale is None else scale
    out, S = run_chunk(d, B, T, H, dk, dv, scale, lb, chunk, bf16)
    o = oracle_inputs(d, bf16)
    ref_out, ref_S = kda_forward(o["q"], o["k"], o["v"], o["g"], o["beta_logits"], o["a_log"],
                                 o["dt_bias"], scale, lb, o["initial_state"])
    _check(out, S, ref_out, ref_S, bf16)


def test_tiny_fp32_workload():
    """B=1, T=64, H=2, dk=dv=32, fp32, chunk 16, zero initial state, seed 0."""
    w = synth.TINY_F32
    d = synth.workload_inputs(w)
    out, S = run_chunk(d, w.B, w.T, w.H, w.dk, w.dv, w.q_scale, w.lower_bound, w.chunk, False)
    ref_out, ref_S = kda_forward(d["q"], d["k"], d["v"], d["g"], d["beta_logits"], d["a_log"],
                                 d["dt_bias"], w.q_scale, w.lower_bound, None)
    _check(out, S, ref_out, ref_S, False)


@pytest.mark.parametrize("lb", [-5.0, -0.05])
@pytest.mark.parametrize("chunk", [16, 64])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (128, 32), (32, 64)])
def test_fp32_ragged(dk, dv, chunk, lb):
    _case(B=2, T=150, H=2, dk=dk, dv=dv, lb=lb, chunk=chunk, bf16=False, seed=dk + dv + chunk)


@pytest.mark.parametrize("lb", [-5.0, -0.05])
@pytest.mark.parametrize("chunk", [16, 64])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 300])
def test_bf16_ragged(T, chunk, lb):
    _case(B=2, T=T, H=3, dk=128, dv=128, lb=lb, chunk=chunk, bf16=True, seed=T + chunk)


def test_bf16_small_head_dims():
    _case(B=1, T=97, H=2, dk=64, dv=32, lb=-1.0, chunk=64, bf16=True, seed=5)


def test_no_decay_lower_bound_zero():
    _case(B=1, T=130, H=2, dk=64, dv=64, lb=0.0, chunk=64, bf16=False, seed=6)


def test_empty_sequence_returns_initial_state():
    """T = 0: nothing to read or write but the state, which passes through unchanged."""
    d = synth.chunk_inputs(2, 1, 2, 32, 32, 1, state_std=0.3)
    s0 = to_dev(d["initial_state"])
    s1 = torch.full_like(s0, float("nan"))
    dummy = torch.zeros(16, device="cuda")  # zero-size tensors still need aligned addresses
    kda_chunk_fwd(dummy, dummy, dummy, dummy, dummy, to_dev(d["a_log"]), to_dev(d["dt_bias"]),
                  0.2, -1.0, s0, dummy, s1, 2, 0, 2, 32, 32, 16, dtype=0)
    torch.cuda.synchronize()
    assert torch.equal(s1, s0)


def test_state_passthrough_two_calls_equal_one():
    """kernel_delta_attention initial_state / return_state: splitting a sequence and
    passing the state through equals one pass (on the GPU path itself)."""
    B, T, H, dk, dv = 2, 200, 2, 128, 64
    d = synth.chunk_inputs(B, T, H, dk, dv, 11, state_std=0.2)
    full_o, full_S = run_chunk(d, B, T, H, dk, dv, 0.1, -0.5, 64, False)
    cut = 77
    d1 = {n: (x[:, :cut] if n in ("q", "k", "v", "g", "beta_logits") else x) for n, x in d.items()}
    d2 = {n: (x[:, cut:] if n in ("q", "k", "v", "g", "beta_logits") else x) for n, x in d.items()}
    o1, S1 = run_chunk(d1, B, cut, H, dk, dv, 0.1, -0.5, 64, False)
    d2["initial_state"] = S1
    o2, S2 = run_chunk(d2, B, T - cut, H, dk, dv, 0.1, -0.5, 64, False)
    assert max_abs(np.concatenate([o1, o2], 1), full_o) <= F32_ATOL
    assert max_abs(S2, full_S) <= F32_ATOL


def test_final_state_may_alias_initial_state():
    B, T, H, dk, dv = 1, 100, 2, 64, 64
    d = synth.chunk_inputs(B, T, H, dk, dv, 12, state_std=0.2)
    io = torch.float32
    s = to_dev(d["initial_state"])
    out = torch.empty(B, T, H, dv, device="cuda")
    kda_chunk_fwd(*(to_dev(d[n], io) for n in ("q", "k", "v")), to_dev(d["g"]),
                  to_dev(d["beta_logits"]), to_dev(d["a_log"]), to_dev(d["dt_bias"]), 0.2, -2.0,
                  s, out, s, B, T, H, dk, dv, 64)
    torch.cuda.synchronize()
    ref_o, ref_S = kda_forward(d["q"], d["k"], d["v"], d["g"], d["beta_logits"], d["a_log"],
                               d["dt_bias"], 0.2, -2.0, d["initial_state"])
    assert max_abs(out.cpu().numpy(), ref_o) <= F32_ATOL
    assert max_abs(s.cpu().numpy(), ref_S) <= F32_ATOL


@pytest.mark.parametrize("bf16", [False, True])
def test_varlen_small_with_empty_and_ragged_sequences(bf16):
    lens = [70, 0, 1, 129, 64, 5]
    H, dk, dv = 2, 128, 64
    d = synth.varlen_inputs(lens, H, dk, dv, seed=13, state_std=0.1)
    out, S = run_varlen(d, H, dk, dv, 0.09, -3.0, 64, bf16)
    o = oracle_inputs(d, bf16)
    ref_out, ref_S = kda_forward_varlen(o["q"], o["k"], o["v"], o["g"], o["beta_logits"],
                                        o["a_log"], o["dt_bias"], d["cu_seqlens"], 0.09, -3.0,
                                        o["initial_state"])
    _check(out, S, ref_out, ref_S, bf16)
    np.testing.assert_array_equal(S[1], d["initial_state"][1])


def test_varlen_tensor_core_path_small():
    """dk = dv = 128, bf16, chunk 64 (the tensor-core kernel) with empty, single-token,
    exactly-one-chunk and ragged sequences; no bounded wait may have given up."""
    from gated_delta_rule_55_gb300 import kda_device_error
    kda_device_error(reset=True)
    lens = [130, 0, 1, 64, 200, 63]
    H, dk, dv = 2, 128, 128
    d = synth.varlen_inputs(lens, H, dk, dv, seed=14, state_std=0.1)
    for lb in (-5.0, -0.1):
        out, S = run_varlen(d, H, dk, dv, 0.09, lb, 64, True)
        o = oracle_inputs(d, True)
        ref_out, ref_S = kda_forward_varlen(o["q"], o["k"], o["v"], o["g"], o["beta_logits"],
                                            o["a_log"], o["dt_bias"], d["cu_seqlens"], 0.09,
                                            lb, o["initial_state"])
        _check(out, S, ref_out, ref_S, True)
        np.testing.assert_array_equal(S[1], d["initial_state"][1])
    assert kda_device_error(reset=True) == 0


def test_prefill_workload_B4_T4096_full():
    """B=4, T=4096, H=32, dk=dv=128, bf16 q/k/v, chunk 64, zero initial state, through the
    single-pass kernel: every element of all 128 (b, h) pairs against the oracle."""
    w, d, (ref_out, ref_S) = workload_reference(synth.PREFILL_B4.name)
    out, S = run_chunk(d, w.B, w.T, w.H, w.dk, w.dv, w.q_scale, w.lower_bound, w.chunk, True)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(S))
    check_full("prefill B4 T4096 H32, kda_chunk_fwd", out, ref_out, S, ref_S)


def test_varlen_workload_8seq_full():
    """8 packed sequences of 512..8192 tokens (seeded), H=16, bf16, chunk 64, seeded
    N(0, 0.02) initial states, single pass: every (sequence, head) pair, every element."""
    w, d, (ref_out, ref_S) = workload_reference(synth.VARLEN_8.name)
    out, S = run_varlen(d, w.H, w.dk, w.dv, w.q_scale, w.lower_bound, w.chunk, True)
    check_full("varlen 8 seq H16, kda_chunk_fwd_varlen", out, ref_out, S, ref_S,
               d["cu_seqlens"])
