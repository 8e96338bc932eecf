"""Parity of the workspace (two-launch) chunked forward -- kda_chunk_fwd_ws and
kda_chunk_fwd_varlen_ws -- with the fp64 oracle, through the C ABI.

The two-launch path serves bf16 q/k/v with dk = dv = 128 and 64-token chunks; the bar is
that of the single-pass bf16 path: max |gpu - oracle| / max |oracle| <= 2e-2 per tensor
(out and final state), the oracle fed the same bf16-rounded q/k/v.  Other configurations
ignore the workspace and must give the single-pass results exactly.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_55_gb300 as kda
from gated_delta_rule_55_gb300 import synth
from gpu_helpers import (BF16_REL, check_full, check_rel, ensure_built, max_abs, oracle_inputs, rel_err,
                         run_chunk, run_varlen, to_dev, workload_reference, workspace)
from oracle import kda_forward, kda_forward_varlen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    kda.kda_device_error(reset=True)
    yield
    assert kda.kda_device_error(reset=True) == 0, "a bounded wait gave up"


def _check(out, S, ref_out, ref_S):
    check_rel(None, "out", out, ref_out)
    check_rel(None, "final_state", S, ref_S)


def _case(B, T, H, lb, seed, state_std=0.1, scale=None):
    d = synth.chunk_inputs(B, T, H, 128, 128, seed, state_std)
    scale = 128 ** -0.5 if scale is None else scale
    out, S = run_chunk(d, B, T, H, 128, 128, scale, lb, 64, True, ws=True)
    o = oracle_inputs(d, True)
    ref_out, ref_S = kda_forward(o["q"], o["k"], o["v"], o["g"], o["beta_logits"], o["a_log"],
                                 o["dt_bias"], scale, lb, o["initial_state"])
    _check(out, S, ref_out, ref_S)
    return out, S


@pytest.mark.parametrize("lb", [-5.0, -0.05])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 130, 300])
def test_bf16_ragged(T, lb):
    _case(B=2, T=T, H=3, lb=lb, seed=100 + T)


def test_zero_initial_state_and_scale():
    d = synth.chunk_inputs(1, 200, 2, 128, 128, 7, state_std=0.0)
    d["initial_state"] = None
    out, S = run_chunk(d, 1, 200, 2, 128, 128, 0.3, -2.0, 64, True, ws=True)
    o = oracle_inputs(d, True)
    ref_out, ref_S = kda_forward(o["q"], o["k"], o["v"], o["g"], o["beta_logits"], o["a_log"],
                                 o["dt_bias"], 0.3, -2.0, None)
    _check(out, S, ref_out, ref_S)


def test_matches_single_pass_path():
    """Both tensor-core paths compute the same algebra; their difference is rounding."""
    B, T, H = 2, 257, 4
    d = synth.chunk_inputs(B, T, H, 128, 128, 9, state_std=0.1)
    o1, S1 = run_chunk(d, B, T, H, 128, 128, 0.09, -1.0, 64, True, ws=False)
    o2, S2 = run_chunk(d, B, T, H, 128, 128, 0.09, -1.0, 64, True, ws=True)
    assert rel_err(o2, o1) <= 1e-2 and rel_err(S2, S1) <= 1e-2


def test_state_passthrough_two_calls_equal_one():
    B, T, H = 2, 200, 2
    d = synth.chunk_inputs(B, T, H, 128, 128, 11, state_std=0.2)
    full_o, full_S = run_chunk(d, B, T, H, 128, 128, 0.1, -0.5, 64, True, ws=True)
    cut = 128  # a chunk boundary: the two halves see the same chunking as one pass
    d1 = {n: (x[:, :cut] if n in ("q", "k", "v", "g", "beta_logits") else x) for n, x in d.items()}
    d2 = {n: (x[:, cut:] if n in ("q", "k", "v", "g", "beta_logits") else x) for n, x in d.items()}
    o1, S1 = run_chunk(d1, B, cut, H, 128, 128, 0.1, -0.5, 64, True, ws=True)
    d2["initial_state"] = S1
    o2, S2 = run_chunk(d2, B, T - cut, H, 128, 128, 0.1, -0.5, 64, True, ws=True)
    assert rel_err(np.concatenate([o1, o2], 1), full_o) <= 1e-2
    assert rel_err(S2, full_S) <= 1e-2


def test_empty_sequence_passes_state_through():
    d = synth.chunk_inputs(2, 1, 2, 128, 128, 1, state_std=0.3)
    s0 = to_dev(d["initial_state"])
    s1 = torch.full_like(s0, float("nan"))
    dummy = torch.zeros(16, device="cuda", dtype=torch.bfloat16)
    f = torch.zeros(16, device="cuda")
    kda.kda_chunk_fwd_ws(dummy, dummy, dummy, f, f, to_dev(d["a_log"]), to_dev(d["dt_bias"]),
                         0.2, -1.0, s0, dummy, s1, 2, 0, 2, 128, 128, 64, workspace=None)
    torch.cuda.synchronize()
    assert torch.equal(s1, s0)


def test_other_configurations_ignore_the_workspace():
    """fp32 inputs (the SIMT kernel) through the workspace entry give the plain entry's
    results bit for bit."""
    B, T, H = 1, 100, 2
    d = synth.chunk_inputs(B, T, H, 128, 128, 3, state_std=0.1)
    o1, S1 = run_chunk(d, B, T, H, 128, 128, 0.1, -1.0, 64, False, ws=False)
    o2, S2 = run_chunk(d, B, T, H, 128, 128, 0.1, -1.0, 64, False, ws=True)
    assert np.array_equal(o1, o2) and np.array_equal(S1, S2)


def test_varlen_small_with_empty_and_ragged_sequences():
    lens = [130, 0, 1, 64, 200, 63, 0]
    H = 2
    d = synth.varlen_inputs(lens, H, 128, 128, seed=14, state_std=0.1)
    for lb in (-5.0, -0.1):
        out, S = run_varlen(d, H, 128, 128, 0.09, lb, 64, True, ws=True)
        o = oracle_inputs(d, True)
        ref_out, ref_S = kda_forward_varlen(o["q"], o["k"], o["v"], o["g"], o["beta_logits"],
                                            o["a_log"], o["dt_bias"], d["cu_seqlens"], 0.09,
                                            lb, o["initial_state"])
        _check(out, S, ref_out, ref_S)
        np.testing.assert_array_equal(S[1], d["initial_state"][1])
        np.testing.assert_array_equal(S[6], d["initial_state"][6])


def test_varlen_tails_at_every_sub_chunk_boundary():
    """Packed sequences whose last chunk ends just before, at and just after each 16-token
    sub-chunk boundary and each 8-token half (the prep's gate totals stop at the last live
    token of a sub-chunk; the rows past it are zeroed), each sequence's output and final
    state compared with the oracle on its own."""
    tails = [1, 7, 8, 9, 15, 16, 17, 24, 31, 32, 33, 40, 47, 48, 49, 56, 63]
    lens = [64 + t for t in tails] + [t for t in tails]
    H = 2
    d = synth.varlen_inputs(lens, H, 128, 128, seed=23, state_std=0.1)
    for lb in (-5.0, -0.5):
        out, S = run_varlen(d, H, 128, 128, 0.09, lb, 64, True, ws=True)
        o = oracle_inputs(d, True)
        ref_out, ref_S = kda_forward_varlen(o["q"], o["k"], o["v"], o["g"], o["beta_logits"],
                                            o["a_log"], o["dt_bias"], d["cu_seqlens"], 0.09,
                                            lb, o["initial_state"])
        cu = d["cu_seqlens"]
        for i, L in enumerate(lens):
            a, b = int(cu[i]), int(cu[i + 1])
            check_rel(f"varlen_tail[len={L} lb={lb}]", "out", out[a:b], ref_out[a:b])
            check_rel(f"varlen_tail[len={L} lb={lb}]", "final_state", S[i], ref_S[i])


def test_varlen_many_short_sequences():
    """More sequences than one pass of the chunk-offset scan (1024), mostly shorter than a
    chunk, a few spanning several chunks."""
    rng = np.random.default_rng(21)
    lens = rng.integers(0, 6, 1300)
    lens[[5, 700, 1299]] = [64, 130, 257]
    H = 1
    d = synth.varlen_inputs([int(x) for x in lens], H, 128, 128, seed=22, state_std=0.05)
    out, S = run_varlen(d, H, 128, 128, 0.09, -2.0, 64, True, ws=True)
    o = oracle_inputs(d, True)
    ref_out, ref_S = kda_forward_varlen(o["q"], o["k"], o["v"], o["g"], o["beta_logits"],
                                        o["a_log"], o["dt_bias"], d["cu_seqlens"], 0.09, -2.0,
                                        o["initial_state"])
    _check(out, S, ref_out, ref_S)


def test_multi_record_ctas_odd_head_count():
    """More (chunk, head) records (16 x 23 = 368) than the prep's persistent CTAs (two per
    SM), so CTAs walk several records (head and chunk indices stepped by the grid size, with
    a carry: the grid size is not a multiple of 23) and stage the next record's tiles while
    they finish the current one; the last chunk is partial (1000 = 15 x 64 + 40)."""
    _case(B=1, T=1000, H=23, lb=-3.0, seed=31)


def test_varlen_multi_record_ctas_odd_head_count():
    """Packed sequences with more records than persistent CTAs (an odd head count, empty,
    single-chunk and partial sequences among them), every output compared."""
    lens = [1000, 37, 0, 513, 64, 700]
    H = 11
    d = synth.varlen_inputs(lens, H, 128, 128, seed=32, state_std=0.1)
    out, S = run_varlen(d, H, 128, 128, 0.09, -1.5, 64, True, ws=True)
    o = oracle_inputs(d, True)
    ref_out, ref_S = kda_forward_varlen(o["q"], o["k"], o["v"], o["g"], o["beta_logits"],
                                        o["a_log"], o["dt_bias"], d["cu_seqlens"], 0.09, -1.5,
                                        o["initial_state"])
    _check(out, S, ref_out, ref_S)
    np.testing.assert_array_equal(S[2], d["initial_state"][2])


def test_prefill_workload_B4_T4096_full():
    """B=4, T=4096, H=32, bf16, chunk 64, zero initial state, through the workspace (the
    benchmarked call): every output element and final-state entry of all 128 (b, h) pairs
    against the oracle, which runs over the pairs in a pool of host processes."""
    w, d, (ref_out, ref_S) = workload_reference(synth.PREFILL_B4.name)
    out, S = run_chunk(d, w.B, w.T, w.H, w.dk, w.dv, w.q_scale, w.lower_bound, w.chunk, True,
                       ws=True)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(S))
    check_full("prefill B4 T4096 H32, kda_chunk_fwd_ws", out, ref_out, S, ref_S)


def test_varlen_workload_8seq_full():
    """The 8-sequence packed workload (27,268 tokens, H=16, seeded N(0, 0.02) initial
    states) through the workspace: every (sequence, head) pair, every element."""
    w, d, (ref_out, ref_S) = workload_reference(synth.VARLEN_8.name)
    out, S = run_varlen(d, w.H, w.dk, w.dv, w.q_scale, w.lower_bound, w.chunk, True, ws=True)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(S))
    check_full("varlen 8 seq H16, kda_chunk_fwd_varlen_ws", out, ref_out, S, ref_S,
               d["cu_seqlens"])


# One (chunk, head) record of the forward workspace: four bf16 [64 x 128] tiles, one bf16
# [64 x 64] tile and 256 fp32 values.
_REC = 4 * 64 * 128 * 2 + 64 * 64 * 2 + 256 * 4


def _split_counts(w, N, total, H):
    """(chains, split sequences) of the scan plan, read from the packed forward's workspace:
    after the records come the (N + 1) chunk offsets and the chain table (N + 16 int4),
    each 256-byte aligned, then the two counts."""
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    off = (total // 64 + N) * H * _REC + al((N + 1) * 4) + al((N + 16) * 16)
    c = w.view(torch.uint8)[off:off + 8].cpu().numpy().view(np.int32)
    return int(c[0]), int(c[1])


def _varlen_split_case(lens, H, seed, lb, splits, initial=True):
    d = synth.varlen_inputs(lens, H, 128, 128, seed=seed, state_std=0.1)
    if not initial:
        d["initial_state"] = None
    kept = []
    out, S = run_varlen(d, H, 128, 128, 0.09, lb, 64, True, ws=True, keep_ws=kept)
    N, total = len(lens), int(sum(lens))
    assert _split_counts(kept[0], N, total, H) == (N + 2 * splits, splits)
    o = oracle_inputs(d, True)
    ref_out, ref_S = kda_forward_varlen(o["q"], o["k"], o["v"], o["g"], o["beta_logits"],
                                        o["a_log"], o["dt_bias"], d["cu_seqlens"], 0.09, lb,
                                        o["initial_state"])
    _check(out, S, ref_out, ref_S)
    # the same call again gives the same bits (the plan and the correction are deterministic)
    out2, S2 = run_varlen(d, H, 128, 128, 0.09, lb, 64, True, ws=True)
    assert np.array_equal(out, out2) and np.array_equal(S, S2)
    return d, S


def test_varlen_split_one_long_sequence():
    """One sequence much longer than the rest (65 chunks against at most 8): its scan is cut
    at chunk 33 into three chains (the first part from the initial state, the second from
    zero and from the identity) and corrected afterwards; an empty and a one-token sequence
    ride along."""
    d, S = _varlen_split_case([4133, 300, 500, 65, 1, 0], H=4, seed=41, lb=-2.0, splits=1)
    np.testing.assert_array_equal(S[5], d["initial_state"][5])


@pytest.mark.parametrize("lb,initial", [(-5.0, True), (-0.1, False)])
def test_varlen_split_two_sequences_ragged_ends(lb, initial):
    """Two long sequences (41 and 34 chunks, both ending in a partial chunk) split at chunks
    21 and 17, strong and weak decay, with and without initial states."""
    _varlen_split_case([64 * 40 + 17, 64 * 33 + 5, 200, 0], H=3, seed=42, lb=lb, splits=2,
                       initial=initial)


def test_varlen_equal_lengths_split_together():
    """Equal lengths: only cutting every chain shortens the longest, so all three are split
    (20 chunks into 10 + 10, the cut on a chunk boundary at token 640)."""
    _varlen_split_case([64 * 20] * 3, H=2, seed=43, lb=-1.0, splits=3)


def test_varlen_short_chains_are_not_split():
    """Chains under 16 chunks stay whole, however uneven the lengths."""
    _varlen_split_case([64 * 14 + 3, 64, 10], H=2, seed=44, lb=-1.0, splits=0)


def test_varlen_many_sequences_past_the_plan_sort():
    """5,000 packed sequences (mostly under one chunk, two long ones): more chains than the
    plan sorts on chip (4,096) or keeps the chunk counts of (2,048), and more than two per
    SM, so nothing is split and the chain table keeps sequence order."""
    rng = np.random.default_rng(45)
    lens = [int(x) for x in rng.integers(0, 6, 5000)]
    lens[10], lens[3000] = 64 * 40, 64 * 18 + 5
    _varlen_split_case(lens, H=1, seed=46, lb=-2.0, splits=0)


def test_varlen_at_the_sequence_limit():
    """65,535 packed sequences (the most the entry accepts; all but five empty), no initial or
    final states: the scan's grid stops at the 65,535 CTAs of its y extent, and the outputs
    of the five non-empty sequences match the oracle."""
    N, H = 65535, 1
    lens = np.zeros(N, dtype=np.int64)
    picks = [0, 1000, 30000, 65000, N - 1]
    lens[picks] = [130, 64, 1, 200, 77]
    d = synth.varlen_inputs([int(x) for x in lens], H, 128, 128, seed=47, state_std=None)
    total = int(lens.sum())
    q, k, v = (to_dev(d[n], torch.bfloat16) for n in ("q", "k", "v"))
    cu = torch.from_numpy(d["cu_seqlens"].astype(np.int32)).cuda()
    out = torch.full((total, H, 128), float("nan"), device="cuda", dtype=torch.bfloat16)
    w = workspace(kda.kda_chunk_fwd_varlen_workspace_size(N, total, H, 128, 128, 64, 1))
    kda.kda_chunk_fwd_varlen_ws(q, k, v, to_dev(d["g"]), to_dev(d["beta_logits"]),
                                to_dev(d["a_log"]), to_dev(d["dt_bias"]), 0.09, -2.0, cu, N,
                                total, None, out, None, H, 128, 128, 64, workspace=w)
    torch.cuda.synchronize()
    out = out.float().cpu().numpy()
    o = oracle_inputs(d, True)
    cu_h = d["cu_seqlens"]
    for n in picks:
        a, b = int(cu_h[n]), int(cu_h[n + 1])
        ref, _ = kda_forward(o["q"][None, a:b], o["k"][None, a:b], o["v"][None, a:b],
                             o["g"][None, a:b], o["beta_logits"][None, a:b], o["a_log"],
                             o["dt_bias"], 0.09, -2.0, None)
        check_rel(None, f"out seq {n}", out[a:b], ref[0])
