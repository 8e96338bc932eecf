"""Seeded random packed configurations through kda_chunk_fwd_varlen_ws against the fp64
oracle: sequence counts, lengths (empty, one token, ragged, and up to two sequences long
enough for the plan to split their chains), head counts, gate lower bounds and initial
states drawn at random.  Each case holds the bf16 bar (max-norm relative error <= 2e-2 for
the packed output and the final states); across the cases the plan must have split chains
at least once, so the split path is part of what is drawn.  The case count is
KDA_RANDOM_CASES (default 12), so that a longer sweep runs the same code.
"""
import os

import numpy as np
import pytest
import torch

import gated_delta_rule_55_gb300 as kda
from gated_delta_rule_55_gb300 import synth
from gpu_helpers import check_rel, ensure_built, oracle_inputs, oracle_pool, run_varlen
from oracle import pool as opool

pytestmark = pytest.mark.gpu

RECORD = 74752  # workspace bytes per (64-token chunk, head) record


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    kda.kda_device_error(reset=True)
    yield
    assert kda.kda_device_error(reset=True) == 0, "a bounded wait gave up"


def _split_count(ws, N, total, H):
    # the plan's counts follow the records, the chunk offsets and the chain table
    al = lambda x: (x + 255) // 256 * 256
    off = (total // 64 + N) * H * RECORD + al((N + 1) * 4) + al((N + 16) * 16)
    return int(ws.view(torch.uint8)[off:off + 8].cpu().numpy().view(np.int32)[1])


def _cases(n, seed):
    rng = np.random.default_rng(seed)
    for case in range(n):
        N = int(rng.integers(1, 10))
        H = int(rng.integers(1, 4))
        lens = rng.integers(0, 500, N)
        for j in rng.choice(N, size=min(int(rng.integers(0, 3)), N), replace=False):
            lens[j] = int(rng.integers(1024, 3000))
        if case % 4 == 0:
            lens[rng.integers(0, N)] = int(rng.integers(0, 2))  # empty or one token
        if lens.sum() == 0:
            lens[0] = 37
        yield (case, [int(x) for x in lens], H, float(rng.choice([-5.0, -2.0, -0.1])),
               bool(rng.integers(0, 2)))


def test_random_packed_configurations():
    ex = oracle_pool()
    splits = 0
    for case, lens, H, lb, init in _cases(int(os.environ.get("KDA_RANDOM_CASES", "12")), 2024):
        d = synth.varlen_inputs(lens, H, 128, 128, seed=5000 + case,
                                state_std=0.1 if init else None)
        kept = []
        out, S = run_varlen(d, H, 128, 128, 0.09, lb, 64, True, ws=True, keep_ws=kept)
        splits += _split_count(kept[0], len(lens), sum(lens), H)
        o = oracle_inputs(d, True)
        ref_out, ref_S = opool.forward_varlen(ex, o["q"], o["k"], o["v"], o["g"],
                                              o["beta_logits"], o["a_log"], o["dt_bias"],
                                              d["cu_seqlens"], 0.09, lb, o["initial_state"])
        label = f"random_varlen[{case}: N={len(lens)} H={H} max_len={max(lens)} lb={lb}]"
        check_rel(label, "out", out, ref_out)
        check_rel(label, "final_state", S, ref_S)
    assert splits > 0, "no drawn case split a chain"
