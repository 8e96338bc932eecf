"""kda_chunk_fwd_noalloc: the workspace chunked forward with the library's own device
scratch array as its workspace, for callers that cannot allocate device memory.

Host checks (no GPU): the entry is exported; the binding's copy of the array size equals
the header's; a configuration at the array's limit passes the capacity check (it stops at
the device check on a machine without a GPU) while the next larger one is rejected; argument
errors come before the capacity check.  GPU checks: two calls in a row give bit-identical
results, equal to kda_chunk_fwd_ws with a caller workspace, and match the fp64 oracle; a
configuration that fills the array to within half a megabyte of its end matches
kda_chunk_fwd_ws bit for bit.

This file is collected last, so that a run stopping at the first failure has run every
other test before it.
"""
import os
import re

import numpy as np
import pytest
import torch

import gated_delta_rule_55_gb300 as kda
from gated_delta_rule_55_gb300 import build_lib, synth

FAKE = 0x10000
RECORD = 74752  # workspace bytes per (64-token chunk, head) record


@pytest.fixture(scope="module")
def L():
    build_lib.build()
    return kda.lib()


def _raw(L, B, T, H, dtype=1, chunk=64, dk=128, lb=-1.0):
    return L.kda_chunk_fwd_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0.0, lb, None,
                                   FAKE, None, B, T, H, dk, 128, chunk, dtype, None)


def test_capacity_constant_matches_header():
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "include", "kda.h")).read()
    m = re.search(r"#define KDA_NOALLOC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", hdr)
    assert m, "KDA_NOALLOC_SCRATCH_BYTES not found in include/kda.h"
    assert kda.kda.NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


def test_capacity_and_rejection(L):
    cap = kda.kda.NOALLOC_SCRATCH_BYTES
    fit = cap // RECORD  # records that fit
    assert kda.kda_chunk_fwd_workspace_size(1, 64 * fit, 1, 128, 128, 64, 1) == fit * RECORD
    assert kda.kda_chunk_fwd_workspace_size(1, 64 * fit + 1, 1, 128, 128, 64, 1) > cap
    assert _raw(L, 1, 64 * fit + 1, 1) == -12   # one record past the array
    assert _raw(L, 4, 4096, 32) == -12          # the 612 MB prefill workspace
    # argument errors are reported before the capacity check, as kda_chunk_fwd reports them
    assert _raw(L, 4, 4096, 32, dtype=7) == -7
    assert _raw(L, 4, 4096, 32, lb=-6.0) == -5
    assert _raw(L, 1, 64, 2, dtype=7) == -7


def test_without_device(L):
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this case is only meaningful without one")
    fit = kda.kda.NOALLOC_SCRATCH_BYTES // RECORD
    assert _raw(L, 1, 64 * fit, 1) == -9       # at the limit: passes the capacity check
    assert _raw(L, 1, 64, 2) == -9             # scratch lookup needs a device
    assert _raw(L, 1, 64, 2, dtype=0) == -9    # fp32: no workspace, stops at the device check


def _run(entry, d, B, T, H, scale, lb, **kw):
    from gpu_helpers import to_dev
    q, k, v = (to_dev(d[n], torch.bfloat16) for n in ("q", "k", "v"))
    rest = [to_dev(d[n]) for n in ("g", "beta_logits", "a_log", "dt_bias")]
    s0 = to_dev(d["initial_state"])
    out = torch.full((B, T, H, 128), float("nan"), device="cuda", dtype=torch.bfloat16)
    s1 = torch.full((B, H, 128, 128), float("nan"), device="cuda")
    entry(q, k, v, *rest, scale, lb, s0, out, s1, B, T, H, 128, 128, 64, **kw)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), s1.cpu().numpy()


@pytest.mark.gpu
def test_two_calls_equal_workspace_entry_and_oracle(L):
    from gpu_helpers import BF16_REL, oracle_inputs, rel_err, workspace
    from oracle import kda_forward
    B, T, H = 2, 300, 4
    d = synth.chunk_inputs(B, T, H, 128, 128, 31, state_std=0.1)
    kda.kda_device_error(reset=True)
    o1, S1 = _run(kda.kda_chunk_fwd_noalloc, d, B, T, H, 0.09, -2.0)
    o2, S2 = _run(kda.kda_chunk_fwd_noalloc, d, B, T, H, 0.09, -2.0)
    w = workspace(kda.kda_chunk_fwd_workspace_size(B, T, H, 128, 128, 64, 1))
    o3, S3 = _run(kda.kda_chunk_fwd_ws, d, B, T, H, 0.09, -2.0, workspace=w)
    assert kda.kda_device_error(reset=True) == 0
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(S1, S2)
    np.testing.assert_array_equal(o1, o3)
    np.testing.assert_array_equal(S1, S3)
    o = oracle_inputs(d, True)
    ref_o, ref_S = kda_forward(o["q"], o["k"], o["v"], o["g"], o["beta_logits"], o["a_log"],
                               o["dt_bias"], 0.09, -2.0, o["initial_state"])
    assert rel_err(o1, ref_o) <= BF16_REL and rel_err(S1, ref_S) <= BF16_REL


@pytest.mark.gpu
def test_configuration_near_the_array_end(L):
    """B=1, T=7168, H=32: 3,584 records, within 0.6 MB of the array's end; twice, equal to
    kda_chunk_fwd_ws bit for bit."""
    from gpu_helpers import workspace
    B, T, H = 1, 7168, 32
    need = kda.kda_chunk_fwd_workspace_size(B, T, H, 128, 128, 64, 1)
    assert 0 < kda.kda.NOALLOC_SCRATCH_BYTES - need < 600_000
    d = synth.chunk_inputs(B, T, H, 128, 128, 33, state_std=0.05)
    kda.kda_device_error(reset=True)
    o1, S1 = _run(kda.kda_chunk_fwd_noalloc, d, B, T, H, 0.09, -0.5)
    o2, S2 = _run(kda.kda_chunk_fwd_noalloc, d, B, T, H, 0.09, -0.5)
    o3, S3 = _run(kda.kda_chunk_fwd_ws, d, B, T, H, 0.09, -0.5, workspace=workspace(need))
    assert kda.kda_device_error(reset=True) == 0
    assert np.all(np.isfinite(o1)) and np.all(np.isfinite(S1))
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(S1, S2)
    np.testing.assert_array_equal(o1, o3)
    np.testing.assert_array_equal(S1, S3)
