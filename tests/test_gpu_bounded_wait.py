"""The give-up path of the kernels' bounded waits: kda_selftest_bounded_wait makes one wait on
an mbarrier that nothing arrives on run out after 2 ms; the wait must end by itself, record
bit 3 of kda_device_error, and leave the device usable (a forward afterwards matches the
oracle and records no error)."""
import time

import numpy as np
import pytest
import torch

import gated_delta_rule_55_gb300 as kda
from gated_delta_rule_55_gb300 import synth
from gpu_helpers import BF16_REL, bf16_round, ensure_built, rel_err, run_chunk
from oracle import kda_forward

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def test_wait_runs_out_and_reports():
    kda.kda_device_error(reset=True)
    t0 = time.perf_counter()
    kda.kda_selftest_bounded_wait(2_000_000)
    torch.cuda.synchronize()
    took = time.perf_counter() - t0
    assert took < 5.0, took
    err = kda.kda_device_error(reset=True)
    assert err & 8, err
    assert err & 7 == 0, err
    assert kda.kda_device_error(reset=True) == 0  # the reset cleared it

    # the context is still usable
    B, T, H = 1, 130, 2
    d = synth.chunk_inputs(B, T, H, 128, 128, 5, 0.02)
    out, S = run_chunk(d, B, T, H, 128, 128, 128 ** -0.5, -2.0, 64, True, ws=True)
    o = dict(d)
    for n in ("q", "k", "v"):
        o[n] = bf16_round(d[n])
    ref_out, ref_S = kda_forward(o["q"], o["k"], o["v"], o["g"], o["beta_logits"], o["a_log"],
                                 o["dt_bias"], 128 ** -0.5, -2.0, o["initial_state"])
    assert rel_err(out, ref_out) <= BF16_REL
    assert rel_err(S, ref_S) <= BF16_REL
    assert kda.kda_device_error(reset=True) == 0
