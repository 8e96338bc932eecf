"""kda_chunk_fwd_noalloc: the workspace chunked forward with the library's own device
scratch array as its workspace.

Host checks (no GPU): the entry is exported, a configuration whose workspace exceeds the
array is rejected before any device work, and a valid call stops at the device check on a
machine without a GPU.  GPU checks: two calls in a row give bit-identical results, equal to
kda_chunk_fwd_ws with a caller workspace, and match the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_55_gb300 as kda
from gated_delta_rule_55_gb300 import build_lib, synth

FAKE = 0x10000


@pytest.fixture(scope="module")
def L():
    build_lib.build()
    return kda.lib()


def _raw(L, B, T, H, dtype=1, chunk=64):
    return L.kda_chunk_fwd_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0.0, -1.0, None,
                                   FAKE, None, B, T, H, 128, 128, chunk, dtype, None)


def test_capacity_and_rejection(L):
    cap = kda.kda.NOALLOC_SCRATCH_BYTES
    assert kda.kda_chunk_fwd_workspace_size(1, 4096, 32, 128, 128, 64, 1) <= cap
    assert kda.kda_chunk_fwd_workspace_size(4, 4096, 32, 128, 128, 64, 1) > cap
    assert _raw(L, 4, 4096, 32) == -12         # workspace would exceed the array
    assert _raw(L, 1, 64, 2, dtype=7) == -7    # argument errors as for kda_chunk_fwd


def test_without_device(L):
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this case is only meaningful without one")
    assert _raw(L, 1, 64, 2) == -9             # scratch lookup needs a device
    assert _raw(L, 1, 64, 2, dtype=0) == -9    # fp32: no workspace, stops at the device check


@pytest.mark.gpu
def test_two_calls_equal_workspace_entry_and_oracle(L):
    from gpu_helpers import BF16_REL, oracle_inputs, rel_err, to_dev, workspace
    from oracle import kda_forward
    B, T, H = 2, 300, 4
    d = synth.chunk_inputs(B, T, H, 128, 128, 31, state_std=0.1)
    q, k, v = (to_dev(d[n], torch.bfloat16) for n in ("q", "k", "v"))
    rest = [to_dev(d[n]) for n in ("g", "beta_logits", "a_log", "dt_bias")]
    s0 = to_dev(d["initial_state"])

    def run(entry, **kw):
        out = torch.full((B, T, H, 128), float("nan"), device="cuda", dtype=torch.bfloat16)
        s1 = torch.full((B, H, 128, 128), float("nan"), device="cuda")
        entry(q, k, v, *rest, 0.09, -2.0, s0, out, s1, B, T, H, 128, 128, 64, **kw)
        torch.cuda.synchronize()
        return out.float().cpu().numpy(), s1.cpu().numpy()

    kda.kda_device_error(reset=True)
    o1, S1 = run(kda.kda_chunk_fwd_noalloc)
    o2, S2 = run(kda.kda_chunk_fwd_noalloc)
    w = workspace(kda.kda_chunk_fwd_workspace_size(B, T, H, 128, 128, 64, 1))
    o3, S3 = run(kda.kda_chunk_fwd_ws, workspace=w)
    assert kda.kda_device_error(reset=True) == 0
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(S1, S2)
    np.testing.assert_array_equal(o1, o3)
    np.testing.assert_array_equal(S1, S3)
    o = oracle_inputs(d, True)
    ref_o, ref_S = kda_forward(o["q"], o["k"], o["v"], o["g"], o["beta_logits"], o["a_log"],
                               o["dt_bias"], 0.09, -2.0, o["initial_state"])
    assert rel_err(o1, ref_o) <= BF16_REL and rel_err(S1, ref_S) <= BF16_REL
