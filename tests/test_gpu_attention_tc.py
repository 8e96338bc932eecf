"""Parity of kda_attention_fwd_ws -- the kernel_delta_attention call on the two-launch
tensor-core path (bf16, dk = dv = 128, 64-token chunks) -- with the fp64 oracle
``kda_attention``: every combination of use_qk_l2norm and order, per-head decays of the
page's example (N(0, 1) * -0.01, either sign), moderate and steep negative decays and no
decay, ragged lengths, with and without an initial state.  Bar: max |gpu - oracle| /
max |oracle| <= 2e-2 per tensor, the oracle fed the same bf16-rounded q, k, v.  Keys and
queries of the runs without L2 normalisation have norm about 1 (see test_gpu_attention)."""
import numpy as np
import pytest
import torch

import gated_delta_rule_55_gb300 as kda
from gpu_helpers import bf16_round, check_rel, ensure_built, to_dev, workspace
from oracle import kda_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    kda.kda_device_error(reset=True)
    yield
    assert kda.kda_device_error(reset=True) == 0, "a bounded wait gave up"


def _inputs(B, T, H, seed, norm, decay, state):
    r = np.random.default_rng(700 + seed)
    s = 1.0 if norm else 128 ** -0.5
    d = {"q": r.normal(size=(B, T, H, 128)) * s, "k": r.normal(size=(B, T, H, 128)) * s,
         "v": r.normal(size=(B, T, H, 128)), "beta": r.uniform(0.0, 1.0, size=(B, T, H))}
    d["decay"] = {None: None,
                  "page": lambda: r.normal(size=(B, T, H)) * -0.01,
                  "neg": lambda: -r.uniform(0.0, 1.5, size=(B, T, H)),
                  "steep": lambda: -r.uniform(0.0, 5.0, size=(B, T, H))}[decay]
    if decay is not None:
        d["decay"] = d["decay"]()
    d["s0"] = r.normal(size=(B, H, 128, 128)) * 0.1 if state else None
    return d


def _run(d, B, T, H, scale, norm, order):
    q, k, v = (to_dev(d[n], torch.bfloat16) for n in ("q", "k", "v"))
    out = torch.full((B, T, H, 128), float("nan"), device="cuda", dtype=torch.bfloat16)
    s1 = torch.full((B, H, 128, 128), float("nan"), device="cuda")
    nb = kda.kda_attention_fwd_workspace_size(B, T, H, 128, 128, 64, use_qk_l2norm=norm,
                                              order=order)
    assert nb > 0 or T == 0
    kda.kda_attention_fwd_ws(q, k, v, to_dev(d["beta"]), to_dev(d["decay"]), to_dev(d["s0"]),
                             out, s1, B, T, H, 128, 128, softmax_scale=scale, chunk=64,
                             use_qk_l2norm=norm, order=order, workspace=workspace(nb))
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), s1.cpu().numpy()


def _check(d, out, S, scale, norm, order):
    o = dict(d)
    for n in ("q", "k", "v"):
        o[n] = bf16_round(d[n])
    ref_o, ref_S = kda_attention(o["q"], o["k"], o["v"], o["beta"], o["decay"], o["s0"], scale,
                                 norm, order)
    check_rel(None, "out", out, ref_o)
    check_rel(None, "final_state", S, ref_S)


@pytest.mark.parametrize("decay", [None, "page", "neg", "steep"])
@pytest.mark.parametrize("order", ["decay_first", "literal"])
@pytest.mark.parametrize("norm", [True, False])
def test_variants(norm, order, decay):
    B, T, H = 2, 200, 3
    d = _inputs(B, T, H, 1, norm, decay, True)
    out, S = _run(d, B, T, H, 0.3, norm, order)
    _check(d, out, S, 0.3, norm, order)


@pytest.mark.parametrize("T", [1, 63, 64, 65, 130,
                               79, 80, 81, 95, 96, 97, 111, 112, 113])  # 16-token boundaries
@pytest.mark.parametrize("order", ["decay_first", "literal"])
def test_ragged_lengths(T, order):
    B, H = 2, 2
    d = _inputs(B, T, H, T, True, "neg", T % 2 == 1)
    out, S = _run(d, B, T, H, None, True, order)
    _check(d, out, S, None, True, order)


def test_many_records_odd_head_count():
    """More records (B 2 x 16 chunks x 23 heads) than the prep's persistent CTAs."""
    B, T, H = 2, 1000, 23
    d = _inputs(B, T, H, 9, True, "page", True)
    out, S = _run(d, B, T, H, 0.1, True, "decay_first")
    _check(d, out, S, 0.1, True, "decay_first")


def test_other_configurations_ignore_the_workspace():
    """fp32 inputs through the workspace entry run kda_attention_fwd's kernels: same bits."""
    B, T, H, dk, dv = 1, 90, 2, 128, 128
    d = _inputs(B, T, H, 4, True, "neg", True)
    outs = []
    for entry in ("plain", "ws"):
        q, k, v = (to_dev(d[n]) for n in ("q", "k", "v"))
        out = torch.full((B, T, H, dv), float("nan"), device="cuda")
        s1 = torch.full((B, H, dk, dv), float("nan"), device="cuda")
        args = (q, k, v, to_dev(d["beta"]), to_dev(d["decay"]), to_dev(d["s0"]), out, s1, B, T,
                H, dk, dv)
        if entry == "plain":
            kda.kda_attention_fwd(*args, softmax_scale=0.2)
        else:
            assert kda.kda_attention_fwd_workspace_size(B, T, H, dk, dv, dtype=kda.KDA_F32) == 0
            kda.kda_attention_fwd_ws(*args, softmax_scale=0.2, workspace=None)
        torch.cuda.synchronize()
        outs.append((out.cpu().numpy(), s1.cpu().numpy()))
    np.testing.assert_array_equal(outs[0][0], outs[1][0])
    np.testing.assert_array_equal(outs[0][1], outs[1][1])


def test_decay_outside_the_range_is_reported():
    """A per-head decay outside the tensor-core path's range [-5, 1]: the call completes and
    records bit 5 of kda_device_error (a 16-token sub-chunk's summed decay leaves [-80, 16]);
    at the range's edge nothing is recorded."""
    B, T, H = 1, 100, 2
    kda.kda_device_error(reset=True)
    d = _inputs(B, T, H, 41, True, "neg", False)
    d["decay"] = np.full((B, T, H), -5.0)  # the edge: inside
    _run(d, B, T, H, None, True, "decay_first")
    assert kda.kda_device_error(reset=True) == 0
    d["decay"] = np.full((B, T, H), -6.0)
    _run(d, B, T, H, None, True, "decay_first")
    assert kda.kda_device_error(reset=True) == 32
