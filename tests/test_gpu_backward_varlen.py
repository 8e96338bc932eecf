"""kda_chunk_bwd_varlen (packed sequences) against the oracle backward run on each sequence
alone (its own initial state and final-state cotangent; da_log and ddt_bias summed over the
sequences), and against kda_chunk_bwd when every sequence has the same length.  bf16:
max-norm relative error <= 2e-2 per gradient tensor, the oracle fed the same bf16-rounded
q, k, v and d_out."""
import os

import numpy as np
import pytest
import torch

import gated_delta_rule_55_gb300 as kda
from gated_delta_rule_55_gb300 import synth
from gpu_helpers import (BF16_REL, bf16_round, bwd_err, ensure_built, param_grad_scales, rel_err,
                         to_dev, workspace)
from oracle import kda_backward

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _packed(lengths, H, seed):
    d = synth.varlen_inputs(lengths, H, 128, 128, seed)
    total = int(d["cu_seqlens"][-1])
    r = np.random.default_rng(700 + seed)
    d["d_out"] = r.normal(size=(total, H, 128))
    d["d_final_state"] = r.normal(size=(len(lengths), H, 128, 128))
    return d, total


def _run(d, total, N, H, scale, lb):
    io = torch.bfloat16
    q, k, v = (to_dev(d[n], io) for n in ("q", "k", "v"))
    g, bl, al, db = (to_dev(d[n]) for n in ("g", "beta_logits", "a_log", "dt_bias"))
    cu = torch.from_numpy(d["cu_seqlens"].astype(np.int32)).cuda()
    dout = to_dev(d["d_out"], io)
    out = {"dq": torch.full((total, H, 128), float("nan"), device="cuda", dtype=io),
           "dk": torch.full((total, H, 128), float("nan"), device="cuda", dtype=io),
           "dv": torch.full((total, H, 128), float("nan"), device="cuda", dtype=io),
           "dg": torch.full((total, H, 128), float("nan"), device="cuda"),
           "dbeta_logits": torch.full((total, H), float("nan"), device="cuda"),
           "da_log": torch.full((H,), float("nan"), device="cuda"),
           "ddt_bias": torch.full((128, H), float("nan"), device="cuda"),
           "dinitial_state": torch.full((N, H, 128, 128), float("nan"), device="cuda")}
    w = workspace(kda.kda_chunk_bwd_varlen_workspace_size(N, total, H, 128, 128))
    kda.kda_chunk_bwd_varlen(q, k, v, g, bl, al, db, scale, lb, cu, N, total,
                             to_dev(d["initial_state"]), dout, to_dev(d["d_final_state"]),
                             out["dq"], out["dk"], out["dv"], out["dg"], out["dbeta_logits"],
                             out["da_log"], out["ddt_bias"], out["dinitial_state"], H, 128, 128,
                             workspace=w)
    torch.cuda.synchronize()
    return {n: t.float().cpu().numpy() for n, t in out.items()}


def _oracle(d, lengths, H, scale, lb):
    cu = d["cu_seqlens"]
    per = {"dq": [], "dk": [], "dv": [], "dg": [], "dbeta_logits": [], "dinitial_state": []}
    da = np.zeros(H)
    ddt = np.zeros((128, H))
    for i, L in enumerate(lengths):
        a, b = int(cu[i]), int(cu[i + 1])
        sl = lambda x: x[a:b][None]  # noqa: E731
        r = kda_backward(bf16_round(sl(d["q"])), bf16_round(sl(d["k"])), bf16_round(sl(d["v"])),
                         sl(d["g"]), sl(d["beta_logits"]), d["a_log"], d["dt_bias"],
                         bf16_round(sl(d["d_out"])), d["d_final_state"][i:i + 1], scale, lb,
                         d["initial_state"][i:i + 1])
        for n in ("dq", "dk", "dv", "dg", "dbeta_logits"):
            per[n].append(r[n][0])
        per["dinitial_state"].append(r["dinitial_state"][0])
        da += r["da_log"]
        ddt += r["ddt_bias"]
    ref = {n: np.concatenate(v, axis=0) for n, v in per.items() if n != "dinitial_state"}
    ref["dinitial_state"] = np.stack(per["dinitial_state"])
    ref["da_log"], ref["ddt_bias"] = da, ddt
    return ref


@pytest.mark.parametrize("lengths,lb", [
    ([70, 0, 129, 64, 1], -2.0),   # ragged tails, an empty sequence, a one-token sequence
    ([300, 45], -5.0),
])
def test_varlen_backward_matches_per_sequence_oracle(lengths, lb):
    H, scale = 2, 128 ** -0.5
    d, total = _packed(lengths, H, len(lengths))
    gpu = _run(d, total, len(lengths), H, scale, lb)
    ref = _oracle(d, lengths, H, scale, lb)
    scales = param_grad_scales(ref["dg"], d["g"], d["dt_bias"])
    for n in ref:
        e = bwd_err(n, gpu[n], ref[n], scales)
        assert e <= BF16_REL, (n, e)
    assert kda.kda_device_error(1) == 0


def test_varlen_backward_tails_at_every_half_sub_chunk_boundary():
    """Sequences whose last chunk ends just before, at and just after each 8-token boundary
    (the per-chunk kernel's token work runs on half sub-chunks of 8 tokens, each 64-thread
    group taking one half of an early and one of a late sub-chunk), each sequence's dq, dk,
    dv, dg and initial-state gradient compared with the oracle run on it alone.

    dbeta_logits is judged over the packed tensor, as in the other tests: per token it is
    (1 - beta) lam . u, a 128-term dot product whose terms cancel, so the bf16 rounding of its
    operands (the last chunk's dS' is the final-state cotangent rounded to bf16) shows as a
    few per cent of the largest value in a 70-token sequence (2.8% at length 73 with this
    seed, the same before and after the pairing of half sub-chunks), against 0.4% of the
    packed tensor's largest value."""
    tails = [1, 7, 8, 9, 15, 16, 17, 23, 24, 25, 31, 32, 33, 40, 47, 48, 49, 56, 57, 63]
    lengths = [64 + t for t in tails]
    H, scale, lb = 2, 128 ** -0.5, -3.0
    d, total = _packed(lengths, H, 21)
    gpu = _run(d, total, len(lengths), H, scale, lb)
    ref = _oracle(d, lengths, H, scale, lb)
    cu = d["cu_seqlens"]
    for i, L in enumerate(lengths):
        a, b = int(cu[i]), int(cu[i + 1])
        for n in ("dq", "dk", "dv", "dg"):
            e = rel_err(gpu[n][a:b], ref[n][a:b])
            assert e <= BF16_REL, (L, n, e)
        e = rel_err(gpu["dinitial_state"][i], ref["dinitial_state"][i])
        assert e <= BF16_REL, (L, "dinitial_state", e)
    e = rel_err(gpu["dbeta_logits"], ref["dbeta_logits"])
    assert e <= BF16_REL, ("dbeta_logits", e)
    scales = param_grad_scales(ref["dg"], d["g"], d["dt_bias"])
    for n in ("da_log", "ddt_bias"):
        e = bwd_err(n, gpu[n], ref[n], scales)
        assert e <= BF16_REL, (n, e)
    assert kda.kda_device_error(1) == 0


def _random_cases(n, seed):
    rng = np.random.default_rng(seed)
    for case in range(n):
        N = int(rng.integers(1, 7))
        H = int(rng.integers(1, 4))
        lens = rng.integers(0, 400, N)
        if rng.random() < 0.5:
            lens[rng.integers(0, N)] = int(rng.integers(600, 1500))
        if case % 3 == 0:
            lens[rng.integers(0, N)] = int(rng.integers(0, 2))  # empty or one token
        if lens.sum() == 0:
            lens[0] = 41
        yield case, [int(x) for x in lens], H, float(rng.choice([-5.0, -2.0, -0.1]))


def test_random_packed_configurations():
    """Seeded random packed configurations (sequence counts, lengths with empty and
    one-token sequences and a long one, head counts, gate lower bounds) through
    kda_chunk_bwd_varlen against the per-sequence oracle backward.  The case count is
    KDA_RANDOM_CASES (default 4), so that a longer sweep runs the same code."""
    n = int(os.environ.get("KDA_RANDOM_CASES", "4"))
    scale = 128 ** -0.5
    for case, lens, H, lb in _random_cases(n, 77):
        d, total = _packed(lens, H, 3000 + case)
        gpu = _run(d, total, len(lens), H, scale, lb)
        ref = _oracle(d, lens, H, scale, lb)
        scales = param_grad_scales(ref["dg"], d["g"], d["dt_bias"])
        for name in ref:
            e = bwd_err(name, gpu[name], ref[name], scales)
            assert e <= BF16_REL, (case, lens, H, lb, name, e)
    assert kda.kda_device_error(1) == 0


def test_varlen_backward_equals_fixed_length_backward():
    """Equal lengths: the packed layout is the fixed-length layout, so the gradients agree
    with kda_chunk_bwd exactly (da_log and ddt_bias up to the order of their atomic sums)."""
    N, T, H, scale, lb = 2, 150, 2, 128 ** -0.5, -2.0
    d, total = _packed([T] * N, H, 9)
    gpu = _run(d, total, N, H, scale, lb)
    io = torch.bfloat16
    q, k, v = (to_dev(d[n].reshape(N, T, H, 128), io) for n in ("q", "k", "v"))
    g = to_dev(d["g"].reshape(N, T, H, 128))
    bl = to_dev(d["beta_logits"].reshape(N, T, H))
    al, db = to_dev(d["a_log"]), to_dev(d["dt_bias"])
    dout = to_dev(d["d_out"].reshape(N, T, H, 128), io)
    f = {"dq": torch.empty(N, T, H, 128, device="cuda", dtype=io),
         "dk": torch.empty(N, T, H, 128, device="cuda", dtype=io),
         "dv": torch.empty(N, T, H, 128, device="cuda", dtype=io),
         "dg": torch.empty(N, T, H, 128, device="cuda"),
         "dbeta_logits": torch.empty(N, T, H, device="cuda"),
         "da_log": torch.empty(H, device="cuda"), "ddt_bias": torch.empty(128, H, device="cuda"),
         "dinitial_state": torch.empty(N, H, 128, 128, device="cuda")}
    w = workspace(kda.kda_chunk_bwd_workspace_size(N, T, H, 128, 128))
    kda.kda_chunk_bwd(q, k, v, g, bl, al, db, scale, lb, to_dev(d["initial_state"]), dout,
                      to_dev(d["d_final_state"]), f["dq"], f["dk"], f["dv"], f["dg"],
                      f["dbeta_logits"], f["da_log"], f["ddt_bias"], f["dinitial_state"], N, T, H,
                      128, 128, workspace=w)
    torch.cuda.synchronize()
    for n, t in f.items():
        fixed = t.float().cpu().numpy()
        if n in ("da_log", "ddt_bias"):
            assert rel_err(gpu[n], fixed) <= 1e-5, n
        else:
            assert np.array_equal(gpu[n].reshape(fixed.shape), fixed), n


def test_varlen_training_pair():
    """kda_chunk_fwd_train_varlen matches kda_chunk_fwd_varlen_ws (last-bit bf16 differences:
    the query scale rides in the operands) and leaves records from which
    kda_chunk_bwd_saved_varlen reproduces kda_chunk_bwd_varlen exactly."""
    lengths, H, scale, lb = [200, 64, 3, 0, 77], 2, 128 ** -0.5, -3.0
    N = len(lengths)
    d, total = _packed(lengths, H, 21)
    io = torch.bfloat16
    q, k, v = (to_dev(d[n], io) for n in ("q", "k", "v"))
    g, bl, al, db = (to_dev(d[n]) for n in ("g", "beta_logits", "a_log", "dt_bias"))
    cu = torch.from_numpy(d["cu_seqlens"].astype(np.int32)).cuda()
    s0 = to_dev(d["initial_state"])
    out = torch.full((total, H, 128), float("nan"), device="cuda", dtype=io)
    s1 = torch.full((N, H, 128, 128), float("nan"), device="cuda")
    w = workspace(kda.kda_chunk_bwd_varlen_workspace_size(N, total, H, 128, 128))
    kda.kda_chunk_fwd_train_varlen(q, k, v, g, bl, al, db, scale, lb, cu, N, total, s0, out, s1,
                                   H, 128, 128, workspace=w)
    ref_out = torch.full_like(out, float("nan"))
    ref_s1 = torch.full_like(s1, float("nan"))
    w0 = workspace(kda.kda_chunk_fwd_varlen_workspace_size(N, total, H, 128, 128))
    kda.kda_chunk_fwd_varlen_ws(q, k, v, g, bl, al, db, scale, lb, cu, N, total, s0, ref_out,
                                ref_s1, H, 128, 128, workspace=w0)
    torch.cuda.synchronize()
    assert rel_err(out.float().cpu().numpy(), ref_out.float().cpu().numpy()) <= 1e-2
    assert rel_err(s1.cpu().numpy(), ref_s1.cpu().numpy()) <= 1e-5

    dout = to_dev(d["d_out"], io)
    dfin = to_dev(d["d_final_state"])

    def grads():
        return [torch.full((total, H, 128), float("nan"), device="cuda", dtype=io),
                torch.full((total, H, 128), float("nan"), device="cuda", dtype=io),
                torch.full((total, H, 128), float("nan"), device="cuda", dtype=io),
                torch.full((total, H, 128), float("nan"), device="cuda"),
                torch.full((total, H), float("nan"), device="cuda"),
                torch.full((H,), float("nan"), device="cuda"),
                torch.full((128, H), float("nan"), device="cuda"),
                torch.full((N, H, 128, 128), float("nan"), device="cuda")]
    saved, fresh = grads(), grads()
    kda.kda_chunk_bwd_saved_varlen(q, k, v, g, bl, al, db, scale, lb, cu, N, total, s0, dout,
                                   dfin, *saved, H, 128, 128, workspace=w)
    w2 = workspace(kda.kda_chunk_bwd_varlen_workspace_size(N, total, H, 128, 128))
    kda.kda_chunk_bwd_varlen(q, k, v, g, bl, al, db, scale, lb, cu, N, total, s0, dout, dfin,
                             *fresh, H, 128, 128, workspace=w2)
    torch.cuda.synchronize()
    for i, (a_, b_) in enumerate(zip(saved, fresh)):
        x, y = a_.float().cpu().numpy(), b_.float().cpu().numpy()
        if i in (5, 6):  # da_log, ddt_bias: atomic sums
            assert rel_err(x, y) <= 1e-5, i
        else:
            assert np.array_equal(x, y), i
    assert kda.kda_device_error(1) == 0


def test_varlen_backward_many_sequences():
    """Forty packed sequences of random lengths 0..150: the per-chunk kernel's binary search
    over the chunk offsets and the reverse scan's per-sequence chunk ranges."""
    H, scale, lb = 2, 128 ** -0.5, -2.0
    lengths = list(np.random.default_rng(41).integers(0, 150, size=40))
    d, total = _packed(lengths, H, 41)
    gpu = _run(d, total, len(lengths), H, scale, lb)
    ref = _oracle(d, lengths, H, scale, lb)
    scales = param_grad_scales(ref["dg"], d["g"], d["dt_bias"])
    for n in ref:
        e = bwd_err(n, gpu[n], ref[n], scales)
        assert e <= BF16_REL, (n, e)
    assert kda.kda_device_error(1) == 0


def test_varlen_backward_all_sequences_empty():
    """No tokens at all: the state cotangent passes straight through (d_initial_state =
    d_final_state) and the parameter gradients are zero.  The per-token tensors are empty,
    so small placeholder buffers stand in for their (never read) pointers."""
    N, H = 3, 2
    r = np.random.default_rng(5)
    s0 = to_dev(r.normal(size=(N, H, 128, 128)) * 0.02)
    dfin_h = r.normal(size=(N, H, 128, 128)).astype(np.float32)
    dfin = to_dev(dfin_h)
    cu = torch.zeros(N + 1, dtype=torch.int32, device="cuda")
    xb = torch.zeros(H * 128, device="cuda", dtype=torch.bfloat16)
    xf = torch.zeros(H * 128, device="cuda")
    al, db = to_dev(r.uniform(-1, 1, H)), to_dev(r.normal(size=(128, H)) * 0.1)
    da = torch.full((H,), float("nan"), device="cuda")
    ddt = torch.full((128, H), float("nan"), device="cuda")
    dinit = torch.full((N, H, 128, 128), float("nan"), device="cuda")
    w = workspace(kda.kda_chunk_bwd_varlen_workspace_size(N, 0, H, 128, 128))
    kda.kda_chunk_bwd_varlen(xb, xb, xb, xf, xf, al, db, 128 ** -0.5, -2.0, cu, N, 0, s0, xb,
                             dfin, xb, xb, xb, xf, xf, da, ddt, dinit, H, 128, 128, workspace=w)
    torch.cuda.synchronize()
    assert np.array_equal(dinit.cpu().numpy(), dfin_h)
    assert not torch.any(da).item() and not torch.any(ddt).item()
    assert kda.kda_device_error(1) == 0


def test_backward_without_sequences():
    """B = 0: nothing to differentiate; the parameter gradients are zeroed."""
    H = 2
    da = torch.full((H,), float("nan"), device="cuda")
    ddt = torch.full((128, H), float("nan"), device="cuda")
    x = torch.empty(16, device="cuda", dtype=torch.bfloat16)
    f = torch.empty(16, device="cuda")
    kda.kda_chunk_bwd(x, x, x, f, f, f, f, 0.1, -1.0, None, x, None, x, x, x, f, f, da, ddt, None,
                      0, 64, H, 128, 128, dtype=kda.KDA_BF16, workspace=None)
    torch.cuda.synchronize()
    assert not torch.any(da).item() and not torch.any(ddt).item()
