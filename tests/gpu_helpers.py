"""Shared helpers of the GPU parity tests: move seeded host inputs to the device, call the
library through its C ABI, and compare against the fp64 oracle.

Tolerances (written into the tests): fp32 paths max |gpu - oracle| <= 1e-4; the bf16
chunked path max |gpu - oracle| / max |oracle| <= 2e-2 per tensor, the oracle being fed
the same bf16-rounded q/k/v.  Next to that max-norm figure the bf16 checks record the
elementwise relative error with a floor, max |gpu - oracle| / max(|oracle|, 1e-3 max|oracle|)
(its maximum and 99th percentile), which the test session prints at its end.
"""
import functools
import os

import numpy as np
import torch

import gated_delta_rule_55_gb300 as kda
from gated_delta_rule_55_gb300 import build_lib

F32_ATOL = 1e-4
BF16_REL = 2e-2

_built = False


def ensure_built():
    global _built
    if not _built:
        build_lib.build()
        kda.lib()
        _built = True


def to_dev(x, dtype=torch.float32):
    if x is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(x)).to(device="cuda", dtype=dtype)


def bf16_round(x):
    """The values a bf16 tensor holds, as fp64 (round-to-nearest-even)."""
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).to(torch.float64).numpy()


def max_abs(a, b):
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64)))) if np.size(a) else 0.0


def rel_err(gpu, ref):
    ref = np.asarray(ref, np.float64)
    den = float(np.max(np.abs(ref))) if ref.size else 1.0
    return max_abs(gpu, ref) / max(den, 1e-30)


def elem_rel(gpu, ref, floor=1e-3):
    """Elementwise relative error with a floor: |gpu - ref| / max(|ref|, floor * max|ref|);
    returns (maximum, 99th percentile)."""
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0, 0.0
    gpu = np.asarray(gpu, np.float64)
    top = max(float(np.max(np.abs(ref))), 1e-30)
    r = np.abs(gpu - ref) / np.maximum(np.abs(ref), floor * top)
    return float(np.max(r)), float(np.quantile(r, 0.99))


# (label, tensor, elements, max-norm relative error, elementwise max, elementwise p99)
PARITY = []


def check_rel(label, tensor, gpu, ref, bound=BF16_REL):
    """Records the max-norm and elementwise errors of one output tensor and asserts the
    max-norm bound (max |gpu - ref| / max |ref| <= bound)."""
    if label is None:  # the running test's id
        label = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0].split("::")[-1]
    e = rel_err(gpu, ref)
    emax, e99 = elem_rel(gpu, ref)
    PARITY.append((label, tensor, int(np.size(ref)), e, emax, e99))
    assert e <= bound, f"{label} {tensor}: max-norm relative error {e:.3e} > {bound}"


def param_grad_scales(dg_ref, g, dt_bias):
    """Summed magnitudes of the terms of the two parameter gradients (from the oracle's dg):
    da_log[h] = sum over tokens and channels of dg * (g + dt_bias), ddt_bias[c, h] = sum over
    tokens of dg.  Both are sums with heavy cancellation, so their error is judged against
    these magnitudes (the standard bound for a sum of terms with a relative error each)."""
    dg_ref = np.asarray(dg_ref, np.float64)
    H = dg_ref.shape[-2]
    x = np.asarray(g, np.float64) + np.asarray(dt_bias, np.float64).T.reshape(
        (1,) * (dg_ref.ndim - 2) + (H, -1))
    lead = tuple(range(dg_ref.ndim - 2))
    da = np.abs(dg_ref * x).sum(axis=lead + (dg_ref.ndim - 1,))       # [H]
    ddt = np.abs(dg_ref).sum(axis=lead).T                              # [dk, H]
    return {"da_log": da, "ddt_bias": ddt}


def sum_err(gpu, ref, scale):
    """max |gpu - ref| / max(scale): the error of a sum against its terms' magnitudes."""
    return max_abs(gpu, ref) / max(float(np.max(np.abs(scale))), 1e-30)


def bwd_err(name, gpu, ref, scales):
    """The bf16 error measure of one backward output: max-norm relative, except for the two
    parameter gradients (sum_err against param_grad_scales)."""
    if name in scales:
        return sum_err(gpu, ref, scales[name])
    return rel_err(gpu, ref)


def workspace(nbytes):
    """A device workspace of ``nbytes`` (256-byte aligned, as cudaMalloc returns), or None."""
    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device="cuda")


def run_chunk(d, B, T, H, dk, dv, scale, lb, chunk, bf16, want_state=True, alias=False,
              ws=False):
    """Call kda_chunk_fwd (or, with ``ws``, kda_chunk_fwd_ws) on host inputs ``d`` (numpy,
    [B,T,H,.] layouts)."""
    io = torch.bfloat16 if bf16 else torch.float32
    q, k, v = (to_dev(d[n], io) for n in ("q", "k", "v"))
    g, bl = to_dev(d["g"]), to_dev(d["beta_logits"])
    a_log, dt_bias = to_dev(d["a_log"]), to_dev(d["dt_bias"])
    s0 = to_dev(d.get("initial_state"))
    out = torch.full((B, T, H, dv), float("nan"), device="cuda", dtype=io)
    if alias:
        s1 = s0
    else:
        s1 = torch.full((B, H, dk, dv), float("nan"), device="cuda") if want_state else None
    if ws:
        w = workspace(kda.kda_chunk_fwd_workspace_size(B, T, H, dk, dv, chunk,
                                                       1 if bf16 else 0))
        kda.kda_chunk_fwd_ws(q, k, v, g, bl, a_log, dt_bias, scale, lb, s0, out, s1, B, T, H,
                             dk, dv, chunk, workspace=w)
    else:
        kda.kda_chunk_fwd(q, k, v, g, bl, a_log, dt_bias, scale, lb, s0, out, s1, B, T, H, dk,
                          dv, chunk)
    torch.cuda.synchronize()
    return (out.float().cpu().numpy(), None if s1 is None else s1.cpu().numpy())


def run_varlen(d, H, dk, dv, scale, lb, chunk, bf16, ws=False, keep_ws=None):
    io = torch.bfloat16 if bf16 else torch.float32
    total = d["q"].shape[0]
    N = len(d["cu_seqlens"]) - 1
    q, k, v = (to_dev(d[n], io) for n in ("q", "k", "v"))
    cu = torch.from_numpy(d["cu_seqlens"].astype(np.int32)).cuda()
    out = torch.full((total, H, dv), float("nan"), device="cuda", dtype=io)
    s1 = torch.full((N, H, dk, dv), float("nan"), device="cuda")
    args = (q, k, v, to_dev(d["g"]), to_dev(d["beta_logits"]), to_dev(d["a_log"]),
            to_dev(d["dt_bias"]), scale, lb, cu, N, total, to_dev(d.get("initial_state")), out,
            s1, H, dk, dv, chunk)
    if ws:
        w = workspace(kda.kda_chunk_fwd_varlen_workspace_size(N, total, H, dk, dv, chunk,
                                                              1 if bf16 else 0))
        kda.kda_chunk_fwd_varlen_ws(*args, workspace=w)
        if keep_ws is not None:
            keep_ws.append(w)
    else:
        kda.kda_chunk_fwd_varlen(*args)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), s1.cpu().numpy()


def oracle_inputs(d, bf16):
    """The inputs the oracle sees: bf16-rounded q/k/v when the GPU path takes bf16."""
    o = dict(d)
    if bf16:
        for n in ("q", "k", "v"):
            o[n] = bf16_round(d[n])
    return o


def bf16_round32(x):
    """The values a bf16 tensor holds, kept in fp32 (every bf16 value is exact in fp32)."""
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).to(torch.float32).numpy()


_POOL = None


def oracle_pool():
    """One pool of spawned oracle workers for the whole test session (every host core)."""
    global _POOL
    if _POOL is None:
        from oracle import pool
        _POOL = pool.Pool()
    return _POOL.ex


def close_oracle_pool():
    global _POOL
    if _POOL is not None:
        _POOL.close()
        _POOL = None


@functools.lru_cache(maxsize=None)
def workload_reference(name):
    """Inputs and the fp64 oracle's full result for a named prefill workload, computed once
    per session over every (sequence, head) pair in the oracle pool; the oracle sees the
    bf16-rounded q/k/v that the GPU receives."""
    from gated_delta_rule_55_gb300 import synth
    from oracle import pool
    w = synth.WORKLOADS[name]
    d = synth.workload_inputs(w)
    o = {n: bf16_round32(d[n]) for n in ("q", "k", "v")} if w.dtype == "bf16" else d
    ex = oracle_pool()
    if w.kind == "chunk":
        ref = pool.forward(ex, o["q"], o["k"], o["v"], d["g"], d["beta_logits"], d["a_log"],
                           d["dt_bias"], w.q_scale, w.lower_bound, d["initial_state"])
    else:
        ref = pool.forward_varlen(ex, o["q"], o["k"], o["v"], d["g"], d["beta_logits"],
                                  d["a_log"], d["dt_bias"], d["cu_seqlens"], w.q_scale,
                                  w.lower_bound, d["initial_state"])
    return w, d, ref


def check_full(label, out, ref_out, S, ref_S, cu_seqlens=None):
    """Every element of a full-size run against the oracle: the whole-tensor max-norm bound
    (recorded with the elementwise figures) for the output and the final state, and the same
    bound for every (sequence, head) pair on its own, so that a pair of small magnitude
    cannot hide behind the others.  ``out`` is [B, T, H, dv], or [total_T, H, dv] with
    ``cu_seqlens``; states are [nseq, H, dk, dv]."""
    check_rel(label, "out", out, ref_out)
    check_rel(label, "final_state", S, ref_S)
    out = np.asarray(out, np.float64)
    ref_out = np.asarray(ref_out, np.float64)
    if cu_seqlens is None:
        err = np.max(np.abs(out - ref_out), axis=(1, 3))                   # [B, H]
        top = np.max(np.abs(ref_out), axis=(1, 3))
    else:
        cu = np.asarray(cu_seqlens, np.int64)
        live = [n for n in range(len(cu) - 1) if cu[n + 1] > cu[n]]
        starts = cu[live]
        err = np.maximum.reduceat(np.max(np.abs(out - ref_out), axis=2), starts, axis=0)
        top = np.maximum.reduceat(np.max(np.abs(ref_out), axis=2), starts, axis=0)
    pair_out = err / np.maximum(top, 1e-30)
    pair_S = (np.max(np.abs(np.asarray(S, np.float64) - ref_S), axis=(2, 3)) /
              np.maximum(np.max(np.abs(ref_S), axis=(2, 3)), 1e-30))
    worst = float(max(pair_out.max(), pair_S.max()))
    PARITY.append((label + " (worst pair)", "out+state", int(pair_out.size), worst,
                   float("nan"), float("nan")))
    assert pair_out.max() <= BF16_REL, (label, float(pair_out.max()))
    assert pair_S.max() <= BF16_REL, (label, float(pair_S.max()))
