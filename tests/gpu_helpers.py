"""Shared helpers of the GPU parity tests: move seeded host inputs to the device, call the
library through its C ABI, and compare against the fp64 oracle.

Tolerances (written into the tests): fp32 paths max |gpu - oracle| <= 1e-4; the bf16
chunked path max |gpu - oracle| / max |oracle| <= 2e-2 per tensor, the oracle being fed
the same bf16-rounded q/k/v.
"""
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


def run_varlen(d, H, dk, dv, scale, lb, chunk, bf16, ws=False):
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
