"""Seeded synthetic inputs for the KDA forward pass.

This module only draws random numbers with the shapes, layouts and distributions of the
workloads; it holds none of the method's arithmetic, so both the CUDA path (tests,
benchmark) and the CPU oracle can be fed from it.  Every array is fp32 on the host; the
caller rounds q/k/v to bf16 where a workload asks for it and hands the SAME rounded values
to both sides.

Distributions (standard deviations, not variances): q, k, v, g, beta logits ~ N(0, 1);
a_log ~ U(-1, 1) per head; dt_bias ~ N(0, 0.1) per (channel, head); states ~ N(0, 0.02).
Generators are ``numpy.random.default_rng`` seeded with a small integer list, so any
(workload, step) pair can be regenerated independently.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class Workload:
    """One named workload; sizes and the knobs of its input recipe."""
    name: str
    kind: str  # "chunk", "varlen" or "decode"
    H: int
    dk: int
    dv: int
    B: int = 1
    T: int = 0
    dtype: str = "f32"  # q/k/v/out dtype of the chunked path ("f32" or "bf16")
    chunk: int = 64
    lower_bound: float = -5.0
    scale: float | None = None  # None -> dk ** -0.5
    seed: int = 0
    state_std: float | None = None  # None -> zero initial state
    n_seqs: int = 0
    len_range: tuple = (0, 0)
    steps: int = 1
    extra: dict = field(default_factory=dict)

    @property
    def q_scale(self) -> float:
        return self.scale if self.scale is not None else self.dk ** -0.5


# The five workloads the library is measured and checked on.
TINY_F32 = Workload("tiny_f32_B1_T64_H2_d32_c16", "chunk", H=2, dk=32, dv=32, B=1, T=64,
                    dtype="f32", chunk=16, scale=1 / math.sqrt(32), seed=0)
DECODE_B64 = Workload("decode_f32_B64_H32_d128", "decode", H=32, dk=128, dv=128, B=64,
                      scale=1 / math.sqrt(128), seed=1, state_std=0.02)
PREFILL_B4 = Workload("prefill_bf16_B4_T4096_H32_d128_c64", "chunk", H=32, dk=128, dv=128,
                      B=4, T=4096, dtype="bf16", chunk=64, scale=1 / math.sqrt(128), seed=2)
VARLEN_8 = Workload("varlen_bf16_8seq_512to8192_H16_d128_c64", "varlen", H=16, dk=128,
                    dv=128, dtype="bf16", chunk=64, scale=1 / math.sqrt(128), seed=3,
                    state_std=0.02, n_seqs=8, len_range=(512, 8192))
DECODE_B512 = Workload("decode_f32_B512_H32_d128_x32", "decode", H=32, dk=128, dv=128,
                       B=512, scale=1 / math.sqrt(128), seed=4, state_std=0.02, steps=32)

WORKLOADS = {w.name: w for w in (TINY_F32, DECODE_B64, PREFILL_B4, VARLEN_8, DECODE_B512)}


def _rng(*key):
    return np.random.default_rng([int(x) for x in key])


def _normal(rng, shape, std=1.0):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def gate_params(H, dk, seed):
    """``a_log [H] ~ U(-1, 1)`` and ``dt_bias [dk, H] ~ N(0, 0.1)`` (model parameters)."""
    rng = _rng(seed, 7)
    a_log = rng.uniform(-1.0, 1.0, size=H).astype(np.float32)
    dt_bias = _normal(rng, (dk, H), 0.1)
    return a_log, dt_bias


def chunk_inputs(B, T, H, dk, dv, seed, state_std=None):
    """Inputs of the chunked forward in ``[B, T, H, .]`` layouts (all fp32 on the host)."""
    rng = _rng(seed, 1)
    d = {
        "q": _normal(rng, (B, T, H, dk)),
        "k": _normal(rng, (B, T, H, dk)),
        "v": _normal(rng, (B, T, H, dv)),
        "g": _normal(rng, (B, T, H, dk)),
        "beta_logits": _normal(rng, (B, T, H)),
    }
    d["a_log"], d["dt_bias"] = gate_params(H, dk, seed)
    d["initial_state"] = (None if state_std is None
                          else _normal(_rng(seed, 2), (B, H, dk, dv), state_std))
    return d


def varlen_lengths(n_seqs, lo, hi, seed):
    """Sequence lengths drawn uniformly from ``[lo, hi]`` (inclusive)."""
    rng = _rng(seed, 3)
    return rng.integers(lo, hi, size=n_seqs, endpoint=True).astype(np.int64)


def varlen_inputs(lengths, H, dk, dv, seed, state_std=0.02):
    """Packed inputs ``[total_T, H, .]`` plus ``cu_seqlens [N+1]`` (int32) and per-sequence
    initial states ``[N, H, dk, dv]``."""
    lengths = np.asarray(lengths, dtype=np.int64)
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    total = int(cu[-1])
    rng = _rng(seed, 1)
    d = {
        "q": _normal(rng, (total, H, dk)),
        "k": _normal(rng, (total, H, dk)),
        "v": _normal(rng, (total, H, dv)),
        "g": _normal(rng, (total, H, dk)),
        "beta_logits": _normal(rng, (total, H)),
        "cu_seqlens": cu,
    }
    d["a_log"], d["dt_bias"] = gate_params(H, dk, seed)
    d["initial_state"] = (None if state_std is None
                          else _normal(_rng(seed, 2), (len(lengths), H, dk, dv), state_std))
    return d


def decode_token_inputs(B, H, dk, dv, seed, step=0):
    """One decode token in the page-4 layouts: ``q, k, g [B, dk, H]``, ``v [B, H, dv]``,
    ``beta_logits [B, 1, H]``."""
    rng = _rng(seed, 10, step)
    return {
        "q": _normal(rng, (B, dk, H)),
        "k": _normal(rng, (B, dk, H)),
        "g": _normal(rng, (B, dk, H)),
        "v": _normal(rng, (B, H, dv)),
        "beta_logits": _normal(rng, (B, 1, H)),
    }


def decode_state(B, H, dk, dv, seed, std=0.02):
    """Initial decode state ``[B, H, dk, dv]`` ~ N(0, std)."""
    return _normal(_rng(seed, 2), (B, H, dk, dv), std)


def workload_inputs(w: Workload):
    """Inputs of a named workload (the first token only for decode workloads)."""
    if w.kind == "chunk":
        return chunk_inputs(w.B, w.T, w.H, w.dk, w.dv, w.seed, w.state_std)
    if w.kind == "varlen":
        lens = varlen_lengths(w.n_seqs, *w.len_range, w.seed)
        return varlen_inputs(lens, w.H, w.dk, w.dv, w.seed, w.state_std)
    if w.kind == "decode":
        d = decode_token_inputs(w.B, w.H, w.dk, w.dv, w.seed, 0)
        d["a_log"], d["dt_bias"] = gate_params(w.H, w.dk, w.seed)
        d["S"] = decode_state(w.B, w.H, w.dk, w.dv, w.seed, w.state_std or 0.02)
        return d
    raise ValueError(w.kind)
