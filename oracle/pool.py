"""Runs the fp64 oracle over independent problems in spawned worker processes.

TEST INFRASTRUCTURE, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of ``bench.py`` use it.

It holds none of the method's arithmetic.  Different (sequence, head) pairs never interact
in the recurrence (the kernel_delta_attention page keeps one memory per batch element and
head; the recurrent page's ``cu_seqlens`` gives every packed sequence its own), so a large
problem is cut into groups of pairs, each group is handed unchanged to ``kda_forward`` /
``kda_decode_step`` in a worker process, and the results are put back in place.  Workers
are started with the ``spawn`` method, so a pool may be created after CUDA has been
initialised in the parent, and each worker runs its numpy single-threaded.
"""
from __future__ import annotations

import multiprocessing as mp
import os
from concurrent.futures import ProcessPoolExecutor

import numpy as np

_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def default_workers() -> int:
    return max(1, os.cpu_count() or 1)


def _call(name, kwargs):
    from oracle import kda_oracle
    return getattr(kda_oracle, name)(**kwargs)


def _ready(_i=0):
    return os.getpid()


class Pool:
    """A process pool of ``workers`` spawned workers (default: every host core), each with
    single-threaded numpy.  ``ex`` is the executor; ``close()`` shuts it down."""

    def __init__(self, workers=None):
        self.workers = workers or default_workers()
        self._saved = {v: os.environ.get(v) for v in _THREAD_VARS}
        for v in _THREAD_VARS:
            os.environ[v] = "1"  # inherited by the workers; the parent's numpy is unaffected
        self.ex = ProcessPoolExecutor(max_workers=self.workers,
                                      mp_context=mp.get_context("spawn"))
        list(self.ex.map(_ready, range(4 * self.workers)))

    def close(self):
        if self.ex is not None:
            self.ex.shutdown(wait=True, cancel_futures=True)
            self.ex = None
            for v, x in self._saved.items():
                if x is None:
                    os.environ.pop(v, None)
                else:
                    os.environ[v] = x

    def __enter__(self):
        return self.ex

    def __exit__(self, *exc):
        self.close()


def _run(ex, name, tasks):
    futs = [ex.submit(_call, name, kw) for kw in tasks]
    return [f.result() for f in futs]


def _head_groups(H, n_outer, workers):
    """Contiguous head ranges so that n_outer * len(ranges) is at least the worker count."""
    per = max(1, (H * n_outer) // max(1, workers))
    per = min(H, max(1, per))
    return [(h, min(H, h + per)) for h in range(0, H, per)]


def forward(ex, q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound,
            initial_state=None, workers=None):
    """``kda_forward`` over ``[B, T, H, .]`` inputs, one task per (batch element, head
    range).  Same return value as ``kda_forward``: ``(out [B,T,H,dv], state [B,H,dk,dv])``."""
    B, T, H, dk = np.shape(q)
    dv = np.shape(v)[-1]
    groups = _head_groups(H, B, workers or default_workers())
    tasks, where = [], []
    for b in range(B):
        for h0, h1 in groups:
            tasks.append(dict(
                q=q[b:b + 1, :, h0:h1], k=k[b:b + 1, :, h0:h1], v=v[b:b + 1, :, h0:h1],
                g=g[b:b + 1, :, h0:h1], beta_logits=beta_logits[b:b + 1, :, h0:h1],
                a_log=a_log[h0:h1], dt_bias=dt_bias[:, h0:h1], scale=scale,
                lower_bound=lower_bound,
                initial_state=None if initial_state is None
                else initial_state[b:b + 1, h0:h1]))
            where.append((b, h0, h1))
    out = np.zeros((B, T, H, dv))
    state = np.zeros((B, H, dk, dv))
    for (b, h0, h1), (o, s) in zip(where, _run(ex, "kda_forward", tasks)):
        out[b, :, h0:h1] = o[0]
        state[b, h0:h1] = s[0]
    return out, state


def forward_varlen(ex, q, k, v, g, beta_logits, a_log, dt_bias, cu_seqlens, scale,
                   lower_bound, initial_state=None, workers=None):
    """``kda_forward_varlen`` over packed ``[total_T, H, .]`` inputs, one task per
    (sequence, head range).  Same return value as ``kda_forward_varlen``."""
    total, H, dk = np.shape(q)
    dv = np.shape(v)[-1]
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    groups = _head_groups(H, N, workers or default_workers())
    tasks, where = [], []
    for n in range(N):
        a, b = int(cu[n]), int(cu[n + 1])
        for h0, h1 in groups:
            tasks.append(dict(
                q=q[None, a:b, h0:h1], k=k[None, a:b, h0:h1], v=v[None, a:b, h0:h1],
                g=g[None, a:b, h0:h1], beta_logits=beta_logits[None, a:b, h0:h1],
                a_log=a_log[h0:h1], dt_bias=dt_bias[:, h0:h1], scale=scale,
                lower_bound=lower_bound,
                initial_state=None if initial_state is None
                else initial_state[n:n + 1, h0:h1]))
            where.append((n, a, b, h0, h1))
    out = np.zeros((total, H, dv))
    state = np.zeros((N, H, dk, dv))
    for (n, a, b, h0, h1), (o, s) in zip(where, _run(ex, "kda_forward", tasks)):
        out[a:b, h0:h1] = o[0]
        state[n, h0:h1] = s[0]
    return out, state


def _decode_chain(tokens, a_log, dt_bias, scale, lower_bound, S):
    from oracle import kda_oracle
    outs = []
    for t in tokens:
        o, S = kda_oracle.kda_decode_step(**t, a_log=a_log, dt_bias=dt_bias, scale=scale,
                                          lower_bound=lower_bound, S=S)
        outs.append(o)
    return np.stack(outs), S


def decode_chain(ex, tokens, a_log, dt_bias, scale, lower_bound, S0, workers=None):
    """Consecutive ``kda_decode_step`` calls (the state passed from one to the next) for a
    list of tokens in the kda_tkg layouts, one task per head range.  Returns
    ``(outs [steps, B, H, dv], state [B, H, dk, dv])``."""
    B, H, dk, dv = np.shape(S0)
    groups = _head_groups(H, 1, workers or default_workers())
    futs = []
    for h0, h1 in groups:
        sub = [{"q": t["q"][:, :, h0:h1], "k": t["k"][:, :, h0:h1], "g": t["g"][:, :, h0:h1],
                "v": t["v"][:, h0:h1], "beta_logits": t["beta_logits"][:, :, h0:h1]}
               for t in tokens]
        futs.append(ex.submit(_decode_chain, sub, a_log[h0:h1], dt_bias[:, h0:h1], scale,
                              lower_bound, S0[:, h0:h1]))
    outs = np.zeros((len(tokens), B, H, dv))
    state = np.zeros((B, H, dk, dv))
    for (h0, h1), f in zip(groups, futs):
        o, s = f.result()
        outs[:, :, h0:h1] = o
        state[:, h0:h1] = s
    return outs, state


def recurrent(ex, query, key, value, g=None, g_gamma=None, gk=None, gv=None,
              softmax_scale=None, initial_state=None, workers=None, reverse=False):
    """``recurrent_attention`` (either order, fixed-length sequences) over
    ``[B, T, Hq, D]`` inputs, one task per (batch element, range of query heads); each range
    covers whole groups of query heads sharing a key / value head.  Same return value as
    ``recurrent_attention``."""
    B, T, Hq, D = np.shape(query)
    Hkv = np.shape(key)[2]
    grp = Hq // Hkv
    per = max(1, (Hkv * B) // max(1, workers or default_workers()))
    per = min(Hkv, per)
    tasks, where = [], []
    for b in range(B):
        for k0 in range(0, Hkv, per):
            k1 = min(Hkv, k0 + per)
            h0, h1 = k0 * grp, k1 * grp
            sl = lambda x: None if x is None else x[b:b + 1, :, h0:h1]  # noqa: E731
            tasks.append(dict(
                query=query[b:b + 1, :, h0:h1], key=key[b:b + 1, :, k0:k1],
                value=value[b:b + 1, :, k0:k1], g=sl(g), gk=sl(gk), gv=sl(gv),
                g_gamma=None if g_gamma is None else g_gamma[b:b + 1, h0:h1],
                softmax_scale=softmax_scale, reverse=reverse,
                initial_state=None if initial_state is None else initial_state[b:b + 1, h0:h1]))
            where.append((b, h0, h1))
    out = np.zeros((B, T, Hq, D))
    state = np.zeros((B, Hq, D, D))
    for (b, h0, h1), (o, s) in zip(where, _run(ex, "recurrent_attention", tasks)):
        out[b, :, h0:h1] = o[0]
        state[b, h0:h1] = s[0]
    return out, state
