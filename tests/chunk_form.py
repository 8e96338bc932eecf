"""The chunked (WY / UT-transform) form of the KDA recurrence, written out in numpy.

Test helper, not the oracle: it restates, step by step and in plain numpy, the chunk
algebra that the CUDA kernels implement, so the tests can show that it equals the
oracle's token scan (an exact re-association, so fp64 agreement is ~1e-12) and that its
factorised gate exponentials stay finite in fp32 at the steepest allowed gate.

Derivation (decay-first recurrence of the ``kernel_delta_attention`` page's "core
recurrence"): with ``S_t = D_t S_{t-1} + k_t u_t^T`` and ``u_t = beta_t (v_t - (D_t
S_{t-1})^T k_t)``, and ``G_r = sum_{s<=r} gamma_s`` inside a chunk of C tokens,

    S_r = diag(e^{G_r}) S_0 + sum_{s<=r} diag(e^{G_r - G_s}) k_s u_s^T.

Substituting gives, with rows indexed by token,

    (I + diag(beta) L) U = diag(beta) (V - K~ S_0),   L_rs = sum_c k_r k_s e^{G_r - G_s} (s < r)
    U = T V - (T K~) S_0,  T = (I + diag(beta) L)^{-1} diag(beta),  K~_r = e^{G_r} * k_r
    O = Q~ S_0 + M U,      M_rs = sum_c q_r k_s e^{G_r - G_s} (s <= r), Q~_r = e^{G_r} * q_r
    S_C = diag(e^{G_C}) S_0 + K^T U,   K^_s = e^{G_C - G_s} * k_s.

``e^{G_r - G_s}`` is split with one reference per 16-token sub-chunk R: ``P_R`` is G just
before the sub-chunk starts (``P_0 = 0``), ``e_r = e^{G_r - P_R(r)}`` lies in
``[e^{-16*5}, 1]`` for ``lower_bound >= -5``, the key side uses ``k_s / e_s`` (at most
``e^{80}``), and pairs of different sub-chunks pick up the per-channel constant
``e^{P_R - P_S} <= 1``.  No factor leaves the fp32 range.
"""
from __future__ import annotations

import numpy as np

SUB = 16


def chunk_core(q_hat, k_hat, v, gamma, beta, S0, C, dtype=np.float64):
    """Chunked forward for ONE (batch, head) pair after the prologue.

    ``q_hat, k_hat, gamma [T, dk]`` (q_hat already scaled), ``v [T, dv]``, ``beta [T]``,
    ``S0 [dk, dv]``.  Returns ``(out [T, dv], S_T [dk, dv])``.  A ragged last chunk is
    handled by simply using fewer rows.
    """
    f = lambda x: np.asarray(x, dtype=dtype)  # noqa: E731
    q_hat, k_hat, v, gamma, beta, S = map(f, (q_hat, k_hat, v, gamma, beta, S0))
    T, dk = k_hat.shape
    out = np.zeros((T, v.shape[1]), dtype=dtype)
    with np.errstate(over="raise", invalid="raise", under="ignore"):
        for t0 in range(0, T, C):
            n = min(C, T - t0)
            sl = slice(t0, t0 + n)
            G = np.cumsum(gamma[sl], axis=0)
            R = np.arange(n) // SUB
            nsub = int(R[-1]) + 1
            P = np.zeros((nsub, dk), dtype=dtype)
            for r in range(1, nsub):
                P[r] = G[SUB * r - 1]
            e = np.exp(G - P[R])
            Xk = k_hat[sl] * e
            Xq = q_hat[sl] * e
            Kd = k_hat[sl] / e
            A = np.zeros((n, n), dtype=dtype)
            Mq = np.zeros((n, n), dtype=dtype)
            for rb in range(nsub):
                rows = slice(rb * SUB, min(n, rb * SUB + SUB))
                for sb in range(rb + 1):
                    cols = slice(sb * SUB, min(n, sb * SUB + SUB))
                    Kb = Kd[cols] if sb == rb else Kd[cols] * np.exp(P[rb] - P[sb])
                    A[rows, cols] = Xk[rows] @ Kb.T
                    Mq[rows, cols] = Xq[rows] @ Kb.T
            L = np.tril(A, -1)
            Mq = np.tril(Mq, 0)
            b = beta[sl]
            Tm = np.linalg.solve(np.eye(n, dtype=dtype) + b[:, None] * L, np.diag(b))
            EP = np.exp(P[R])
            Kt = Xk * EP  # e^{G_r} k_r
            Qt = Xq * EP  # e^{G_r} q_r
            W = Tm @ Kt
            Ut = Tm @ v[sl]
            U = Ut - W @ S
            out[sl] = Qt @ S + Mq @ U
            Gc = G[n - 1]
            Kh = Kd * np.exp(Gc - P[R])  # e^{G_C - G_s} k_s
            S = np.exp(Gc)[:, None] * S + Kh.T @ U
    return out, S
