"""Plain fp64 CPU oracle for the Kimi / Kernel Delta Attention (KDA) forward pass.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module: only
``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may call it.  It shares no code with the CUDA library.

What it computes, and from which passage
----------------------------------------
* Recurrence -- ejkernel ``kernel_delta_attention`` module page, "The core recurrence":
  a per-(batch, head) memory ``h`` of shape ``[dk, dv]``; every token decays it with
  ``exp(decay_t)``, adds ``k_t (x) (beta_t * (v_t - h @ k_t))`` and emits ``o_t = h_t @ q_t``.
  ``h @ x`` contracts over the key axis (``h`` is ``[dk, dv]``), so it is ``h^T x`` here.
* Gate, beta, scale -- NKI "KDA TKG Kernel API Reference", ``kda_tkg`` parameters:
  the raw per-channel gate ``g`` becomes ``lower_bound * sigmoid(exp(a_log) * (g + dt_bias))``;
  ``beta`` arrives as logits and goes through a sigmoid; q and k are L2-normalised and
  ``scale`` is folded into the normalised query.
* State passthrough -- ``kernel_delta_attention`` page, ``initial_state`` / ``return_state``
  parameters; ``kda_tkg``'s ``S`` is read and overwritten in place.
* Varlen packing -- ejkernel ``recurrent`` module page, ``cu_seqlens`` parameter.

Readings where the pages are silent or ambiguous
------------------------------------------------
1. Decay before delta (``order="decay_first"``, the default): the error term is taken
   against the decayed memory, ``S' = diag(exp(gamma)) S``, ``u = beta (v - S'^T k)``,
   ``S <- S' + k u^T``.  The recurrence as printed uses the undecayed memory inside the
   error term; that literal reading is kept as ``order="literal"``.  Both agree when the
   gate is identically zero.
2. The output is read after the update (``o_t = h_t @ q_t``).
3. L2 normalisation is ``x / sqrt(sum(x^2) + 1e-6)`` over the head dimension (epsilon
   unstated on the pages).
4. ``scale`` multiplies the normalised query; default ``dk ** -0.5``.
5. The gate is per channel (``[..., dk]``) and raw, as in ``kda_tkg``; beta is a logit.
6. Outputs are returned in fp64; dtype handling (bf16 inputs) is the caller's business:
   callers pass the already-rounded values.

The algorithm is the plain token-by-token scan: no chunking, no blocking and no
re-association, vectorised only over independent (batch, head) pairs.
"""
from __future__ import annotations

import numpy as np

L2_EPS = 1e-6


def sigmoid(x):
    """Logistic function 1 / (1 + exp(-x)) in fp64 (``kda_tkg`` beta and gate)."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-x))


def activate_gate(g, a_log, dt_bias, lower_bound):
    """Per-channel log-decay ``gamma = lower_bound * sigmoid(exp(a_log) * (g + dt_bias))``.

    ``kda_tkg`` parameters g / a_log / dt_bias / lower_bound.  ``g`` has the head axis
    second-to-last and the channel axis last (``[..., H, dk]``); ``a_log`` is ``[H]``;
    ``dt_bias`` is ``[dk, H]`` exactly as the page lays it out.  Returns fp64 ``[..., H, dk]``.
    """
    g = np.asarray(g, dtype=np.float64)
    a = np.exp(np.asarray(a_log, dtype=np.float64))[:, None]  # [H, 1]
    bias = np.asarray(dt_bias, dtype=np.float64).T  # [H, dk]
    return float(lower_bound) * sigmoid(a * (g + bias))


def l2_normalize(x, eps=L2_EPS):
    """``x / sqrt(sum(x^2) + eps)`` over the last axis (reading 3)."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def kda_token(S, q_hat, k_hat, v, gamma, beta, order="decay_first"):
    """Advance the memory by one token; returns ``(o, S_new)``.

    Shapes (any leading batch dims ``...``): ``S [..., dk, dv]``, ``q_hat, k_hat, gamma
    [..., dk]``, ``v [..., dv]``, ``beta [...]``.  ``q_hat`` already carries ``scale``.
    ``kernel_delta_attention`` page, "The core recurrence" (with reading 1 for the order).
    """
    decay = np.exp(gamma)[..., :, None]  # diag(exp(gamma)) acting on the rows of S
    b = np.asarray(beta)[..., None]
    if order == "decay_first":
        S_dec = decay * S
        pred = np.einsum("...ij,...i->...j", S_dec, k_hat)  # S'^T k
        u = b * (v - pred)
        S_new = S_dec + k_hat[..., :, None] * u[..., None, :]
    elif order == "literal":
        pred = np.einsum("...ij,...i->...j", S, k_hat)  # h_{t-1} @ k_t, undecayed
        u = b * (v - pred)
        S_new = decay * S + k_hat[..., :, None] * u[..., None, :]
    else:
        raise ValueError(f"unknown order {order!r}")
    o = np.einsum("...ij,...i->...j", S_new, q_hat)  # o_t = h_t @ q_t, after the update
    return o, S_new


def kda_forward(q, k, v, g, beta_logits, a_log, dt_bias, scale=None, lower_bound=-5.0,
                initial_state=None, order="decay_first"):
    """Whole-sequence KDA forward, the plain token scan.

    Layouts follow ``kernel_delta_attention.run``: ``q, k, g [B, T, H, dk]``,
    ``v [B, T, H, dv]``, ``beta_logits [B, T, H]``, ``initial_state [B, H, dk, dv]``
    (``None`` means zeros); gate parameters as in ``kda_tkg`` (``a_log [H]``,
    ``dt_bias [dk, H]``).  Returns ``(out [B, T, H, dv], final_state [B, H, dk, dv])``
    in fp64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if scale is None:
        scale = dk ** -0.5
    gamma = activate_gate(g, a_log, dt_bias, lower_bound)  # [B, T, H, dk]
    beta = sigmoid(beta_logits)  # [B, T, H]
    q_hat = float(scale) * l2_normalize(q)
    k_hat = l2_normalize(k)
    if initial_state is None:
        S = np.zeros((B, H, dk, dv), dtype=np.float64)
    else:
        S = np.array(initial_state, dtype=np.float64, copy=True)
    out = np.zeros((B, T, H, dv), dtype=np.float64)
    for t in range(T):
        o, S = kda_token(S, q_hat[:, t], k_hat[:, t], v[:, t], gamma[:, t], beta[:, t], order)
        out[:, t] = o
    return out, S


def kda_forward_varlen(q, k, v, g, beta_logits, a_log, dt_bias, cu_seqlens, scale=None,
                       lower_bound=-5.0, initial_state=None, order="decay_first"):
    """Packed variable-length forward (``cu_seqlens`` convention of the ejkernel
    ``recurrent`` page): sequence ``n`` owns tokens ``cu_seqlens[n]:cu_seqlens[n+1]`` of
    the packed ``[total_T, H, .]`` tensors and starts from ``initial_state[n]``.

    Returns ``(out [total_T, H, dv], final_state [N, H, dk, dv])``.
    """
    q = np.asarray(q, dtype=np.float64)
    total_T, H, dk = q.shape
    dv = np.shape(v)[-1]
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    out = np.zeros((total_T, H, dv), dtype=np.float64)
    final = np.zeros((N, H, dk, dv), dtype=np.float64)
    for n in range(N):
        a, b = int(cu[n]), int(cu[n + 1])
        s0 = None if initial_state is None else np.asarray(initial_state)[n:n + 1]
        o, s = kda_forward(np.asarray(q)[None, a:b], np.asarray(k)[None, a:b],
                           np.asarray(v)[None, a:b], np.asarray(g)[None, a:b],
                           np.asarray(beta_logits)[None, a:b], a_log, dt_bias, scale,
                           lower_bound, s0, order)
        out[a:b] = o[0]
        final[n] = s[0]
    return out, final


def kda_decode_step(q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound, S,
                    order="decay_first"):
    """One token for B requests in the ``kda_tkg`` layouts.

    ``q, k, g [B, dk, H]`` (head innermost), ``v [B, H, dv]``, ``beta_logits [B, 1, H]``,
    ``a_log [1, H]`` or ``[H]``, ``dt_bias [dk, H]``, ``S [B, H, dk, dv]``.
    Returns ``(out [B, H, dv], S_new [B, H, dk, dv])``; the input ``S`` is not modified
    (the kernel's in-place contract is the caller's to emulate).
    """
    q = np.swapaxes(np.asarray(q, dtype=np.float64), 1, 2)  # -> [B, H, dk]
    k = np.swapaxes(np.asarray(k, dtype=np.float64), 1, 2)
    g = np.swapaxes(np.asarray(g, dtype=np.float64), 1, 2)
    v = np.asarray(v, dtype=np.float64)
    gamma = activate_gate(g, np.reshape(a_log, -1), dt_bias, lower_bound)
    beta = sigmoid(np.asarray(beta_logits, dtype=np.float64)[:, 0, :])  # [B, H]
    q_hat = float(scale) * l2_normalize(q)
    k_hat = l2_normalize(k)
    S = np.asarray(S, dtype=np.float64)
    return kda_token(S, q_hat, k_hat, v, gamma, beta, order)


def kda_attention(query, key, value, beta, decay=None, initial_state=None, softmax_scale=None,
                  use_qk_l2norm=True, order="decay_first"):
    """The ``kernel_delta_attention`` / ``kda_attention`` call of the ejkernel
    ``kernel_delta_attention`` page, as the plain token scan.

    Parameters as on that page: ``query, key [B, T, H, dk]``, ``value [B, T, H, dv]``,
    ``beta [B, T, H]`` -- a per-token learning rate used as given (the page's example
    passes probabilities through a sigmoid itself) --, ``decay [B, T, H]`` -- a per-head
    log-decay, the same for every key channel, ``None`` meaning zeros (full retention) --,
    ``initial_state [B, H, dk, dv]`` (``None`` means zeros), ``softmax_scale`` (default
    ``dk ** -0.5``, applied to the query), ``use_qk_l2norm`` (normalise q and k over the head
    dimension before use).  ``use_chunked`` only selects an algorithm for the same result,
    so it has no counterpart here.  Returns ``(out [B, T, H, dv], final_state)`` in fp64.
    """
    q = np.asarray(query, dtype=np.float64)
    k = np.asarray(key, dtype=np.float64)
    v = np.asarray(value, dtype=np.float64)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    scale = dk ** -0.5 if softmax_scale is None else float(softmax_scale)
    if use_qk_l2norm:
        q = l2_normalize(q)
        k = l2_normalize(k)
    q_hat = scale * q
    d = (np.zeros((B, T, H)) if decay is None else np.asarray(decay, dtype=np.float64))
    gamma = np.broadcast_to(d[..., None], (B, T, H, dk))  # one log-decay for every channel
    b = np.asarray(beta, dtype=np.float64)
    if initial_state is None:
        S = np.zeros((B, H, dk, dv), dtype=np.float64)
    else:
        S = np.array(initial_state, dtype=np.float64, copy=True)
    out = np.zeros((B, T, H, dv), dtype=np.float64)
    for t in range(T):
        o, S = kda_token(S, q_hat[:, t], k[:, t], v[:, t], gamma[:, t], b[:, t], order)
        out[:, t] = o
    return out, S


def kda_backward(q, k, v, g, beta_logits, a_log, dt_bias, d_out, d_final_state=None,
                 scale=None, lower_bound=-5.0, initial_state=None, order="decay_first"):
    """Gradients of ``L = sum(d_out * out) + sum(d_final_state * final_state)`` for the
    forward of ``kda_forward`` (same arguments and layouts), by reverse-mode differentiation
    of the token scan.  The pages give no backward: this is the chain rule applied to each
    step of the recurrence, in reverse token order.

    Per token (decay first; ``D = diag(exp(gamma))``)::

        S' = D S;  p = S'^T k^;  u = beta (v - p);  S_new = S' + k^ u^T;  o = S_new^T q^

    with the adjoint ``dS`` of ``S_new`` (``d_final_state`` at the end)::

        dS   += q^ do^T;          dq^ = S_new do
        du    = dS^T k^;          dk^ = dS u
        dv    = beta du;          dbeta = du . (v - p);   dp = -beta du
        dS'   = dS + k^ dp^T;     dk^ += S' dp
        dgamma = exp(gamma) * rowsum(dS' * S);            dS (previous) = D dS'

    (literal order: ``p`` reads ``S``, so ``dk^ += S dp`` and ``dS (previous) = D dS + k^ dp^T``,
    ``dgamma = exp(gamma) * rowsum(dS * S)``).  Then through the L2 norms, the scale, the
    beta sigmoid and the gate ``lower_bound * sigmoid(exp(a_log) (g + dt_bias))``.

    Returns a dict: ``dq, dk, dv, dg, dbeta_logits, da_log [H], ddt_bias [dk, H],
    dinitial_state``, all fp64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if scale is None:
        scale = dk ** -0.5
    a = np.exp(np.asarray(a_log, dtype=np.float64))            # [H]
    bias = np.asarray(dt_bias, dtype=np.float64).T             # [H, dk]
    z = a[:, None] * (g + bias)                                # [B, T, H, dk]
    sz = sigmoid(z)
    gamma = float(lower_bound) * sz
    beta = sigmoid(beta_logits)
    nq = np.sqrt(np.sum(q * q, axis=-1, keepdims=True) + L2_EPS)
    nk = np.sqrt(np.sum(k * k, axis=-1, keepdims=True) + L2_EPS)
    q_hat = float(scale) * q / nq
    k_hat = k / nk
    S = (np.zeros((B, H, dk, dv)) if initial_state is None
         else np.array(initial_state, dtype=np.float64, copy=True))
    states = [S]                                               # state before each token
    for t in range(T):
        _, S = kda_token(S, q_hat[:, t], k_hat[:, t], v[:, t], gamma[:, t], beta[:, t], order)
        states.append(S)
    d_out = np.asarray(d_out, dtype=np.float64)
    dS = (np.zeros((B, H, dk, dv)) if d_final_state is None
          else np.array(d_final_state, dtype=np.float64, copy=True))
    dq_hat = np.zeros_like(q)
    dk_hat = np.zeros_like(k)
    dvv = np.zeros_like(v)
    dbeta = np.zeros((B, T, H))
    dgamma = np.zeros_like(g)
    for t in range(T - 1, -1, -1):
        S_prev, S_new = states[t], states[t + 1]
        e = np.exp(gamma[:, t])                                # [B, H, dk]
        kh, qh, b = k_hat[:, t], q_hat[:, t], beta[:, t]
        do = d_out[:, t]                                       # [B, H, dv]
        S_dec = e[..., :, None] * S_prev
        base = S_dec if order == "decay_first" else S_prev     # what the error term reads
        p = np.einsum("bhij,bhi->bhj", base, kh)
        u = b[..., None] * (v[:, t] - p)
        dS = dS + qh[..., :, None] * do[..., None, :]
        dq_hat[:, t] = np.einsum("bhij,bhj->bhi", S_new, do)
        du = np.einsum("bhij,bhi->bhj", dS, kh)
        dk_t = np.einsum("bhij,bhj->bhi", dS, u)
        dvv[:, t] = b[..., None] * du
        dbeta[:, t] = np.sum(du * (v[:, t] - p), axis=-1)
        dp = -b[..., None] * du
        dk_t += np.einsum("bhij,bhj->bhi", base, dp)
        if order == "decay_first":
            dS_dec = dS + kh[..., :, None] * dp[..., None, :]
            dgamma[:, t] = e * np.sum(dS_dec * S_prev, axis=-1)
            dS = e[..., :, None] * dS_dec
        else:
            dgamma[:, t] = e * np.sum(dS * S_prev, axis=-1)
            dS = e[..., :, None] * dS + kh[..., :, None] * dp[..., None, :]
        dk_hat[:, t] = dk_t
    # L2 norms (x^ = x / n, n = sqrt(|x|^2 + eps)): dx = dx^ / n - x (x . dx^) / n^3
    dqn = float(scale) * dq_hat
    dq = dqn / nq - q * np.sum(q * dqn, axis=-1, keepdims=True) / nq ** 3
    dk_ = dk_hat / nk - k * np.sum(k * dk_hat, axis=-1, keepdims=True) / nk ** 3
    dz = dgamma * float(lower_bound) * sz * (1.0 - sz)         # d/dz of lb sigmoid(z)
    return {
        "dq": dq, "dk": dk_, "dv": dvv,
        "dg": dz * a[:, None],
        "dbeta_logits": dbeta * beta * (1.0 - beta),
        "da_log": np.sum(dz * z, axis=(0, 1, 3)),
        "ddt_bias": np.sum(dz * a[:, None], axis=(0, 1)).T,
        "dinitial_state": dS,
    }


def recurrent_attention(query, key, value, g=None, g_gamma=None, gk=None, gv=None,
                        softmax_scale=None, initial_state=None, reverse=False, cu_seqlens=None):
    """The ``recurrent_attention`` call of the ejkernel ``recurrent`` page, as a plain token
    loop.  The page lists the parameters but prints no recurrence; the reading used here is
    the gated linear recurrence its gate names describe (all gates are log-space decays):

        a_t = g_t + gk_t + g_gamma    (key axis; each term only when given)
        h_t = diag(exp(a_t)) h_{t-1} diag(exp(gv_t)) + k_t v_t^T,    o_t = h_t^T (scale q_t)

    Layouts as on the page: ``query [B, T, Hq, D]``, ``key, value [B, T, Hkv, D]`` (query head
    ``h`` reads key/value head ``h // (Hq / Hkv)``), ``g, gk, gv [B, T, Hq, D]``,
    ``g_gamma [B, Hq]``, ``initial_state [B, Hq, D, D]`` (``None``: zeros).  ``reverse`` runs
    each sequence from its last token to its first.  With ``cu_seqlens`` the tensors are
    packed (``B = 1``) and sequence ``n`` owns tokens ``cu_seqlens[n]:cu_seqlens[n + 1]``,
    with ``initial_state [N, Hq, D, D]``.  Returns ``(out [B, T, Hq, D], final_state)``,
    fp64.
    """
    q = np.asarray(query, dtype=np.float64)
    k = np.asarray(key, dtype=np.float64)
    v = np.asarray(value, dtype=np.float64)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    grp = Hq // Hkv
    scale = D ** -0.5 if softmax_scale is None else float(softmax_scale)
    a = np.zeros((B, T, Hq, D))
    if g is not None:
        a = a + np.asarray(g, dtype=np.float64)
    if gk is not None:
        a = a + np.asarray(gk, dtype=np.float64)
    if g_gamma is not None:
        a = a + np.asarray(g_gamma, dtype=np.float64)[:, None, :, None]
    bv = np.zeros((B, T, Hq, D)) if gv is None else np.asarray(gv, dtype=np.float64)
    kk = np.repeat(k, grp, axis=2)  # key / value head of every query head
    vv = np.repeat(v, grp, axis=2)
    if cu_seqlens is None:
        spans = [(b, 0, T) for b in range(B)]
        nstate = B
    else:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        spans = [(0, int(cu[n]), int(cu[n + 1])) for n in range(len(cu) - 1)]
        nstate = len(cu) - 1
    out = np.zeros((B, T, Hq, D))
    final = np.zeros((nstate, Hq, D, D))
    for n, (b, lo, hi) in enumerate(spans):
        h = (np.zeros((Hq, D, D)) if initial_state is None
             else np.array(initial_state[n], dtype=np.float64, copy=True))
        order = range(hi - 1, lo - 1, -1) if reverse else range(lo, hi)
        for t in order:
            h = np.exp(a[b, t])[:, :, None] * h * np.exp(bv[b, t])[:, None, :]
            h = h + kk[b, t][:, :, None] * vv[b, t][:, None, :]
            out[b, t] = np.einsum("hij,hi->hj", h, scale * q[b, t])
        final[n] = h
    return out, final
