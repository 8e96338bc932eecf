"""Thin ctypes binding of libkda (include/kda.h): the same entry-point names, argument
marshalling only.  Every step of the computation runs in the library's CUDA kernels;
there is no CPU or PyTorch fallback, and every call fails loudly when the library is
missing or returns an error.

Tensor arguments may be ``torch.Tensor`` (CUDA, contiguous), raw device addresses
(``int``) or ``None`` for the nullable ones.  ``stream`` defaults to torch's current
stream on the current device.
"""
from __future__ import annotations

import ctypes
import os

from .build_lib import LIB_PATH

KDA_F32 = 0
KDA_BF16 = 1
STATUS_NAMES = {
    0: "KDA_OK", -1: "KDA_ERR_NULL_POINTER", -2: "KDA_ERR_BAD_SHAPE", -3: "KDA_ERR_HEAD_DIM",
    -4: "KDA_ERR_CHUNK", -5: "KDA_ERR_LOWER_BOUND", -6: "KDA_ERR_MISALIGNED",
    -7: "KDA_ERR_DTYPE", -8: "KDA_ERR_LAUNCH", -9: "KDA_ERR_DEVICE", -10: "KDA_ERR_SCALE",
    -11: "KDA_ERR_TOO_LARGE", -12: "KDA_ERR_WORKSPACE", -13: "KDA_ERR_FLAGS",
}
# Exported symbols, in declaration order of include/kda.h.
EXPORTS = ("kda_chunk_fwd", "kda_chunk_fwd_varlen", "kda_chunk_fwd_workspace_size",
           "kda_chunk_fwd_varlen_workspace_size", "kda_chunk_fwd_ws", "kda_chunk_fwd_varlen_ws",
           "kda_chunk_fwd_noalloc", "kda_chunk_bwd_workspace_size", "kda_chunk_bwd",
           "kda_chunk_bwd_varlen_workspace_size", "kda_chunk_bwd_varlen",
           "kda_chunk_fwd_train_varlen", "kda_chunk_bwd_saved_varlen",
           "kda_chunk_fwd_train", "kda_chunk_bwd_saved", "kda_recurrent_attention_fwd", "kda_attention_fwd",
           "kda_attention_fwd_ws", "kda_attention_fwd_workspace_size",
           "kda_recurrent_attention_fwd_ws", "kda_recurrent_attention_fwd_workspace_size",
           "kda_decode_step",
           "kda_status_string",
           "kda_version", "kda_device_error", "kda_selftest_bounded_wait")
KDA_ATTN_NO_QK_L2NORM = 1
KDA_ATTN_RECURRENT = 2
KDA_ATTN_ORDER_LITERAL = 4


class KDAError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)} "
                         f"({kda_status_string(status)})")


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_Z = ctypes.c_size_t


def lib(path: str | None = None) -> ctypes.CDLL:
    """The loaded libkda.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libkda.so is not built ({p}); run "
                           "`python -m gated_delta_rule_55_gb300.build_lib`")
    L = ctypes.CDLL(p)
    L.kda_chunk_fwd.argtypes = [_P, _P, _P, _P, _P, _P, _P, _F, _F, _P, _P, _P,
                                _I, _I, _I, _I, _I, _I, _I, _P]
    L.kda_chunk_fwd_varlen.argtypes = [_P, _P, _P, _P, _P, _P, _P, _F, _F, _P, _I, _I,
                                       _P, _P, _P, _I, _I, _I, _I, _I, _P]
    L.kda_chunk_fwd_workspace_size.argtypes = [_I] * 7
    L.kda_chunk_fwd_varlen_workspace_size.argtypes = [_I] * 7
    L.kda_chunk_fwd_workspace_size.restype = _Z
    L.kda_chunk_fwd_varlen_workspace_size.restype = _Z
    L.kda_chunk_fwd_ws.argtypes = L.kda_chunk_fwd.argtypes[:-1] + [_P, _Z, _P]
    L.kda_chunk_fwd_varlen_ws.argtypes = L.kda_chunk_fwd_varlen.argtypes[:-1] + [_P, _Z, _P]
    L.kda_chunk_fwd_noalloc.argtypes = L.kda_chunk_fwd.argtypes
    L.kda_recurrent_attention_fwd.argtypes = ([_P] * 7 + [_F] + [_P] * 4 + [_I] * 8 + [_P])
    L.kda_recurrent_attention_fwd_ws.argtypes = ([_P] * 7 + [_F] + [_P] * 4 + [_I] * 8 +
                                                 [_P, _Z, _P])
    L.kda_recurrent_attention_fwd_workspace_size.argtypes = [_I] * 8
    L.kda_recurrent_attention_fwd_workspace_size.restype = _Z
    L.kda_chunk_bwd_workspace_size.argtypes = [_I] * 6
    L.kda_chunk_bwd_workspace_size.restype = _Z
    L.kda_chunk_bwd.argtypes = ([_P] * 7 + [_F, _F] + [_P] * 11 + [_I] * 6 + [_P, _Z, _P])
    L.kda_chunk_bwd_saved.argtypes = L.kda_chunk_bwd.argtypes
    L.kda_chunk_bwd_varlen_workspace_size.argtypes = [_I] * 6
    L.kda_chunk_bwd_varlen_workspace_size.restype = _Z
    L.kda_chunk_bwd_varlen.argtypes = ([_P] * 7 + [_F, _F, _P, _I, _I] + [_P] * 11 + [_I] * 4 +
                                       [_P, _Z, _P])
    L.kda_chunk_bwd_saved_varlen.argtypes = L.kda_chunk_bwd_varlen.argtypes
    L.kda_chunk_fwd_train_varlen.argtypes = L.kda_chunk_fwd_varlen_ws.argtypes
    L.kda_chunk_fwd_train.argtypes = L.kda_chunk_fwd_ws.argtypes
    L.kda_attention_fwd.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _F, _I, _I, _I, _I, _I, _I,
                                    _I, _I, _P]
    L.kda_attention_fwd_ws.argtypes = L.kda_attention_fwd.argtypes[:-1] + [_P, _Z, _P]
    L.kda_attention_fwd_workspace_size.argtypes = [_I] * 8
    L.kda_attention_fwd_workspace_size.restype = _Z
    L.kda_decode_step.argtypes = [_P, _P, _P, _P, _P, _P, _P, _F, _F, _P, _P,
                                  _I, _I, _I, _I, _P]
    L.kda_device_error.argtypes = [_I]
    L.kda_selftest_bounded_wait.argtypes = [ctypes.c_ulonglong, _P]
    L.kda_selftest_bounded_wait.restype = _I
    for f in ("kda_chunk_fwd", "kda_chunk_fwd_varlen", "kda_chunk_fwd_ws",
              "kda_chunk_fwd_varlen_ws", "kda_chunk_fwd_noalloc", "kda_chunk_bwd",
              "kda_chunk_bwd_saved", "kda_chunk_fwd_train", "kda_chunk_bwd_varlen",
              "kda_chunk_fwd_train_varlen", "kda_chunk_bwd_saved_varlen",
              "kda_attention_fwd", "kda_attention_fwd_ws", "kda_recurrent_attention_fwd",
              "kda_recurrent_attention_fwd_ws",
              "kda_decode_step", "kda_version", "kda_device_error"):
        getattr(L, f).restype = _I
    L.kda_status_string.argtypes = [_I]
    L.kda_status_string.restype = ctypes.c_char_p
    if path is None:
        _lib = L
    return L


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_cuda or not x.is_contiguous():
        raise ValueError("tensor arguments must be contiguous CUDA tensors")
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _dtype_code(x, dtype):
    if dtype is not None:
        return dtype
    import torch
    if x.dtype == torch.float32:
        return KDA_F32
    if x.dtype == torch.bfloat16:
        return KDA_BF16
    raise ValueError(f"unsupported q/k/v dtype {x.dtype}")


def _check(fn, status):
    if status != 0:
        raise KDAError(fn, status)


def kda_status_string(status: int) -> str:
    return lib().kda_status_string(int(status)).decode()


def kda_version() -> int:
    return lib().kda_version()


def kda_device_error(reset: bool = True) -> int:
    """Bitmask of device-side errors recorded since the last reset (synchronises)."""
    r = lib().kda_device_error(int(bool(reset)))
    if r < 0:
        raise KDAError("kda_device_error", r)
    return r


def kda_selftest_bounded_wait(limit_ns: int, stream=None) -> None:
    """Launch one bounded wait that runs out (sets bit 3 of kda_device_error)."""
    _check("kda_selftest_bounded_wait", lib().kda_selftest_bounded_wait(int(limit_ns),
                                                                         _stream(stream)))


def kda_chunk_fwd(q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound,
                  initial_state, out, final_state, B, T, H, dk, dv, chunk=64, dtype=None,
                  stream=None):
    """Chunked forward over B equal-length sequences (see include/kda.h)."""
    _check("kda_chunk_fwd", lib().kda_chunk_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta_logits), _ptr(a_log), _ptr(dt_bias),
        float(scale), float(lower_bound), _ptr(initial_state), _ptr(out), _ptr(final_state),
        B, T, H, dk, dv, chunk, _dtype_code(q, dtype), _stream(stream)))


def kda_chunk_fwd_varlen(q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound,
                         cu_seqlens, N, total_T, initial_state, out, final_state, H, dk, dv,
                         chunk=64, dtype=None, stream=None):
    """Chunked forward over N packed sequences (see include/kda.h)."""
    _check("kda_chunk_fwd_varlen", lib().kda_chunk_fwd_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta_logits), _ptr(a_log), _ptr(dt_bias),
        float(scale), float(lower_bound), _ptr(cu_seqlens), N, total_T, _ptr(initial_state),
        _ptr(out), _ptr(final_state), H, dk, dv, chunk, _dtype_code(q, dtype),
        _stream(stream)))


def kda_chunk_fwd_workspace_size(B, T, H, dk, dv, chunk=64, dtype=KDA_BF16) -> int:
    """Device workspace bytes kda_chunk_fwd_ws needs (0: none)."""
    return int(lib().kda_chunk_fwd_workspace_size(B, T, H, dk, dv, chunk, dtype))


def kda_chunk_fwd_varlen_workspace_size(N, total_T, H, dk, dv, chunk=64, dtype=KDA_BF16) -> int:
    """Device workspace bytes kda_chunk_fwd_varlen_ws needs (0: none)."""
    return int(lib().kda_chunk_fwd_varlen_workspace_size(N, total_T, H, dk, dv, chunk, dtype))


def _ws(workspace):
    """(pointer, bytes) of a workspace given as a CUDA tensor, (address, bytes) or None."""
    if workspace is None:
        return None, 0
    if isinstance(workspace, tuple):
        return workspace
    return _ptr(workspace), workspace.numel() * workspace.element_size()


def kda_chunk_fwd_ws(q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound,
                     initial_state, out, final_state, B, T, H, dk, dv, chunk=64, dtype=None,
                     workspace=None, stream=None):
    """kda_chunk_fwd through a caller workspace (two-launch path; see include/kda.h)."""
    wp, wb = _ws(workspace)
    _check("kda_chunk_fwd_ws", lib().kda_chunk_fwd_ws(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta_logits), _ptr(a_log), _ptr(dt_bias),
        float(scale), float(lower_bound), _ptr(initial_state), _ptr(out), _ptr(final_state),
        B, T, H, dk, dv, chunk, _dtype_code(q, dtype), wp, wb, _stream(stream)))


def kda_chunk_fwd_varlen_ws(q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound,
                            cu_seqlens, N, total_T, initial_state, out, final_state, H, dk, dv,
                            chunk=64, dtype=None, workspace=None, stream=None):
    """kda_chunk_fwd_varlen through a caller workspace (see include/kda.h)."""
    wp, wb = _ws(workspace)
    _check("kda_chunk_fwd_varlen_ws", lib().kda_chunk_fwd_varlen_ws(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta_logits), _ptr(a_log), _ptr(dt_bias),
        float(scale), float(lower_bound), _ptr(cu_seqlens), N, total_T, _ptr(initial_state),
        _ptr(out), _ptr(final_state), H, dk, dv, chunk, _dtype_code(q, dtype), wp, wb,
        _stream(stream)))


NOALLOC_SCRATCH_BYTES = 256 << 20  # include/kda.h KDA_NOALLOC_SCRATCH_BYTES


def kda_chunk_fwd_noalloc(q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound,
                          initial_state, out, final_state, B, T, H, dk, dv, chunk=64,
                          dtype=None, stream=None):
    """kda_chunk_fwd_ws with the library's own scratch array as the workspace (see
    include/kda.h)."""
    _check("kda_chunk_fwd_noalloc", lib().kda_chunk_fwd_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta_logits), _ptr(a_log), _ptr(dt_bias),
        float(scale), float(lower_bound), _ptr(initial_state), _ptr(out), _ptr(final_state),
        B, T, H, dk, dv, chunk, _dtype_code(q, dtype), _stream(stream)))


def kda_chunk_bwd_workspace_size(B, T, H, dk, dv, dtype=KDA_BF16) -> int:
    """Device workspace bytes kda_chunk_bwd needs for q/k/v of `dtype` (0: unsupported)."""
    return int(lib().kda_chunk_bwd_workspace_size(B, T, H, dk, dv, dtype))


def kda_chunk_bwd(q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound, initial_state,
                  d_out, d_final_state, dq, dk, dv, dg, dbeta_logits, da_log, ddt_bias,
                  d_initial_state, B, T, H, dk_dim, dv_dim, dtype=None, workspace=None,
                  stream=None):
    """Gradients of kda_chunk_fwd (see include/kda.h)."""
    wp, wb = _ws(workspace)
    _check("kda_chunk_bwd", lib().kda_chunk_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta_logits), _ptr(a_log), _ptr(dt_bias),
        float(scale), float(lower_bound), _ptr(initial_state), _ptr(d_out), _ptr(d_final_state),
        _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta_logits), _ptr(da_log), _ptr(ddt_bias),
        _ptr(d_initial_state), B, T, H, dk_dim, dv_dim, _dtype_code(q, dtype), wp, wb,
        _stream(stream)))


def kda_chunk_bwd_varlen_workspace_size(N, total_T, H, dk, dv, dtype=KDA_BF16) -> int:
    """Device workspace bytes kda_chunk_bwd_varlen needs (0: unsupported)."""
    return int(lib().kda_chunk_bwd_varlen_workspace_size(N, total_T, H, dk, dv, dtype))


def kda_chunk_bwd_varlen(q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound,
                         cu_seqlens, N, total_T, initial_state, d_out, d_final_state, dq, dk,
                         dv, dg, dbeta_logits, da_log, ddt_bias, d_initial_state, H, dk_dim,
                         dv_dim, dtype=None, workspace=None, stream=None):
    """Gradients of kda_chunk_fwd_varlen (packed sequences; see include/kda.h)."""
    wp, wb = _ws(workspace)
    _check("kda_chunk_bwd_varlen", lib().kda_chunk_bwd_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta_logits), _ptr(a_log), _ptr(dt_bias),
        float(scale), float(lower_bound), _ptr(cu_seqlens), N, total_T, _ptr(initial_state),
        _ptr(d_out), _ptr(d_final_state), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg),
        _ptr(dbeta_logits), _ptr(da_log), _ptr(ddt_bias), _ptr(d_initial_state), H, dk_dim,
        dv_dim, _dtype_code(q, dtype), wp, wb, _stream(stream)))


def kda_chunk_fwd_train_varlen(q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound,
                               cu_seqlens, N, total_T, initial_state, out, final_state, H, dk,
                               dv, chunk=64, dtype=None, workspace=None, stream=None):
    """The packed-sequence training forward (see include/kda.h)."""
    wp, wb = _ws(workspace)
    _check("kda_chunk_fwd_train_varlen", lib().kda_chunk_fwd_train_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta_logits), _ptr(a_log), _ptr(dt_bias),
        float(scale), float(lower_bound), _ptr(cu_seqlens), N, total_T, _ptr(initial_state),
        _ptr(out), _ptr(final_state), H, dk, dv, chunk, _dtype_code(q, dtype), wp, wb,
        _stream(stream)))


def kda_chunk_bwd_saved_varlen(q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound,
                               cu_seqlens, N, total_T, initial_state, d_out, d_final_state, dq,
                               dk, dv, dg, dbeta_logits, da_log, ddt_bias, d_initial_state, H,
                               dk_dim, dv_dim, dtype=None, workspace=None, stream=None):
    """kda_chunk_bwd_varlen reading what kda_chunk_fwd_train_varlen kept in ``workspace``."""
    wp, wb = _ws(workspace)
    _check("kda_chunk_bwd_saved_varlen", lib().kda_chunk_bwd_saved_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta_logits), _ptr(a_log), _ptr(dt_bias),
        float(scale), float(lower_bound), _ptr(cu_seqlens), N, total_T, _ptr(initial_state),
        _ptr(d_out), _ptr(d_final_state), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg),
        _ptr(dbeta_logits), _ptr(da_log), _ptr(ddt_bias), _ptr(d_initial_state), H, dk_dim,
        dv_dim, _dtype_code(q, dtype), wp, wb, _stream(stream)))


def kda_chunk_fwd_train(q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound,
                        initial_state, out, final_state, B, T, H, dk, dv, chunk=64, dtype=None,
                        workspace=None, stream=None):
    """The forward, keeping the backward's records in ``workspace`` (see include/kda.h)."""
    wp, wb = _ws(workspace)
    _check("kda_chunk_fwd_train", lib().kda_chunk_fwd_train(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta_logits), _ptr(a_log), _ptr(dt_bias),
        float(scale), float(lower_bound), _ptr(initial_state), _ptr(out), _ptr(final_state),
        B, T, H, dk, dv, chunk, _dtype_code(q, dtype), wp, wb, _stream(stream)))


def kda_chunk_bwd_saved(q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound,
                        initial_state, d_out, d_final_state, dq, dk, dv, dg, dbeta_logits,
                        da_log, ddt_bias, d_initial_state, B, T, H, dk_dim, dv_dim, dtype=None,
                        workspace=None, stream=None):
    """kda_chunk_bwd reading what kda_chunk_fwd_train kept in ``workspace``."""
    wp, wb = _ws(workspace)
    _check("kda_chunk_bwd_saved", lib().kda_chunk_bwd_saved(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta_logits), _ptr(a_log), _ptr(dt_bias),
        float(scale), float(lower_bound), _ptr(initial_state), _ptr(d_out), _ptr(d_final_state),
        _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta_logits), _ptr(da_log), _ptr(ddt_bias),
        _ptr(d_initial_state), B, T, H, dk_dim, dv_dim, _dtype_code(q, dtype), wp, wb,
        _stream(stream)))


def kda_recurrent_attention_fwd(query, key, value, out, B, T, Hq, Hkv, D, g=None, g_gamma=None,
                                gk=None, gv=None, softmax_scale=None, initial_state=None,
                                final_state=None, cu_seqlens=None, N=0, reverse=False,
                                dtype=None, stream=None):
    """The recurrent page's gated linear recurrence (see include/kda.h)."""
    _check("kda_recurrent_attention_fwd", lib().kda_recurrent_attention_fwd(
        _ptr(query), _ptr(key), _ptr(value), _ptr(g), _ptr(g_gamma), _ptr(gk), _ptr(gv),
        float(softmax_scale or 0.0), _ptr(initial_state), _ptr(out), _ptr(final_state),
        _ptr(cu_seqlens), N, B, T, Hq, Hkv, D, int(bool(reverse)), _dtype_code(query, dtype),
        _stream(stream)))


KDA_REC_PACKED, KDA_REC_VALUE_GATE, KDA_REC_REVERSE = 1, 2, 4  # include/kda.h


def kda_recurrent_attention_fwd_workspace_size(B, T, Hq, Hkv, D, N=0, packed=False,
                                               value_gate=False, reverse=False,
                                               dtype=KDA_BF16):
    """Bytes of workspace kda_recurrent_attention_fwd_ws needs (0: none; see include/kda.h)."""
    flags = ((KDA_REC_PACKED if packed else 0) | (KDA_REC_VALUE_GATE if value_gate else 0) |
             (KDA_REC_REVERSE if reverse else 0))
    return int(lib().kda_recurrent_attention_fwd_workspace_size(N, B, T, Hq, Hkv, D, flags,
                                                                dtype))


def kda_recurrent_attention_fwd_ws(query, key, value, out, B, T, Hq, Hkv, D, g=None,
                                   g_gamma=None, gk=None, gv=None, softmax_scale=None,
                                   initial_state=None, final_state=None, cu_seqlens=None, N=0,
                                   reverse=False, dtype=None, workspace=None, stream=None):
    """kda_recurrent_attention_fwd through a caller workspace (chunked tensor-core path; see
    include/kda.h)."""
    wp, wb = _ws(workspace)
    _check("kda_recurrent_attention_fwd_ws", lib().kda_recurrent_attention_fwd_ws(
        _ptr(query), _ptr(key), _ptr(value), _ptr(g), _ptr(g_gamma), _ptr(gk), _ptr(gv),
        float(softmax_scale or 0.0), _ptr(initial_state), _ptr(out), _ptr(final_state),
        _ptr(cu_seqlens), N, B, T, Hq, Hkv, D, int(bool(reverse)), _dtype_code(query, dtype),
        wp, wb, _stream(stream)))


def kda_attention_fwd(query, key, value, beta, decay, initial_state, out, final_state, B, T, H,
                      dk, dv, softmax_scale=None, chunk=64, use_qk_l2norm=True,
                      use_chunked=True, order="decay_first", dtype=None, stream=None):
    """The kernel_delta_attention call: per-head log-decay (None: no decay), beta as given
    (see include/kda.h)."""
    flags = ((0 if use_qk_l2norm else KDA_ATTN_NO_QK_L2NORM) |
             (0 if use_chunked else KDA_ATTN_RECURRENT) |
             {"decay_first": 0, "literal": KDA_ATTN_ORDER_LITERAL}[order])
    _check("kda_attention_fwd", lib().kda_attention_fwd(
        _ptr(query), _ptr(key), _ptr(value), _ptr(beta), _ptr(decay), _ptr(initial_state),
        _ptr(out), _ptr(final_state), float(softmax_scale or 0.0), B, T, H, dk, dv, chunk,
        flags, _dtype_code(query, dtype), _stream(stream)))


def _attn_flags(use_qk_l2norm, use_chunked, order):
    return ((0 if use_qk_l2norm else KDA_ATTN_NO_QK_L2NORM) |
            (0 if use_chunked else KDA_ATTN_RECURRENT) |
            {"decay_first": 0, "literal": KDA_ATTN_ORDER_LITERAL}[order])


def kda_attention_fwd_workspace_size(B, T, H, dk, dv, chunk=64, use_qk_l2norm=True,
                                     use_chunked=True, order="decay_first", dtype=KDA_BF16):
    """Bytes of workspace kda_attention_fwd_ws needs (0: none; see include/kda.h)."""
    return int(lib().kda_attention_fwd_workspace_size(
        B, T, H, dk, dv, chunk, _attn_flags(use_qk_l2norm, use_chunked, order), dtype))


def kda_attention_fwd_ws(query, key, value, beta, decay, initial_state, out, final_state, B, T,
                         H, dk, dv, softmax_scale=None, chunk=64, use_qk_l2norm=True,
                         use_chunked=True, order="decay_first", dtype=None, workspace=None,
                         stream=None):
    """kda_attention_fwd through a caller workspace (tensor-core path; see include/kda.h)."""
    wp, wb = _ws(workspace)
    _check("kda_attention_fwd_ws", lib().kda_attention_fwd_ws(
        _ptr(query), _ptr(key), _ptr(value), _ptr(beta), _ptr(decay), _ptr(initial_state),
        _ptr(out), _ptr(final_state), float(softmax_scale or 0.0), B, T, H, dk, dv, chunk,
        _attn_flags(use_qk_l2norm, use_chunked, order), _dtype_code(query, dtype), wp, wb,
        _stream(stream)))


def kda_decode_step(q, k, v, g, beta_logits, a_log, dt_bias, scale, lower_bound, out, S,
                    B, H, dk, dv, stream=None):
    """One decode token for B requests, S updated in place (see include/kda.h)."""
    _check("kda_decode_step", lib().kda_decode_step(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta_logits), _ptr(a_log), _ptr(dt_bias),
        float(scale), float(lower_bound), _ptr(out), _ptr(S), B, H, dk, dv, _stream(stream)))
