"""GB300-native (sm_103a) Kimi / Kernel Delta Attention forward: a C-ABI CUDA library
(libkda.so, include/kda.h) and its thin Python binding."""
from .kda import (KDA_BF16, KDA_F32, KDAError, kda_attention_fwd, kda_attention_fwd_ws,  # noqa: F401
                  kda_attention_fwd_workspace_size, kda_chunk_bwd,
                  kda_chunk_bwd_saved, kda_chunk_bwd_saved_varlen, kda_chunk_bwd_varlen,
                  kda_chunk_bwd_varlen_workspace_size, kda_chunk_bwd_workspace_size, kda_chunk_fwd,
                  kda_chunk_fwd_noalloc, kda_chunk_fwd_train, kda_chunk_fwd_train_varlen,
                  kda_chunk_fwd_varlen,
                  kda_chunk_fwd_varlen_workspace_size, kda_chunk_fwd_varlen_ws,
                  kda_chunk_fwd_workspace_size, kda_chunk_fwd_ws, kda_decode_step,
                  kda_device_error, kda_recurrent_attention_fwd, kda_recurrent_attention_fwd_ws,
                  kda_recurrent_attention_fwd_workspace_size, kda_selftest_bounded_wait,
                  kda_status_string,
                  kda_version, lib)

__all__ = ["KDA_BF16", "KDA_F32", "KDAError", "kda_attention_fwd", "kda_attention_fwd_ws",
           "kda_attention_fwd_workspace_size", "kda_chunk_bwd",
           "kda_chunk_bwd_saved", "kda_chunk_bwd_saved_varlen", "kda_chunk_bwd_varlen",
           "kda_chunk_bwd_varlen_workspace_size", "kda_chunk_fwd_train_varlen",
           "kda_chunk_bwd_workspace_size", "kda_chunk_fwd",
           "kda_chunk_fwd_train",
           "kda_chunk_fwd_varlen", "kda_chunk_fwd_workspace_size",
           "kda_chunk_fwd_varlen_workspace_size", "kda_chunk_fwd_ws", "kda_chunk_fwd_varlen_ws",
           "kda_chunk_fwd_noalloc", "kda_recurrent_attention_fwd", "kda_recurrent_attention_fwd_ws",
           "kda_recurrent_attention_fwd_workspace_size", "kda_decode_step",
           "kda_device_error", "kda_selftest_bounded_wait", "kda_status_string",
           "kda_version", "lib"]
