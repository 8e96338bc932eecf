"""fp64 CPU oracle for the KDA forward pass -- test infrastructure, never the product path.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference
legs may import this package.
"""
from .kda_oracle import (  # noqa: F401
    L2_EPS,
    activate_gate,
    kda_attention,
    kda_backward,
    kda_decode_step,
    kda_forward,
    kda_forward_varlen,
    kda_token,
    l2_normalize,
    recurrent_attention,
    sigmoid,
)
