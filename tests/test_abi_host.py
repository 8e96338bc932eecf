"""Host-only checks of the C ABI: the library loads, exports every symbol include/kda.h
declares, and rejects bad arguments on the host with the documented status codes before
anything touches a device.  No compute call is made."""
import ctypes
import os
import re

import pytest

import gated_delta_rule_55_gb300 as kda
from gated_delta_rule_55_gb300 import build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")
FAKE = 0x10000  # a 16-byte-aligned non-NULL address; never dereferenced by these tests


@pytest.fixture(scope="module")
def L():
    build_lib.build()
    return kda.lib()


def _declared():
    text = open(HEADER).read()
    return re.findall(r"^\s*(?:int|size_t|const char\s*\*)\s*(kda_\w+)\s*\(", text, re.M)


def test_header_declares_the_boundary():
    assert set(_declared()) == set(kda.kda.EXPORTS)


def test_every_declared_symbol_is_exported(L):
    for name in _declared():
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def test_status_strings_and_version(L):
    assert kda.kda_status_string(0) == "ok"
    for code in range(-13, 0):
        assert kda.kda_status_string(code) != "unknown kda status"
    assert kda.kda_status_string(-999) == "unknown kda status"
    assert kda.kda_version() >= 100


def _chunk(L, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, a_log=FAKE, dt_bias=FAKE, scale=0.0,
             lb=-5.0, s0=None, out=FAKE, s1=None, B=1, T=64, H=2, dk=32, dv=32, chunk=16,
             dtype=0)
    a.update(over)
    return L.kda_chunk_fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["a_log"],
                           a["dt_bias"], a["scale"], a["lb"], a["s0"], a["out"], a["s1"],
                           a["B"], a["T"], a["H"], a["dk"], a["dv"], a["chunk"], a["dtype"],
                           None)


def _decode(L, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, a_log=FAKE, dt_bias=FAKE, scale=0.1,
             lb=-5.0, out=FAKE, S=FAKE, B=4, H=2, dk=128, dv=128)
    a.update(over)
    return L.kda_decode_step(a["q"], a["k"], a["v"], a["g"], a["beta"], a["a_log"],
                             a["dt_bias"], a["scale"], a["lb"], a["out"], a["S"], a["B"],
                             a["H"], a["dk"], a["dv"], None)


def _varlen(L, **over):
    a = dict(cu=FAKE, N=2, total=10, H=2, dk=64, dv=64, chunk=64, dtype=1, lb=-1.0)
    a.update(over)
    return L.kda_chunk_fwd_varlen(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0.0, a["lb"],
                                  a["cu"], a["N"], a["total"], None, FAKE, None, a["H"],
                                  a["dk"], a["dv"], a["chunk"], a["dtype"], None)


@pytest.mark.parametrize("over,code", [
    (dict(q=None), -1), (dict(out=None), -1), (dict(dt_bias=None), -1),
    (dict(B=-1), -2), (dict(T=-3), -2), (dict(H=0), -2),
    (dict(dk=48), -3), (dict(dv=256), -3), (dict(dk=16), -3),
    (dict(chunk=32), -4), (dict(chunk=0), -4),
    (dict(lb=0.5), -5), (dict(lb=-5.5), -5), (dict(lb=float("nan")), -5),
    (dict(scale=float("inf")), -10), (dict(scale=float("nan")), -10),
    (dict(dtype=2), -7), (dict(q=FAKE + 4), -6), (dict(s0=FAKE + 8), -6),
    (dict(B=70000, T=1), -11),
])
def test_chunk_fwd_rejects_bad_arguments(L, over, code):
    assert _chunk(L, **over) == code


@pytest.mark.parametrize("over,code", [
    (dict(S=None), -1), (dict(B=-1), -2), (dict(H=0), -2), (dict(dk=256), -3),
    (dict(dv=8), -3), (dict(lb=1.0), -5), (dict(scale=float("nan")), -10),
    (dict(S=FAKE + 4), -6), (dict(q=FAKE + 12), -6),
])
def test_decode_rejects_bad_arguments(L, over, code):
    assert _decode(L, **over) == code


@pytest.mark.parametrize("over,code", [
    (dict(cu=None), -1), (dict(N=-1), -2), (dict(total=-1), -2), (dict(dk=100), -3),
    (dict(chunk=8), -4), (dict(lb=-6.0), -5), (dict(dtype=5), -7), (dict(cu=FAKE + 4), -6),
])
def test_varlen_rejects_bad_arguments(L, over, code):
    assert _varlen(L, **over) == code


def test_valid_call_without_a_device_reports_no_device(L):
    """On a machine without a GPU the first device query fails and the call returns
    KDA_ERR_DEVICE instead of launching (fake pointers are never touched)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this case is only meaningful without one")
    assert _chunk(L) == -9
    assert _decode(L) == -9
    assert _varlen(L) == -9


def test_binding_raises_on_error_status(L):
    with pytest.raises(kda.KDAError) as ei:
        kda.kda_decode_step(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0.1, 3.0, FAKE, FAKE,
                            1, 1, 128, 128, stream=0)
    assert ei.value.status == -5


# Workspace record of the two-launch path per (64-token chunk, head): four bf16 [64 x 128]
# tiles, one bf16 [64 x 64] tile and 256 fp32 values.
REC = 4 * 64 * 128 * 2 + 64 * 64 * 2 + 256 * 4


def test_workspace_size_formula(L):
    ws = kda.kda_chunk_fwd_workspace_size
    assert ws(4, 4096, 32, 128, 128, 64, 1) == 4 * 64 * 32 * REC
    assert ws(2, 65, 3, 128, 128, 64, 1) == 2 * 2 * 3 * REC      # ragged: 2 chunks each
    assert ws(2, 0, 3, 128, 128, 64, 1) == 0                     # no tokens
    # configurations that do not use the two-launch path need none
    assert ws(4, 4096, 32, 128, 128, 64, 0) == 0                 # fp32
    assert ws(4, 4096, 32, 128, 128, 16, 1) == 0                 # 16-token chunks
    assert ws(4, 4096, 32, 64, 128, 64, 1) == 0                  # dk = 64
    assert ws(-1, 4096, 32, 128, 128, 64, 1) == 0                # invalid
    vs = kda.kda_chunk_fwd_varlen_workspace_size
    # upper bound: total_T / 64 + N chunks, plus the (N + 1) int32 offsets rounded to 256 B,
    # plus the area for splitting long chains
    assert vs(8, 1000, 16, 128, 128, 64, 1) == \
        (1000 // 64 + 8) * 16 * REC + 256 + _split_area(8, 1000, 16)
    assert vs(300, 64 * 300, 2, 128, 128, 64, 1) == \
        (300 + 300) * 2 * REC + 1280 + _split_area(300, 64 * 300, 2)
    assert vs(8, 1000, 16, 128, 128, 64, 0) == 0


def _split_area(N, total, H, max_split=8):
    """The chain-split area of a packed forward: the chain table (N + 2 max_split int4), the
    counts (256 B), the split list (max_split int4), three fp32 [128 x 128] states per split
    sequence and head, and one bf16 row of 128 per (token, head); each part 256-byte
    aligned."""
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    return (al((N + 2 * max_split) * 16) + 256 + al(max_split * 16) +
            max_split * 3 * H * 128 * 128 * 4 + al(total * H * 128 * 2))


def _chunk_ws(L, ws, nbytes, **over):
    a = dict(B=1, T=64, H=2, dk=128, dv=128, chunk=64, dtype=1)
    a.update(over)
    return L.kda_chunk_fwd_ws(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0.0, -1.0, None, FAKE,
                              None, a["B"], a["T"], a["H"], a["dk"], a["dv"], a["chunk"],
                              a["dtype"], ws, nbytes, None)


def test_workspace_entry_rejects_bad_workspace(L):
    need = kda.kda_chunk_fwd_workspace_size(1, 64, 2, 128, 128, 64, 1)
    assert need == 2 * REC
    assert _chunk_ws(L, None, 0) == -12
    assert _chunk_ws(L, 0x100000, need - 1) == -12          # too small
    assert _chunk_ws(L, 0x100000 + 16, need) == -12         # not 256-byte aligned
    assert _chunk_ws(L, 0x100000, need, dk=100) == -3       # argument errors come first
    v = L.kda_chunk_fwd_varlen_ws(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0.0, -1.0, FAKE, 2,
                                  100, None, FAKE, None, 2, 128, 128, 64, 1, None, 0, None)
    assert v == -12


def test_workspace_entry_without_device(L):
    """A valid workspace call (or one whose configuration needs none, with a NULL
    workspace) reaches the device check and stops there on a machine without a GPU."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this case is only meaningful without one")
    need = kda.kda_chunk_fwd_workspace_size(1, 64, 2, 128, 128, 64, 1)
    assert _chunk_ws(L, 0x100000, need) == -9
    assert _chunk_ws(L, None, 0, dtype=0) == -9              # fp32: no workspace used
    assert _chunk_ws(L, None, 0, chunk=16) == -9


def _attn(L, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, beta=FAKE, decay=None, s0=None, out=FAKE, s1=None,
             scale=0.0, B=1, T=64, H=2, dk=64, dv=64, chunk=64, flags=0, dtype=1)
    a.update(over)
    return L.kda_attention_fwd(a["q"], a["k"], a["v"], a["beta"], a["decay"], a["s0"], a["out"],
                               a["s1"], a["scale"], a["B"], a["T"], a["H"], a["dk"], a["dv"],
                               a["chunk"], a["flags"], a["dtype"], None)


@pytest.mark.parametrize("over,code", [
    (dict(q=None), -1), (dict(beta=None), -1), (dict(out=None), -1), (dict(B=-1), -2),
    (dict(H=0), -2), (dict(dk=48), -3), (dict(dv=16), -3), (dict(chunk=32), -4),
    (dict(dtype=3), -7), (dict(flags=8), -13), (dict(flags=-1), -13),
    (dict(decay=FAKE + 4), -6), (dict(scale=float("nan")), -10), (dict(B=70000, T=1), -11),
])
def test_attention_rejects_bad_arguments(L, over, code):
    assert _attn(L, **over) == code


def test_attention_without_device(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this case is only meaningful without one")
    for flags in (0, 1, 2, 4, 7):
        assert _attn(L, flags=flags) == -9


def _attn_ws(L, ws, nbytes, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, beta=FAKE, decay=None, s0=None, out=FAKE, s1=None,
             scale=0.0, B=1, T=64, H=2, dk=128, dv=128, chunk=64, flags=0, dtype=1)
    a.update(over)
    return L.kda_attention_fwd_ws(a["q"], a["k"], a["v"], a["beta"], a["decay"], a["s0"],
                                  a["out"], a["s1"], a["scale"], a["B"], a["T"], a["H"], a["dk"],
                                  a["dv"], a["chunk"], a["flags"], a["dtype"], ws, nbytes, None)


def test_attention_ws_sizes_and_workspace_checks(L):
    need = kda.kda_attention_fwd_workspace_size(1, 64, 2, 128, 128, 64)
    # the same records as kda_chunk_fwd_ws: one per (64-token chunk, head)
    assert need == kda.kda_chunk_fwd_workspace_size(1, 64, 2, 128, 128, 64, 1) > 0
    assert kda.kda_attention_fwd_workspace_size(1, 64, 2, 128, 128, 64, use_chunked=False) == 0
    assert kda.kda_attention_fwd_workspace_size(1, 64, 2, 128, 128, 16) == 0
    assert kda.kda_attention_fwd_workspace_size(1, 64, 2, 64, 128, 64) == 0
    assert kda.kda_attention_fwd_workspace_size(1, 64, 2, 128, 128, 64, dtype=0) == 0
    assert kda.kda_attention_fwd_workspace_size(1, 0, 2, 128, 128, 64) == 0
    for flags in (0, 1, 4, 5):  # every chunked variant needs its workspace
        assert _attn_ws(L, None, 0, flags=flags) == -12
        assert _attn_ws(L, 0x100000, need - 1, flags=flags) == -12
        assert _attn_ws(L, 0x100080, need, flags=flags) == -12  # not 256-byte aligned
    assert _attn_ws(L, None, 0, dtype=3) == -7               # argument errors first
    assert _attn_ws(L, None, 0, flags=8) == -13


def test_attention_ws_without_device(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this case is only meaningful without one")
    need = kda.kda_attention_fwd_workspace_size(1, 64, 2, 128, 128, 64)
    assert _attn_ws(L, 0x100000, need) == -9
    assert _attn_ws(L, None, 0, flags=2) == -9               # the recurrent mode: no workspace
    assert _attn_ws(L, None, 0, dtype=0) == -9               # fp32: no workspace


def _al(x):
    return (x + 255) // 256 * 256


def _token_bwd_ws(B, T, H, dk, dv):
    nck, ns = (T + 63) // 64, dv // 32
    return (_al(B * H * nck * dk * dv * 4) + _al(B * H * 64 * dk * dv * 4) +
            3 * _al(ns * B * T * H * dk * 4) + _al(ns * B * T * H * 4))


def test_backward_workspace_size_formula(L):
    """Token-level path (fp32, or head dims other than 128): checkpoints every 64 tokens, one
    chunk of states per (sequence, head), and per 32-column value slice three fp32 per-token
    [dk] partial sums and one fp32 per-token scalar, each region 256-byte aligned."""
    B, T, H, dk, dv = 2, 150, 3, 128, 64
    for dt in (kda.KDA_F32, kda.KDA_BF16):
        assert kda.kda_chunk_bwd_workspace_size(B, T, H, dk, dv, dt) == _token_bwd_ws(B, T, H, dk, dv)
    assert kda.kda_chunk_bwd_workspace_size(B, T, H, 128, 128, kda.KDA_F32) == \
        _token_bwd_ws(B, T, H, 128, 128)
    assert kda.kda_chunk_bwd_workspace_size(B, T, H, 48, dv) == 0
    assert kda.kda_chunk_bwd_workspace_size(B, T, H, dk, dv, 2) == 0


def test_chunked_backward_workspace_size_formula(L):
    """Tensor-core path (bf16, dk = dv = 128): per (64-token chunk slot, head) the forward
    records (four 16 KB tiles, an 8 KB M tile, 1 KB of vectors; the region 256-byte aligned),
    then N (8 KB), the entering state and the state adjoint (32 KB each, bf16) and U^T and
    dU^T (16 KB each)."""
    B, T, H = 2, 150, 3
    recs = B * ((T + 63) // 64) * H
    want = _al(recs * (4 * 16384 + 8192 + 1024)) + recs * (8192 + 32768 + 16384 + 32768 + 16384)
    assert kda.kda_chunk_bwd_workspace_size(B, T, H, 128, 128, kda.KDA_BF16) == want


def _bwd(L, ws=0x100000, nbytes=1 << 40, **over):
    a = dict(q=FAKE, dout=FAKE, dq=FAKE, dg=FAKE, B=1, T=64, H=2, dk=64, dv=64, dtype=1)
    a.update(over)
    return L.kda_chunk_bwd(a["q"], FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0.0, -1.0, None,
                           a["dout"], None, a["dq"], FAKE, FAKE, a["dg"], FAKE, FAKE, FAKE,
                           None, a["B"], a["T"], a["H"], a["dk"], a["dv"], a["dtype"], ws,
                           nbytes, None)


@pytest.mark.parametrize("over,code", [
    (dict(q=None), -1), (dict(dout=None), -1), (dict(dq=None), -1), (dict(dg=None), -1),
    (dict(B=-1), -2), (dict(dk=48), -3), (dict(dtype=2), -7), (dict(dq=FAKE + 4), -6),
    (dict(ws=None), -12), (dict(nbytes=16), -12), (dict(ws=0x100000 + 64), -12),
])
def test_backward_rejects_bad_arguments(L, over, code):
    assert _bwd(L, **over) == code


def test_backward_without_device(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this case is only meaningful without one")
    assert _bwd(L) == -9


def _gla(L, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=None, gg=None, gk=None, gv=None, scale=0.0, s0=None,
             out=FAKE, s1=None, cu=None, N=0, B=2, T=16, Hq=4, Hkv=2, D=64, rev=0, dtype=1)
    a.update(over)
    return L.kda_recurrent_attention_fwd(a["q"], a["k"], a["v"], a["g"], a["gg"], a["gk"],
                                         a["gv"], a["scale"], a["s0"], a["out"], a["s1"],
                                         a["cu"], a["N"], a["B"], a["T"], a["Hq"], a["Hkv"],
                                         a["D"], a["rev"], a["dtype"], None)


@pytest.mark.parametrize("over,code", [
    (dict(q=None), -1), (dict(v=None), -1), (dict(out=None), -1), (dict(B=-1), -2),
    (dict(Hq=3), -2), (dict(Hkv=0), -2), (dict(cu=FAKE, B=2), -2), (dict(cu=FAKE, B=1, N=-1), -2),
    (dict(D=48), -3), (dict(scale=float("inf")), -10), (dict(dtype=4), -7),
    (dict(gk=FAKE + 8), -6),
])
def test_recurrent_attention_rejects_bad_arguments(L, over, code):
    assert _gla(L, **over) == code


def test_recurrent_attention_without_device(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this case is only meaningful without one")
    assert _gla(L) == -9
    assert _gla(L, cu=FAKE, B=1, N=3, rev=1) == -9


def _train(L, ws=0x100000, nbytes=1 << 40, **over):
    a = dict(B=1, T=64, H=2, dk=128, dv=128, chunk=64, dtype=1, out=FAKE)
    a.update(over)
    return L.kda_chunk_fwd_train(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0.0, -1.0, None,
                                 a["out"], None, a["B"], a["T"], a["H"], a["dk"], a["dv"],
                                 a["chunk"], a["dtype"], ws, nbytes, None)


@pytest.mark.parametrize("over,code", [
    (dict(out=None), -1), (dict(H=0), -2), (dict(dk=100), -3), (dict(dtype=0), -7),
    (dict(dtype=3), -7), (dict(dk=64), -3), (dict(dv=64), -3), (dict(chunk=16), -4),
    (dict(chunk=32), -4), (dict(ws=None), -12), (dict(nbytes=16), -12),
    (dict(ws=0x100000 + 64), -12),
])
def test_train_forward_rejects_bad_arguments(L, over, code):
    """The training forward serves the tensor-core configuration only; argument errors come
    before the device check."""
    assert _train(L, **over) == code


def test_train_forward_workspace_is_the_backward_workspace(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this case is only meaningful without one")
    need = kda.kda_chunk_bwd_workspace_size(1, 64, 2, 128, 128, kda.KDA_BF16)
    assert _train(L, nbytes=need - 1) == -12
    assert _train(L, nbytes=need) == -9                      # reaches the device check


def _bwd_saved(L, **over):
    a = dict(B=1, T=64, H=2, dk=128, dv=128, dtype=1)
    a.update(over)
    return L.kda_chunk_bwd_saved(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0.0, -1.0, None,
                                 FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None,
                                 a["B"], a["T"], a["H"], a["dk"], a["dv"], a["dtype"], 0x100000,
                                 1 << 40, None)


@pytest.mark.parametrize("over,code", [
    (dict(dtype=0), -7), (dict(dk=64), -3), (dict(dv=32), -3), (dict(dk=48), -3),
    (dict(B=-1), -2),
])
def test_saved_backward_rejects_other_configurations(L, over, code):
    assert _bwd_saved(L, **over) == code


def test_varlen_backward_workspace_size_formula(L):
    """Packed sequences: the fixed-length chunked layout over total_T / 64 + N chunk slots,
    with the (N + 1) int32 chunk offsets after the forward records."""
    N, total, H = 3, 1000, 2
    recs = (total // 64 + N) * H
    head = _al(recs * (4 * 16384 + 8192 + 1024) + (N + 1) * 4)
    want = head + recs * (8192 + 32768 + 16384 + 32768 + 16384)
    assert kda.kda_chunk_bwd_varlen_workspace_size(N, total, H, 128, 128, kda.KDA_BF16) == want
    assert kda.kda_chunk_bwd_varlen_workspace_size(N, total, H, 128, 128, kda.KDA_F32) == 0
    assert kda.kda_chunk_bwd_varlen_workspace_size(N, total, H, 64, 128, kda.KDA_BF16) == 0


def _bwd_varlen(L, **over):
    a = dict(cu=FAKE, N=2, total=100, H=2, dk=128, dv=128, dtype=1, ws=0x100000, nbytes=1 << 40)
    a.update(over)
    return L.kda_chunk_bwd_varlen(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0.0, -1.0, a["cu"],
                                  a["N"], a["total"], None, FAKE, None, FAKE, FAKE, FAKE, FAKE,
                                  FAKE, FAKE, FAKE, None, a["H"], a["dk"], a["dv"], a["dtype"],
                                  a["ws"], a["nbytes"], None)


@pytest.mark.parametrize("over,code", [
    (dict(cu=None), -1), (dict(N=-1), -2), (dict(dtype=0), -7), (dict(dk=64), -3),
    (dict(dv=32), -3), (dict(ws=None), -12), (dict(nbytes=16), -12),
])
def test_varlen_backward_rejects_bad_arguments(L, over, code):
    assert _bwd_varlen(L, **over) == code


def test_varlen_training_forward_rejects_other_configurations(L):
    def call(**over):
        a = dict(dtype=1, dk=128, chunk=64, ws=0x100000, nbytes=1 << 40)
        a.update(over)
        return L.kda_chunk_fwd_train_varlen(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0.0, -1.0,
                                            FAKE, 2, 100, None, FAKE, None, 2, a["dk"], 128,
                                            a["chunk"], a["dtype"], a["ws"], a["nbytes"], None)
    assert call(dtype=0) == -7
    assert call(dk=64) == -3
    assert call(chunk=16) == -4
    assert call(ws=None) == -12
    assert call(nbytes=64) == -12


@pytest.mark.parametrize("limit", [0, 1_000_000_001, 2**63])
def test_selftest_rejects_unbounded_limits(L, limit):
    """The self-test's wait limit must lie in (0, 1 s]: no argument can make it wait longer."""
    assert L.kda_selftest_bounded_wait(limit, None) == -2


def test_recurrent_workspace_sizes(L):
    """kda_recurrent_attention_fwd_workspace_size: the chunked path's records per (64-token
    chunk slot, query head) -- Q~, K^^T, M and the vector; with a value gate also V^, V~,
    e^{B - Q} and the sub-chunk totals (reverse order uses them too) -- plus, for packed
    sequences, the chunk offsets; 0 where the token-serial kernel runs (fp32, other head
    dims)."""
    f = L.kda_recurrent_attention_fwd_workspace_size
    per = 16384 + 16384 + 8192 + 1024
    vg = 3 * 16384 + 2048
    B, T, Hq, Hkv = 2, 300, 4, 2
    recs = B * ((T + 63) // 64) * Hq
    assert f(0, B, T, Hq, Hkv, 128, 0, 1) == recs * per
    assert f(0, B, T, Hq, Hkv, 128, 2, 1) == recs * (per + vg)
    assert f(0, B, T, Hq, Hkv, 128, 4, 1) == recs * (per + vg)  # reverse
    assert f(0, B, T, Hq, Hkv, 128, 2 | 4, 1) == recs * (per + vg)
    assert f(0, B, T, Hq, Hkv, 128, 2, 0) == 0  # fp32
    assert f(0, B, T, Hq, Hkv, 64, 2, 1) == 0  # D = 64
    N = 3
    recs = (T // 64 + N) * Hq
    assert f(N, 1, T, Hq, Hkv, 128, 1 | 2, 1) == recs * (per + vg) + ((N + 1) * 4 + 255) // 256 * 256
