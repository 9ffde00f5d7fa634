"""CPU checks of the C ABI: the library loads, exports every entry point that
include/usp.h declares, and rejects bad arguments on the host with a status
code before touching the GPU.  No compute call is made here."""
import ctypes

import numpy as np
import pytest

from ulysses_sequence_attention_usp_gb300 import binding as B
from oracle import usp_oracle as O


def test_exports_every_declared_entry_point():
    names = B.header_entry_points()
    assert {"usp_pad_shard", "usp_seq_to_head_rope", "usp_attn_fwd", "usp_attn_bwd",
            "usp_head_to_seq", "usp_attn_bwd_workspace"} <= set(names)
    for n in names:
        assert hasattr(B._lib, n), n


def test_version_and_status_strings():
    assert B.usp_abi_version() == 1
    for s in range(6):
        assert B.usp_status_string(s)
    assert "divisible" in B.usp_status_string(2)


def _dims(**kw):
    base = dict(S=256, P=2, Hq=4, Hkv=2, D=64)
    base.update(kw)
    return B.make_dims(**base)


FAKE = 1 << 20   # 16-byte aligned fake device address: never dereferenced


def _fwd(d, ptr=FAKE, doc=FAKE):
    return B.raw_call("usp_attn_fwd", ctypes.byref(d), ptr, ptr, ptr, doc, ptr, ptr, None)


@pytest.mark.parametrize("kw,status", [
    (dict(P=3), 2), (dict(Hq=6, Hkv=4), 2), (dict(P=4, Hkv=2), 2), (dict(P=0), 2),
    (dict(D=96), 3), (dict(D=256), 3), (dict(S=-1), 1), (dict(Hq=0), 1),
])
def test_fwd_rejects_bad_dims(kw, status):
    assert _fwd(_dims(**kw)) == status


def test_fwd_rejects_bad_pointers():
    d = _dims()
    assert _fwd(d, ptr=None) == 1
    assert _fwd(d, ptr=FAKE + 8) == 1          # misaligned
    assert _fwd(d, doc=None) == 1


def test_causal_flag_and_scale_checked():
    d = _dims()
    d.causal = 2                                # 1 causal, 0 bidirectional, else invalid
    assert _fwd(d) == 1
    d.causal = -1
    assert _fwd(d) == 1
    d = _dims(scale=-1.0)
    assert _fwd(d) == 1
    d = _dims()
    d.zigzag = 2                                # 0 contiguous, 1 zigzag, else invalid
    assert _fwd(d) == 1


def test_window_and_merge_arguments_checked():
    d = _dims()                                 # S_pad = 256
    args = [ctypes.byref(d)] + [FAKE] * 4
    for lo, hi in ((5, 4), (-1, 8), (0, 257)):
        assert B.raw_call("usp_attn_fwd_window", *args, ctypes.c_int64(lo), ctypes.c_int64(hi),
                          FAKE, FAKE, None) == 1
    assert B.raw_call("usp_lse_merge", ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, 2, None,
                      None) == 1
    assert B.raw_call("usp_lse_merge", ctypes.byref(d), FAKE, None, FAKE, FAKE, 1, None,
                      None) == 1


def test_zigzag_pad_shard_cannot_run_in_place():
    d = _dims()
    d.zigzag = 1
    st = B.raw_call("usp_pad_shard", ctypes.byref(d), FAKE, 2, FAKE, None, None, None)
    assert st == 1


def test_bwd_workspace_size_and_checks():
    d = _dims()
    ws = B.usp_attn_bwd_workspace(d)
    assert ws >= 2 * (2 * 2 * 256) * 4              # delta and LSE*log2e, fp32
    assert B.usp_attn_bwd_workspace(_dims(P=3)) == 0
    args = [ctypes.byref(d)] + [FAKE] * 11
    assert B.raw_call("usp_attn_bwd", *args, ctypes.c_size_t(ws - 1), None) == 1
    args = [ctypes.byref(d)] + [FAKE] * 10 + [FAKE + 16]  # workspace not 256-aligned
    assert B.raw_call("usp_attn_bwd", *args, ctypes.c_size_t(ws), None) == 1


def test_rope_table_must_cover_padded_length():
    d = _dims(S=250)                                 # S_pad = 250 (P=2)
    call = lambda n, mode=1: B.raw_call(           # noqa: E731
        "usp_seq_to_head_rope", ctypes.byref(d), FAKE, 4, FAKE, FAKE, n, mode, FAKE * 2, None)
    assert call(249) == 1
    assert call(0, mode=2) == 1
    d2 = _dims(S=251)                                # pads to 252
    assert B.raw_call("usp_seq_to_head_rope", ctypes.byref(d2), FAKE, 4, FAKE, FAKE, 251, 1,
                      FAKE * 2, None) == 1
    # heads of the repacked tensor must divide by P
    assert B.raw_call("usp_seq_to_head_rope", ctypes.byref(d), FAKE, 3, FAKE, FAKE, 256, 1,
                      FAKE * 2, None) == 2


def test_cu_seqlens_host_mirror_validated():
    cu_bad = np.array([0, 100, 90, 256], np.int32)      # not monotone
    d = B.make_dims(256, 2, 4, 2, 64, cu_seqlens=FAKE_TENSOR(4), cu_seqlens_host=cu_bad)
    assert _fwd(d) == 1
    cu_short = np.array([0, 100, 200], np.int32)        # does not end at S
    d = B.make_dims(256, 2, 4, 2, 64, cu_seqlens=FAKE_TENSOR(3), cu_seqlens_host=cu_short)
    assert _fwd(d) == 1


class FAKE_TENSOR:
    """Stands in for a device tensor: only its address and size are used."""
    def __init__(self, n):
        self.n = n

    def numel(self):
        return self.n

    def data_ptr(self):
        return FAKE


def test_empty_sequence_is_a_no_op():
    d = _dims(S=0)
    assert _fwd(d) == 0
    assert B.raw_call("usp_pad_shard", ctypes.byref(d), FAKE, 4, FAKE, FAKE, FAKE, None) == 0


def test_one_shard_geometry_takes_fewer_kv_heads_than_ranks():
    # the K/V all-gather CP path runs on P = 1, which accepts any Hkv | Hq;
    # the same heads over P = 4 shards are refused by the all-to-all
    assert _fwd(_dims(S=0, P=1, Hq=4, Hkv=1)) == 0
    assert _fwd(_dims(S=0, P=4, Hq=4, Hkv=1)) == 2
    d = _dims(S=0, P=1, Hq=4, Hkv=1)
    for H in (4, 1):
        assert B.raw_call("usp_seq_to_head_rope", ctypes.byref(d), FAKE, H, FAKE, FAKE,
                          ctypes.c_int64(0), 0, FAKE + 4096, None) == 0


@pytest.mark.parametrize("n,D,base,f,L", [(300, 64, 1.0e4, 1.0, 0), (4096, 128, 1.0e6, 1.0, 0),
                                          (131072, 128, 1.0e6, 4.0, 32768)])
def test_library_rope_table_matches_oracle(n, D, base, f, L):
    # the product builds its own table; it must agree with the oracle's
    # (both round fp64 cos/sin to fp32; libm and numpy may differ by one
    # fp64 ulp, which can flip an fp32 rounding only very rarely)
    a = B.usp_rope_table(n, D, base, f, L)
    b = O.rope_table_f32(n, D, base, f, L)
    diff = a.view(np.int32).astype(np.int64) - b.view(np.int32).astype(np.int64)
    assert np.max(np.abs(diff)) <= 1
    assert np.count_nonzero(diff) <= max(2, a.size // 10**6)


def test_selftest_wait_limit_validated_on_host():
    assert B.raw_call("usp_selftest_bounded_wait", 0, None) == 1
    assert B.raw_call("usp_selftest_bounded_wait", 2000000, None) == 1
