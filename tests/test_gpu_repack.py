"""GPU parity of shard/pad and the all-to-all repack kernels: bit-exact
against the oracle (permutation, positions, and the fp32 RoPE recipe)."""
import ctypes

import numpy as np
import pytest
import torch

from oracle import usp_oracle as O
from ulysses_sequence_attention_usp_gb300 import binding as B
from ulysses_sequence_attention_usp_gb300.inputs import WORKLOADS, cu_seqlens, normal_bf16

from gpu_util import to_bits, to_dev

pytestmark = pytest.mark.gpu


def _dims(S, P, Hq, Hkv, D, cu=None):
    cu_dev = None if cu is None else torch.from_numpy(np.asarray(cu, np.int32)).cuda()
    return B.make_dims(S, P, Hq, Hkv, D, cu_dev, None if cu is None else np.asarray(cu, np.int32))


PAD_CASES = [
    (7, 4, 4, 4, 64, [0, 3, 7]),
    (30, 4, 8, 4, 128, None),
    (256, 2, 4, 2, 64, None),
    (1, 8, 8, 8, 64, None),
    (65536, 8, 8, 8, 128, list(cu_seqlens([4656, 1304, 590, 542, 8578, 12109, 4191, 6416, 3369,
                                            13083, 8655, 517, 1526]))),
    (32766, 8, 8, 8, 128, None),
]


@pytest.mark.parametrize("S,P,Hq,Hkv,D,cu", PAD_CASES)
def test_pad_shard_positions_docs(S, P, Hq, Hkv, D, cu):
    d = _dims(S, P, Hq, Hkv, D, cu)
    x = normal_bf16((S, Hq, D), 3, "q")
    S_pad = O.padded_len(S, P)
    xs = torch.full((S_pad, Hq, D), 7.0, dtype=torch.bfloat16, device="cuda")
    pos = torch.full((S_pad,), -5, dtype=torch.int32, device="cuda")
    doc = torch.full((S_pad,), -5, dtype=torch.int32, device="cuda")
    B.usp_pad_shard(d, to_dev(x), Hq, xs, pos, doc)
    torch.cuda.synchronize()
    want_pos, want_doc = O.positions_docs(S, P, None if cu is None else np.array(cu))
    assert np.array_equal(pos.cpu().numpy(), want_pos)
    assert np.array_equal(doc.cpu().numpy(), want_doc)
    assert np.array_equal(to_bits(xs), O.shard_pad(x, P))


def test_pad_shard_in_place_zeroes_tail_only():
    S, P, H, D = 30, 4, 4, 64
    d = _dims(S, P, H, H, D)
    x = normal_bf16((32, H, D), 4, "k")
    buf = to_dev(x)
    B.usp_pad_shard(d, buf, H, buf, None, None)
    torch.cuda.synchronize()
    got = to_bits(buf)
    assert np.array_equal(got[:30], x[:30]) and not got[30:].any()


def _repack_case(S, P, Hq, Hkv, D, cu, which, mode, rows=None, base=1.0e4, f=1.0, L=0,
                 rope_len=0, unpadded=False):
    """seq -> head of a padded [S_pad][H][D] source, or (unpadded=True) of the
    caller's [S][H][D] tensor, which the library reads only at valid rows."""
    H = Hq if which == "q" else Hkv
    d = _dims(S, P, Hq, Hkv, D, cu)
    S_pad = O.padded_len(S, P)
    n_pos = rope_len or S_pad
    table = O.rope_table_f32(n_pos, D, base, f, L)
    x = O.shard_pad(normal_bf16((S, H, D), 11, which), P)
    pos, _ = O.positions_docs(S, P, None if cu is None else np.array(cu))
    out = torch.full((P, S_pad, H // P, D), 3.0, dtype=torch.bfloat16, device="cuda")
    tpos = torch.from_numpy(pos.astype(np.int32)).cuda()
    ttab = torch.from_numpy(table).cuda()
    B.usp_seq_to_head_rope(d, to_dev(x[:S] if unpadded else x), H, tpos, ttab, n_pos, mode, out)
    torch.cuda.synchronize()
    got = to_bits(out)
    if rows is None:
        rows = np.arange(S_pad)
    sub = x[rows]
    if mode != 0:
        sub = O.rope_recipe_bf16(sub, pos[rows], table, inverse=mode < 0)
    # the permutation acts row by row: row t, head g*H/P + j -> [g][t][j]
    want = sub.reshape(len(rows), P, H // P, D).transpose(1, 0, 2, 3)
    assert np.array_equal(got[:, rows], want)


@pytest.mark.parametrize("which,mode", [("q", 1), ("k", 1), ("v", 0), ("q", -1)])
def test_seq_to_head_tiny(which, mode):
    _repack_case(256, 2, 4, 2, 64, None, which, mode)


@pytest.mark.parametrize("case", [
    (1000, 2, 8, 2, 128, None),
    (777, 4, 8, 4, 64, [0, 100, 101, 401, 777]),
    (30, 4, 8, 4, 128, None),
    (1, 8, 8, 8, 128, None),
    # one shard, an odd number of rows: the few-head passes take two rows
    # per warp and the last pair holds a single row
    (777, 1, 4, 2, 128, None),
    (255, 1, 2, 2, 64, [0, 100, 255]),
])
def test_seq_to_head_small_ragged(case):
    for which, mode in (("q", 1), ("k", 1), ("v", 0)):
        _repack_case(*case, which, mode)


@pytest.mark.parametrize("case", [
    (30, 4, 8, 4, 128, None),
    (777, 4, 8, 4, 64, [0, 100, 101, 401, 777]),
    (1, 8, 8, 8, 128, None),
    (32766, 8, 32, 8, 128, None),
])
def test_seq_to_head_reads_unpadded_source(case):
    # padding rows come out as zeros without a padded copy of the input: the
    # source tensor holds only the S valid rows
    for which, mode in (("q", 1), ("k", 1), ("v", 0)):
        _repack_case(*case, which, mode, unpadded=True)


@pytest.mark.parametrize("name", ["qwen8k", "long32k_pad", "thd64k"])
def test_seq_to_head_full_workloads(name):
    wl = WORKLOADS[name]
    cu = None
    if wl.thd:
        from ulysses_sequence_attention_usp_gb300.inputs import doc_lengths
        cu = list(cu_seqlens(doc_lengths(wl.S)))
    for which in ("q", "k"):
        _repack_case(wl.S, wl.P, wl.Hq, wl.Hkv, wl.D, cu, which, 1, base=wl.rope_base)


def test_seq_to_head_120k_yarn_sampled_rows():
    wl = WORKLOADS["sp8_120k"]
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, 1, 14999, 15000, wl.S - 1],
                                     rng.integers(0, wl.S, 3000)]))
    _repack_case(wl.S, wl.P, wl.Hq, wl.Hkv, wl.D, None, "q", 1, rows=rows, base=wl.rope_base,
                 f=wl.yarn_factor, L=wl.yarn_orig_ctx, rope_len=wl.rope_len)


def _rows_120k(S, seed):
    """Sampled rows of the 120K workload: shard edges, rows past the
    repack's grid-stride threshold (152*64 blocks x 8 rows = 77 824) and
    random rows."""
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 14999, 15000, 77823, 77824, 77825, S - 2, S - 1]
    return np.unique(np.concatenate([fixed, rng.integers(0, S, 3000),
                                     rng.integers(77824, S, 1000)]))


def test_seq_to_head_120k_yarn_k_sampled_rows():
    wl = WORKLOADS["sp8_120k"]
    _repack_case(wl.S, wl.P, wl.Hq, wl.Hkv, wl.D, None, "k", 1, rows=_rows_120k(wl.S, 1),
                 base=wl.rope_base, f=wl.yarn_factor, L=wl.yarn_orig_ctx, rope_len=wl.rope_len)


@pytest.mark.parametrize("which,mode", [("q", -1), ("k", -1), ("v", 0)])
def test_head_to_seq_120k_sampled_rows(which, mode):
    # the inverse all-to-all of the gradients at full size, in the launch
    # configuration of the benchmark (grid-stride loop beyond 77 824 rows)
    wl = WORKLOADS["sp8_120k"]
    H = wl.Hq if which == "q" else wl.Hkv
    S, P, D = wl.S, wl.P, wl.D
    d = _dims(S, P, wl.Hq, wl.Hkv, D)
    table = O.rope_table_f32(wl.rope_len, D, wl.rope_base, wl.yarn_factor, wl.yarn_orig_ctx)
    pos, _ = O.positions_docs(S, P)
    xh = normal_bf16((P, S, H // P, D), 15, "do")
    out = torch.empty((S, H, D), dtype=torch.bfloat16, device="cuda")
    B.usp_head_to_seq(d, to_dev(xh), H, torch.from_numpy(pos.astype(np.int32)).cuda(),
                      torch.from_numpy(table).cuda(), wl.rope_len, mode, out)
    torch.cuda.synchronize()
    rows = _rows_120k(S, 2)
    got = out[torch.from_numpy(rows).cuda()]
    want = np.ascontiguousarray(xh[:, rows].transpose(1, 0, 2, 3).reshape(len(rows), H, D))
    if mode != 0:
        want = O.rope_recipe_bf16(want, pos[rows], table, inverse=mode < 0)
    assert np.array_equal(to_bits(got), want)


@pytest.mark.parametrize("D,mode", [(128, -1), (128, 0), (64, -1), (64, 1)])
def test_head_to_seq_bit_exact(D, mode):
    S, P, H = 1000, 4, 8
    d = _dims(S, P, H, H, D)
    table = O.rope_table_f32(S, D, 1.0e6)
    pos, _ = O.positions_docs(S, P)
    xh = normal_bf16((P, S, H // P, D), 12, "do")
    out = torch.empty((S, H, D), dtype=torch.bfloat16, device="cuda")
    B.usp_head_to_seq(d, to_dev(xh), H, torch.from_numpy(pos.astype(np.int32)).cuda(),
                      torch.from_numpy(table).cuda(), S, mode, out)
    torch.cuda.synchronize()
    want = O.head_to_seq(xh)
    if mode != 0:
        want = O.rope_recipe_bf16(want, pos, table, inverse=mode < 0)
    assert np.array_equal(to_bits(out), want)


@pytest.mark.parametrize("D,mode", [(128, -1), (64, 0)])
def test_head_to_seq_odd_rows_few_heads(D, mode):
    S, P, H = 777, 1, 2            # two rows per warp, the last pair incomplete
    d = _dims(S, P, H, H, D)
    table = O.rope_table_f32(S, D, 1.0e4)
    pos, _ = O.positions_docs(S, P)
    xh = normal_bf16((P, S, H // P, D), 16, "do")
    out = torch.full((S, H, D), 3.0, dtype=torch.bfloat16, device="cuda")
    B.usp_head_to_seq(d, to_dev(xh), H, torch.from_numpy(pos.astype(np.int32)).cuda(),
                      torch.from_numpy(table).cuda(), S, mode, out)
    torch.cuda.synchronize()
    want = O.head_to_seq(xh)
    if mode != 0:
        want = O.rope_recipe_bf16(want, pos, table, inverse=mode < 0)
    assert np.array_equal(to_bits(out), want)


def test_roundtrip_is_identity():
    S, P, H, D = 4096, 8, 32, 128
    d = _dims(S, P, H, 8, D)
    x = to_dev(normal_bf16((S, H, D), 13, "q"))
    mid = torch.empty((P, S, H // P, D), dtype=torch.bfloat16, device="cuda")
    back = torch.empty_like(x)
    B.usp_seq_to_head_rope(d, x, H, None, None, 0, 0, mid)
    B.usp_head_to_seq(d, mid, H, None, None, 0, 0, back)
    torch.cuda.synchronize()
    assert torch.equal(x.view(torch.int16), back.view(torch.int16))


def test_position_outside_table_is_reported_not_read():
    S, P, H, D = 64, 2, 4, 64
    d = _dims(S, P, H, H, D)
    table = torch.from_numpy(O.rope_table_f32(S, D, 1.0e4)).cuda()
    pos = torch.arange(S, dtype=torch.int32, device="cuda")
    pos[5] = 10**6                       # a caller-made position past the table
    x = to_dev(normal_bf16((S, H, D), 14, "q"))
    out = torch.empty((P, S, H // P, D), dtype=torch.bfloat16, device="cuda")
    B.usp_seq_to_head_rope(d, x, H, pos, table, S, 1, out)
    with pytest.raises(B.UspError) as e:
        B.usp_device_status()
    assert e.value.status == 1
    assert not to_bits(out)[:, 5].any()
    B.usp_device_status()                # cleared after being reported
