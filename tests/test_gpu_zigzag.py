"""GPU parity of the zigzag shard layout (Megatron-LM PR #7 "GLM-5.2 131k
context parallelism", closing comment; reading: rank r holds chunks r and
2P-1-r of 2P): pad/shard, the all-to-all with RoPE both ways bit-exact
against the oracle, and the whole pipeline against full-sequence attention.
"""
import math

import numpy as np
import pytest
import torch

from oracle import usp_oracle as O
from ulysses_sequence_attention_usp_gb300 import binding as B
from ulysses_sequence_attention_usp_gb300.inputs import (WORKLOADS, cu_seqlens, make_inputs,
                                                        normal_bf16)
from ulysses_sequence_attention_usp_gb300.pipeline import UlyssesAttention

from gpu_util import (SampledOracle, check_grad, check_o, check_sampled_full_size, to_bits,
                      to_dev, to_f64)
from test_gpu_attention import _setup

pytestmark = pytest.mark.gpu

CASES = [  # S, P, H, D, doc lengths
    (8, 2, 4, 64, None),
    (1000, 4, 8, 128, None),
    (777, 4, 8, 64, [100, 1, 300, 376]),
    (30, 4, 8, 128, None),
    (1, 8, 8, 128, None),
    (65536, 8, 8, 128, [4656, 1304, 590, 542, 8578, 12109, 4191, 6416, 3369, 13083, 8655,
                        517, 1526]),
]


def _dims(S, P, H, D, lens):
    cu = None if lens is None else np.asarray(cu_seqlens(lens), np.int32)
    cu_dev = None if cu is None else torch.from_numpy(cu).cuda()
    return B.make_dims(S, P, H, H, D, cu_dev, cu, zigzag=True), cu


@pytest.mark.parametrize("S,P,H,D,lens", CASES)
def test_zigzag_pad_shard_and_repack_bit_exact(S, P, H, D, lens):
    d, cu = _dims(S, P, H, D, lens)
    S_pad = O.zigzag_padded_len(S, P)
    x = normal_bf16((S, H, D), 21, "q")
    xs = torch.full((S_pad, H, D), 7.0, dtype=torch.bfloat16, device="cuda")
    pos = torch.full((S_pad,), -5, dtype=torch.int32, device="cuda")
    doc = torch.full((S_pad,), -5, dtype=torch.int32, device="cuda")
    B.usp_pad_shard(d, to_dev(x), H, xs, pos, doc)
    torch.cuda.synchronize()
    want_pos, want_doc = O.positions_docs(S, P, cu, S_pad=S_pad)
    assert np.array_equal(pos.cpu().numpy(), want_pos)
    assert np.array_equal(doc.cpu().numpy(), want_doc)
    x_seq = O.shard_pad_zigzag(x, P)
    assert np.array_equal(to_bits(xs), x_seq)
    # seq -> head with RoPE at the global positions, and back with the inverse
    table = O.rope_table_f32(S_pad, D, 1.0e4)
    tpos, ttab = pos, torch.from_numpy(table).cuda()
    head = torch.empty((P, S_pad, H // P, D), dtype=torch.bfloat16, device="cuda")
    B.usp_seq_to_head_rope(d, xs, H, tpos, ttab, S_pad, 1, head)
    order = O.zigzag_order(S_pad, P)
    x_glob = x_seq[np.argsort(order)]
    want = O.seq_to_head(O.rope_recipe_bf16(x_glob, want_pos, table), P)
    assert np.array_equal(to_bits(head), want)
    back = torch.empty_like(xs)
    B.usp_head_to_seq(d, head, H, tpos, ttab, S_pad, -1, back)
    torch.cuda.synchronize()
    want_back = O.rope_recipe_bf16(O.head_to_seq(want), want_pos, table, inverse=True)[order]
    assert np.array_equal(to_bits(back), want_back)
    B.usp_device_status()


@pytest.mark.parametrize("case,causal", [((1000, 2, 8, 2, 128, None), True),
                                         ((777, 4, 8, 4, 64, [100, 1, 300, 376]), True),
                                         ((777, 4, 8, 4, 64, [100, 1, 300, 376]), False),
                                         ((30, 4, 8, 4, 128, None), True)])
def test_zigzag_pipeline_vs_full_sequence(case, causal):
    wl, inp = _setup(case, seed=5)
    ua = UlyssesAttention(wl.S, wl.P, wl.Hq, wl.Hkv, wl.D, cu_seqlens=inp.cu,
                          rope_base=wl.rope_base, causal=causal, zigzag=True)
    q, k, v, do = (to_dev(x) for x in (inp.q, inp.k, inp.v, inp.do))
    dq, dk, dv = ua.step(q, k, v, do)
    ua.check()
    S, S_pad = wl.S, ua.S_pad
    inv = np.argsort(O.zigzag_order(S_pad, wl.P))       # global row t -> buffer row
    glob = lambda t: to_f64(t)[inv][:S]                  # noqa: E731
    cos, sin = O.rope_cos_sin(S_pad, wl.D, wl.rope_base)
    f = O.bf16_to_f64
    ref = O.full_sequence(f(inp.q), f(inp.k), f(inp.v), f(inp.do), inp.cu, cos, sin,
                          1.0 / math.sqrt(wl.D), causal=causal)
    check_o(glob(ua.o), ref["o"])
    check_grad(glob(dq), ref["dq"], "dq")
    check_grad(glob(dk), ref["dk"], "dk")
    check_grad(glob(dv), ref["dv"], "dv")
    pad = inv[S:]
    assert not to_f64(ua.o)[pad].any() and not to_f64(dq)[pad].any()


def test_zigzag_120k_sampled():
    """The 120K SP8 workload in the zigzag shard layout, as `bench.py
    --zigzag` runs it: sampled rows of O, LSE and dQ and the last 48 keys'
    dK/dV against the oracle, read through the zigzag row map."""
    wl = WORKLOADS["sp8_120k"]
    inp = make_inputs(wl, 0)
    orc = SampledOracle(inp.q, inp.k, inp.v, inp.do, inp.cu, wl)
    ua = UlyssesAttention(wl.S, wl.P, wl.Hq, wl.Hkv, wl.D, cu_seqlens=inp.cu,
                          rope_base=wl.rope_base, yarn_factor=wl.yarn_factor,
                          yarn_orig_ctx=wl.yarn_orig_ctx, rope_len=wl.rope_len,
                          rope_table=orc.table(), zigzag=True)
    q, k, v, do = (to_dev(x) for x in (inp.q, inp.k, inp.v, inp.do))
    dq, dk, dv = ua.step(q, k, v, do)
    ua.check()
    inv = np.argsort(O.zigzag_order(ua.S_pad, wl.P))    # global row t -> buffer row
    check_sampled_full_size(wl, inp, orc, ua.o, ua.lse.reshape(wl.Hq, ua.S_pad), dq, dk, dv,
                            seed=8, buf_of=inv)
