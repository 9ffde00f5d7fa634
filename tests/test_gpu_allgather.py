"""GPU parity of context parallelism with a K/V all-gather
(basetenlabs/Megatron-LM PR #7 "GLM-5.2 131k context parallelism", Purpose:
KV all-gather in the forward, dKV reduce-scatter in the backward, contiguous
partition): the AllGatherCPAttention step against the oracle's per-rank
all-gather path, including fewer KV heads than ranks, documents, padding of
the last shard and bidirectional attention, and the full 120K workload on
sampled rows."""
import math

import numpy as np
import pytest

from oracle import usp_oracle as O
from ulysses_sequence_attention_usp_gb300.inputs import WORKLOADS, make_inputs
from ulysses_sequence_attention_usp_gb300.pipeline import AllGatherCPAttention

from gpu_util import (SampledOracle, check_grad, check_lse, check_o, lse_tol_end_to_end, to_dev,
                      to_f64)
from test_gpu_attention import _setup

pytestmark = pytest.mark.gpu

CASES = [  # (S, P, Hq, Hkv, D, doc lengths), causal
    ((200, 4, 4, 1, 64, None), True),                    # one KV head, four ranks
    ((777, 8, 8, 2, 128, [100, 1, 300, 376]), True),     # Hkv < P, documents
    ((777, 8, 8, 2, 128, [100, 1, 300, 376]), False),    # the same, bidirectional
    ((1000, 3, 6, 3, 64, None), True),                   # P does not divide S
    ((300, 2, 8, 8, 128, None), True),                   # MHA
    ((5, 4, 4, 1, 128, None), True),                     # fewer rows than one tile
]


@pytest.mark.parametrize("case,causal", CASES)
def test_allgather_step_vs_oracle(case, causal):
    wl, inp = _setup(case, seed=11)
    ag = AllGatherCPAttention(wl.S, wl.P, wl.Hq, wl.Hkv, wl.D, cu_seqlens=inp.cu,
                              rope_base=wl.rope_base, causal=causal)
    q, k, v, do = (to_dev(x) for x in (inp.q, inp.k, inp.v, inp.do))
    dq, dk, dv = ag.step(q, k, v, do)
    ag.check()
    f = O.bf16_to_f64
    cos, sin = O.rope_cos_sin(wl.S_pad, wl.D, wl.rope_base)
    scale = 1.0 / math.sqrt(wl.D)
    ref = O.allgather_cp(f(inp.q), f(inp.k), f(inp.v), f(inp.do), inp.cu, cos, sin, scale,
                         wl.P, causal)
    check_o(to_f64(ag.o), ref["o"])
    check_grad(to_f64(dq), ref["dq"], "dq")
    check_grad(to_f64(dk), ref["dk"], "dk")
    check_grad(to_f64(dv), ref["dv"], "dv")
    nq = np.linalg.norm(f(inp.q), axis=-1).max()
    nk = np.linalg.norm(f(inp.k), axis=-1).max()
    check_lse(ag.lse.cpu().numpy().astype(np.float64), ref["lse"],
              lse_tol_end_to_end(nq, nk, scale))
    # each rank's shard is a view of its rows
    S_loc = -(-wl.S // wl.P)
    for r in range(wl.P):
        assert ag.shard(ag.o, r).shape[0] == max(0, min(wl.S, (r + 1) * S_loc) - r * S_loc)


def _allgather_120k():
    wl = WORKLOADS["sp8_120k"]
    inp = make_inputs(wl, 0)
    orc = SampledOracle(inp.q, inp.k, inp.v, inp.do, inp.cu, wl)
    ag = AllGatherCPAttention(wl.S, wl.P, wl.Hq, wl.Hkv, wl.D, rope_base=wl.rope_base,
                              yarn_factor=wl.yarn_factor, yarn_orig_ctx=wl.yarn_orig_ctx,
                              rope_len=wl.rope_len, rope_table=orc.table())
    q, k, v, do = (to_dev(x) for x in (inp.q, inp.k, inp.v, inp.do))
    ag.step(q, k, v, do)
    ag.check()
    return wl, inp, ag, orc


def test_allgather_full_workload_sampled():
    wl, inp, ag, orc = _allgather_120k()
    rng = np.random.default_rng(7)
    S = wl.S
    S_loc = -(-S // wl.P)
    # the first and last row of every rank, and random rows
    edges = [x for r in range(wl.P) for x in (r * S_loc, min(S, (r + 1) * S_loc) - 1)]
    rows = np.unique(np.concatenate([edges, rng.integers(0, S, 8)]))
    for h in sorted({0, wl.Hq - 1, int(rng.integers(0, wl.Hq))}):
        r_o, _ = orc.fwd_rows(h, rows)
        check_o(to_f64(ag.o[rows, h]), r_o)
        check_grad(to_f64(ag.dq[rows, h]), orc.dq_rows(h, rows), "dq")
        check_lse(ag.lse[h, rows].cpu().numpy().astype(np.float64),
                  orc.lse_rows_recipe(h, rows))
    lo = S - 48
    for kh in sorted({0, wl.Hkv - 1}):
        r_dk, r_dv = orc.dkv_tail(kh, lo, S)
        check_grad(to_f64(ag.dk[lo:S, kh]), r_dk, "dk")
        check_grad(to_f64(ag.dv[lo:S, kh]), r_dv, "dv")


@pytest.mark.slow
def test_allgather_120k_first_keys():
    """dK/dV of keys 0..47, which all 120 000 query rows see (the longest
    key-stationary loop; the sum over every rank's query rows is what the
    reduce-scatter of dK/dV adds up)."""
    wl, inp, ag, orc = _allgather_120k()
    keys = np.arange(48)
    r_dk, r_dv = orc.dkv_keys(0, keys, np.arange(wl.S))
    check_grad(to_f64(ag.dk[:48, 0]), r_dk, "dk")
    check_grad(to_f64(ag.dv[:48, 0]), r_dv, "dv")
