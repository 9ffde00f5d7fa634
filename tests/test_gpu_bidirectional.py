"""GPU parity of the bidirectional variant (causal = 0: attention within each
document over all of its keys, padding never a key; zhtmike/verl PR #45
"[trainer] feat: support sequence parallel", What does this PR do) against
the fp64 oracle: the attention kernels on oracle-made inputs, the whole
pipeline against full-sequence attention, and a full-size packed workload on
sampled rows."""
import math

import numpy as np
import pytest
import torch

from oracle import usp_oracle as O
from ulysses_sequence_attention_usp_gb300 import binding as B
from ulysses_sequence_attention_usp_gb300.inputs import WORKLOADS, make_inputs
from ulysses_sequence_attention_usp_gb300.pipeline import UlyssesAttention

from gpu_util import (SampledOracle, check_grad, check_lse, check_o, lse_tol_end_to_end,
                      to_dev, to_f64)
from test_gpu_attention import SMALL, _kernel_inputs, _setup

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", SMALL)
def test_bidirectional_kernels_vs_fp64(case):
    wl, inp = _setup(case, seed=3)
    qh, kh, vh, doh, doc = _kernel_inputs(wl, inp)
    cu_dev = None if inp.cu is None else torch.from_numpy(inp.cu.astype(np.int32)).cuda()
    d = B.make_dims(wl.S, wl.P, wl.Hq, wl.Hkv, wl.D, cu_dev, inp.cu, causal=False)
    P, Sp, hq, D = wl.P, wl.S_pad, wl.Hq // wl.P, wl.D
    tq, tk, tv, tdo = to_dev(qh), to_dev(kh), to_dev(vh), to_dev(doh)
    tdoc = torch.from_numpy(doc.astype(np.int32)).cuda()
    o = torch.full((P, Sp, hq, D), 9.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((P, hq, Sp), 9.0, dtype=torch.float32, device="cuda")
    B.usp_attn_fwd(d, tq, tk, tv, tdoc, o, lse)
    ws_n = B.usp_attn_bwd_workspace(d)
    ws = torch.empty(ws_n, dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.full_like(tq, 9.0), torch.full_like(tk, 9.0), torch.full_like(tv, 9.0)
    B.usp_attn_bwd(d, tq, tk, tv, o, lse, tdo, tdoc, dq, dk, dv, ws, ws_n)
    B.usp_device_status()
    scale = 1.0 / math.sqrt(D)
    for g in range(P):
        qf, kf, vf, dof = (O.bf16_to_f64(x[g]) for x in (qh, kh, vh, doh))
        o_ref, lse_ref = O.attention_fwd(qf, kf, vf, doc, scale, causal=False)
        check_o(to_f64(o[g]), o_ref)
        check_lse(lse[g].cpu().numpy().astype(np.float64), lse_ref)
        dq_ref, dk_ref, dv_ref = O.attention_bwd(qf, kf, vf, dof, doc, scale, causal=False)
        check_grad(to_f64(dq[g]), dq_ref, "dq")
        check_grad(to_f64(dk[g]), dk_ref, "dk")
        check_grad(to_f64(dv[g]), dv_ref, "dv")
        pad = doc < 0
        assert not to_f64(o[g])[pad].any() and not to_f64(dq[g])[pad].any()
        assert not to_f64(dk[g])[pad].any() and not to_f64(dv[g])[pad].any()


@pytest.mark.parametrize("case", [SMALL[1], SMALL[2], SMALL[4], SMALL[6]])
def test_bidirectional_pipeline_vs_full_sequence(case):
    wl, inp = _setup(case, seed=4)
    ua = UlyssesAttention(wl.S, wl.P, wl.Hq, wl.Hkv, wl.D, cu_seqlens=inp.cu,
                          rope_base=wl.rope_base, causal=False)
    q, k, v, do = (to_dev(x) for x in (inp.q, inp.k, inp.v, inp.do))
    dq, dk, dv = ua.step(q, k, v, do)
    ua.check()
    cos, sin = O.rope_cos_sin(wl.S_pad, wl.D, wl.rope_base)
    f = O.bf16_to_f64
    ref = O.full_sequence(f(inp.q), f(inp.k), f(inp.v), f(inp.do), inp.cu, cos, sin,
                          1.0 / math.sqrt(wl.D), causal=False)
    S = wl.S
    check_o(to_f64(ua.o)[:S], ref["o"])
    check_grad(to_f64(dq)[:S], ref["dq"], "dq")
    check_grad(to_f64(dk)[:S], ref["dk"], "dk")
    check_grad(to_f64(dv)[:S], ref["dv"], "dv")
    lse = ua.lse.cpu().numpy().astype(np.float64).reshape(wl.Hq, wl.S_pad)[:, :S]
    nq = np.linalg.norm(f(inp.q), axis=-1).max()
    nk = np.linalg.norm(f(inp.k), axis=-1).max()
    check_lse(lse, ref["lse"], lse_tol_end_to_end(nq, nk, 1.0 / math.sqrt(wl.D)))
    assert not to_f64(ua.o)[S:].any() and not to_f64(dq)[S:].any()


def test_bidirectional_full_size_packed_sampled():
    wl = WORKLOADS["thd64k"]
    inp = make_inputs(wl, 0)
    orc = SampledOracle(inp.q, inp.k, inp.v, inp.do, inp.cu, wl, causal=False)
    ua = UlyssesAttention(wl.S, wl.P, wl.Hq, wl.Hkv, wl.D, cu_seqlens=inp.cu,
                          rope_base=wl.rope_base, causal=False, rope_table=orc.table())
    q, k, v, do = (to_dev(x) for x in (inp.q, inp.k, inp.v, inp.do))
    ua.step(q, k, v, do)
    ua.check()
    rng = np.random.default_rng(6)
    S = wl.S
    rows = np.unique(np.concatenate([[0, 1, 127, 128, S // 2, S - 1], rng.integers(0, S, 10)]))
    lse = ua.lse.reshape(wl.Hq, wl.S_pad)
    got_o, ref_o, got_l, ref_l, got_dq, ref_dq = [], [], [], [], [], []
    heads = sorted({0, wl.Hq - 1, int(rng.integers(0, wl.Hq))})
    for h in heads:
        r_o, r_l = orc.fwd_rows(h, rows)
        got_o.append(to_f64(ua.o[rows, h]))
        ref_o.append(r_o)
        got_l.append(lse[h, rows].cpu().numpy().astype(np.float64))
        ref_l.append(r_l)
        got_dq.append(to_f64(ua.dq[rows, h]))
        ref_dq.append(orc.dq_rows(h, rows))
    check_o(np.concatenate(got_o), np.concatenate(ref_o))
    check_grad(np.concatenate(got_dq), np.concatenate(ref_dq), "dq")
    nq = np.linalg.norm(O.bf16_to_f64(inp.q[rows]), axis=-1).max()
    nk = np.linalg.norm(O.bf16_to_f64(inp.k), axis=-1).max()
    check_lse(np.concatenate(got_l), np.concatenate(ref_l),
              lse_tol_end_to_end(nq, nk, 1.0 / math.sqrt(wl.D)))
    # 1e-3 against fp64 attention of the recipe-rotated bf16 Q, K
    check_lse(np.concatenate(got_l), np.concatenate([orc.lse_rows_recipe(h, rows)
                                                     for h in heads]))
    # dK/dV of a whole short document: every query of that document sees it
    a, b = int(inp.cu[3]), int(inp.cu[4])
    for kh in sorted({0, wl.Hkv - 1}):
        r_dk, r_dv = orc.dkv_tail(kh, a, b, q_lo=a)
        check_grad(to_f64(ua.dk[a:b, kh]), r_dk, "dk")
        check_grad(to_f64(ua.dv[a:b, kh]), r_dv, "dv")
    # dK/dV of the first 48 keys of the longest document (13 083 rows): every
    # query row of the document sees them, the longest key-stationary loop
    d = int(np.argmax(np.diff(inp.cu)))
    a, b = int(inp.cu[d]), int(inp.cu[d + 1])
    keys = np.arange(a, a + 48)
    for kh in sorted({0, wl.Hkv - 1}):
        r_dk, r_dv = orc.dkv_keys(kh, keys, np.arange(a, b))
        check_grad(to_f64(ua.dk[a:a + 48, kh]), r_dk, "dk")
        check_grad(to_f64(ua.dv[a:a + 48, kh]), r_dv, "dv")


def test_bidirectional_120k_sampled():
    """The 120K SP8 workload (YaRN to 131072) in bidirectional mode, as
    `bench.py --bidirectional` runs it: O, LSE and dQ on sampled rows of
    three heads.  Every row sees all 120 000 keys, so each sampled row's
    oracle values are one full row of fp64 attention."""
    wl = WORKLOADS["sp8_120k"]
    inp = make_inputs(wl, 0)
    orc = SampledOracle(inp.q, inp.k, inp.v, inp.do, inp.cu, wl, causal=False)
    ua = UlyssesAttention(wl.S, wl.P, wl.Hq, wl.Hkv, wl.D, cu_seqlens=inp.cu,
                          rope_base=wl.rope_base, yarn_factor=wl.yarn_factor,
                          yarn_orig_ctx=wl.yarn_orig_ctx, rope_len=wl.rope_len,
                          causal=False, rope_table=orc.table())
    q, k, v, do = (to_dev(x) for x in (inp.q, inp.k, inp.v, inp.do))
    ua.step(q, k, v, do)
    ua.check()
    rng = np.random.default_rng(7)
    S = wl.S
    rows = np.unique(np.concatenate([[0, 127, 128, 77824, S - 1], rng.integers(0, S, 6)]))
    lse = ua.lse.reshape(wl.Hq, wl.S_pad)
    heads = sorted({0, wl.Hq - 1, int(rng.integers(0, wl.Hq))})
    got_o, ref_o, got_l, ref_l, got_dq, ref_dq = [], [], [], [], [], []
    for h in heads:
        r_o, r_l = orc.fwd_rows(h, rows)
        got_o.append(to_f64(ua.o[rows, h]))
        ref_o.append(r_o)
        got_l.append(lse[h, rows].cpu().numpy().astype(np.float64))
        ref_l.append(r_l)
        got_dq.append(to_f64(ua.dq[rows, h]))
        ref_dq.append(orc.dq_rows(h, rows))
    check_o(np.concatenate(got_o), np.concatenate(ref_o))
    check_grad(np.concatenate(got_dq), np.concatenate(ref_dq), "dq")
    # 1e-3 against fp64 attention of the recipe-rotated bf16 Q, K
    check_lse(np.concatenate(got_l), np.concatenate([orc.lse_rows_recipe(h, rows)
                                                     for h in heads]))
