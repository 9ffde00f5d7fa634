"""GPU parity of the attention kernels and the whole USP pipeline against
the fp64 oracle.

* kernel parity: the oracle rotates Q/K with the bf16 recipe and permutes
  them itself; those bits go to usp_attn_fwd/usp_attn_bwd, and the results
  are compared with fp64 attention of the same bf16 values;
* end-to-end parity: UlyssesAttention (pad -> all-to-all+RoPE -> attention
  -> all-to-all back, forward and backward) against the oracle's
  full-sequence fp64 computation with exact RoPE (the criterion of loss and
  gradient parity with full-sequence attention);
* full-size workloads, in the launch configuration the benchmark times,
  checked on sampled rows.
"""
import math

import numpy as np
import pytest
import torch

from oracle import usp_oracle as O
from ulysses_sequence_attention_usp_gb300 import binding as B
from ulysses_sequence_attention_usp_gb300.inputs import WORKLOADS, custom_workload, make_inputs
from ulysses_sequence_attention_usp_gb300.pipeline import UlyssesAttention

from gpu_util import (SampledOracle, check_grad, check_lse, check_o, check_sampled_full_size,
                      lse_tol_end_to_end, to_bits, to_dev, to_f64)

pytestmark = pytest.mark.gpu

SMALL = [  # S, P, Hq, Hkv, D, doc lengths (None = one sequence)
    (256, 2, 4, 2, 64, None),             # the tiny workload
    (1000, 2, 8, 2, 128, None),           # several tiles, ragged tail
    (777, 4, 8, 4, 64, [100, 1, 300, 376]),  # packed documents, a doc of length 1
    (130, 2, 2, 2, 128, [1, 129]),        # MHA (G = 1)
    (30, 4, 8, 4, 128, None),             # padded 30 -> 32
    (1, 8, 8, 8, 128, None),              # one token, fewer rows than ranks
    (600, 2, 16, 2, 128, [200, 400]),     # G = 8 as in the packed 64/8 workload
    (300, 2, 8, 2, 128, [100, 0, 150, 0, 50]),  # empty documents in cu_seqlens
    (512, 1, 4, 2, 64, [200, 312]),       # one rank (P = 1): no head split
    (390, 2, 6, 2, 64, [130, 260]),       # G = 3: one query head per forward CTA, 3 slots
]


def _setup(case, seed=0):
    S, P, Hq, Hkv, D, lens = case
    wl = custom_workload(S, P, Hq, Hkv, D, base=1.0e4, thd_lens=lens)
    inp = make_inputs(wl, seed, lens=lens)
    return wl, inp


def _kernel_inputs(wl, inp):
    """Oracle-made head-layout bf16 inputs (RoPE by the bf16 recipe)."""
    P = wl.P
    table = O.rope_table_f32(wl.S_pad, wl.D, wl.rope_base)
    pos, doc = O.positions_docs(wl.S, P, inp.cu)
    qh = O.seq_to_head(O.rope_recipe_bf16(O.shard_pad(inp.q, P), pos, table), P)
    kh = O.seq_to_head(O.rope_recipe_bf16(O.shard_pad(inp.k, P), pos, table), P)
    vh = O.seq_to_head(O.shard_pad(inp.v, P), P)
    doh = O.seq_to_head(O.shard_pad(inp.do, P), P)
    return qh, kh, vh, doh, doc


def _dims(wl, cu):
    cu_dev = None if cu is None else torch.from_numpy(cu.astype(np.int32)).cuda()
    return B.make_dims(wl.S, wl.P, wl.Hq, wl.Hkv, wl.D, cu_dev, cu)


@pytest.mark.parametrize("case", SMALL)
def test_attention_kernels_vs_fp64(case):
    wl, inp = _setup(case)
    qh, kh, vh, doh, doc = _kernel_inputs(wl, inp)
    d = _dims(wl, inp.cu)
    P, Sp, hq, hkv, D = wl.P, wl.S_pad, wl.Hq // wl.P, wl.Hkv // wl.P, wl.D
    tq, tk, tv, tdo = to_dev(qh), to_dev(kh), to_dev(vh), to_dev(doh)
    tdoc = torch.from_numpy(doc.astype(np.int32)).cuda()
    o = torch.full((P, Sp, hq, D), 9.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((P, hq, Sp), 9.0, dtype=torch.float32, device="cuda")
    B.usp_attn_fwd(d, tq, tk, tv, tdoc, o, lse)
    ws_n = B.usp_attn_bwd_workspace(d)
    ws = torch.empty(ws_n, dtype=torch.uint8, device="cuda")
    dq = torch.full_like(tq, 9.0)
    dk = torch.full_like(tk, 9.0)
    dv = torch.full_like(tv, 9.0)
    B.usp_attn_bwd(d, tq, tk, tv, o, lse, tdo, tdoc, dq, dk, dv, ws, ws_n)
    B.usp_device_status()
    scale = 1.0 / math.sqrt(D)
    for g in range(P):
        qf, kf, vf, dof = (O.bf16_to_f64(x[g]) for x in (qh, kh, vh, doh))
        o_ref, lse_ref = O.attention_fwd(qf, kf, vf, doc, scale)
        check_o(to_f64(o[g]), o_ref)
        check_lse(lse[g].cpu().numpy().astype(np.float64), lse_ref)
        dq_ref, dk_ref, dv_ref = O.attention_bwd(qf, kf, vf, dof, doc, scale)
        check_grad(to_f64(dq[g]), dq_ref, "dq")
        check_grad(to_f64(dk[g]), dk_ref, "dk")
        check_grad(to_f64(dv[g]), dv_ref, "dv")
        pad = doc < 0
        assert not to_f64(o[g])[pad].any() and not to_f64(dq[g])[pad].any()
        assert not to_f64(dk[g])[pad].any() and not to_f64(dv[g])[pad].any()


def _recipe_lse(wl, inp, table):
    """fp64 LSE of every head when attention is fed the bf16 rotated Q, K of
    the fp32 recipe with `table` (the GPU's actual attention inputs)."""
    pos, doc = O.positions_docs(wl.S, 1, inp.cu)
    qr = O.bf16_to_f64(O.rope_recipe_bf16(inp.q, pos, table))
    kr = O.bf16_to_f64(O.rope_recipe_bf16(inp.k, pos, table))
    _, lse = O.attention_fwd(qr, kr, O.bf16_to_f64(inp.v), doc, 1.0 / math.sqrt(wl.D))
    return lse


@pytest.mark.parametrize("case", SMALL)
def test_pipeline_vs_full_sequence(case):
    wl, inp = _setup(case, seed=1)
    table = O.rope_table_f32(wl.S_pad, wl.D, wl.rope_base)
    ua = UlyssesAttention(wl.S, wl.P, wl.Hq, wl.Hkv, wl.D, cu_seqlens=inp.cu,
                          rope_base=wl.rope_base, rope_table=table)
    q, k, v, do = (to_dev(x) for x in (inp.q, inp.k, inp.v, inp.do))
    dq, dk, dv = ua.step(q, k, v, do)
    ua.check()
    cos, sin = O.rope_cos_sin(wl.S_pad, wl.D, wl.rope_base)
    f = lambda b: O.bf16_to_f64(b)  # noqa: E731
    ref = O.full_sequence(f(inp.q), f(inp.k), f(inp.v), f(inp.do), inp.cu, cos, sin,
                          1.0 / math.sqrt(wl.D))
    S = wl.S
    check_o(to_f64(ua.o)[:S], ref["o"])
    check_grad(to_f64(dq)[:S], ref["dq"], "dq")
    check_grad(to_f64(dk)[:S], ref["dk"], "dk")
    check_grad(to_f64(dv)[:S], ref["dv"], "dv")
    # loss = sum(O * dO) over the valid rows, from the GPU's O (host arithmetic)
    loss = float((to_f64(ua.o)[:S] * f(inp.do)).sum())
    assert abs(loss - ref["loss"]) <= 1e-2 * float(np.abs(ref["o"] * f(inp.do)).sum())
    lse = ua.lse.cpu().numpy().astype(np.float64).reshape(wl.Hq, wl.S_pad)[:, :S]
    # against exact RoPE, LSE moves by the bf16 rounding of the rotated Q, K
    nq = np.linalg.norm(f(inp.q), axis=-1).max()     # rotation keeps norms
    nk = np.linalg.norm(f(inp.k), axis=-1).max()
    check_lse(lse, ref["lse"], lse_tol_end_to_end(nq, nk, 1.0 / math.sqrt(wl.D)))
    # against the recipe-rotated bf16 Q, K the GPU attends to: 1e-3
    check_lse(lse, _recipe_lse(wl, inp, table))
    # outputs past S (padding) are zero
    assert not to_f64(ua.o)[S:].any() and not to_f64(dq)[S:].any()


def test_attention_is_deterministic():
    wl, inp = _setup((1000, 2, 8, 2, 128, None), seed=2)
    ua = UlyssesAttention(wl.S, wl.P, wl.Hq, wl.Hkv, wl.D, rope_base=wl.rope_base)
    q, k, v = (to_dev(x) for x in (inp.q, inp.k, inp.v))
    a = ua.forward(q, k, v).clone()
    la = ua.lse.clone()
    b = ua.forward(q, k, v)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(la, ua.lse)


@pytest.mark.parametrize("case", [(1000, 2, 8, 2, 128, None), (777, 4, 8, 4, 64, [100, 1, 300, 376])])
def test_graph_replay_equals_eager_steps(case):
    """A step captured in a CUDA graph and replayed gives bitwise the eager
    step's outputs, also after the inputs' contents change (the graph reads
    the same buffers)."""
    wl, inp = _setup(case, seed=4)
    _, inp2 = _setup(case, seed=5)
    ua = UlyssesAttention(wl.S, wl.P, wl.Hq, wl.Hkv, wl.D, cu_seqlens=inp.cu,
                          rope_base=wl.rope_base)
    ins = [to_dev(x) for x in (inp.q, inp.k, inp.v, inp.do)]
    ins2 = [to_dev(x) for x in (inp2.q, inp2.k, inp2.v, inp2.do)]
    outs = lambda: [t.clone() for t in (ua.o, ua.lse, ua.dq, ua.dk, ua.dv)]  # noqa: E731
    eager = []
    for x in (ins, ins2):
        ua.step(*x)
        ua.check()
        eager.append(outs())
    graph = ua.capture_step(*ins)
    for x, ref in zip((ins, ins2), eager):
        for buf, val in zip(ins, x):
            buf.copy_(val)
        graph.replay()
        ua.check()
        for a, b in zip(outs(), ref):
            assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                               b.view(torch.int16) if b.dtype == torch.bfloat16 else b)


# --------------------------------------------------------------- full sizes

def _full_case(name):
    """The full-size workload through the pipeline, with the oracle's RoPE
    table (bitwise the library's up to rare one-ulp entries), so that the
    recipe-rotated Q, K the oracle makes are exactly the GPU's."""
    wl = WORKLOADS[name]
    inp = make_inputs(wl, 0)
    orc = SampledOracle(inp.q, inp.k, inp.v, inp.do, inp.cu, wl)
    ua = UlyssesAttention(wl.S, wl.P, wl.Hq, wl.Hkv, wl.D, cu_seqlens=inp.cu,
                          rope_base=wl.rope_base, yarn_factor=wl.yarn_factor,
                          yarn_orig_ctx=wl.yarn_orig_ctx, rope_len=wl.rope_len,
                          rope_table=orc.table())
    q, k, v, do = (to_dev(x) for x in (inp.q, inp.k, inp.v, inp.do))
    ua.step(q, k, v, do)
    ua.check()
    return wl, inp, ua, orc


@pytest.mark.parametrize("name", ["sp8_120k", "thd64k", "long32k_pad", "qwen8k"])
def test_full_workload_sampled(name):
    wl, inp, ua, orc = _full_case(name)
    rng = np.random.default_rng(5)
    S = wl.S
    rows = np.unique(np.concatenate([[0, 1, 127, 128, S // 2, S - 1], rng.integers(0, S, 10)]))
    o = ua.o[:S]
    lse = ua.lse.reshape(wl.Hq, wl.S_pad)
    dq = ua.dq[:S]
    heads = sorted({0, wl.Hq - 1, int(rng.integers(0, wl.Hq))})
    got_o, ref_o, got_l, ref_l, got_dq, ref_dq = [], [], [], [], [], []
    for h in heads:
        r_o, r_l = orc.fwd_rows(h, rows)
        got_o.append(to_f64(o[rows, h]))
        ref_o.append(r_o)
        got_l.append(lse[h, rows].cpu().numpy().astype(np.float64))
        ref_l.append(r_l)
        got_dq.append(to_f64(dq[rows, h]))
        ref_dq.append(orc.dq_rows(h, rows))
    check_o(np.concatenate(got_o), np.concatenate(ref_o))
    check_grad(np.concatenate(got_dq), np.concatenate(ref_dq), "dq")
    m = (wl.yarn_factor > 1) and (0.1 * math.log(wl.yarn_factor) + 1) or 1.0  # YaRN mscale
    nq = m * np.linalg.norm(O.bf16_to_f64(inp.q[rows]), axis=-1).max()
    nk = m * np.linalg.norm(O.bf16_to_f64(inp.k), axis=-1).max()
    check_lse(np.concatenate(got_l), np.concatenate(ref_l),
              lse_tol_end_to_end(nq, nk, 1.0 / math.sqrt(wl.D)))
    # 1e-3 against fp64 attention of the recipe-rotated bf16 Q, K
    check_lse(np.concatenate(got_l), np.concatenate([orc.lse_rows_recipe(h, rows)
                                                     for h in heads]))
    # dK/dV at the last rows of a document: only queries at or after them
    # see those keys, so the oracle needs just those query rows
    ends = [S] if inp.cu is None else [int(inp.cu[-1]), int(inp.cu[3])]
    for end in ends:
        lo = end - 48
        for kh in sorted({0, wl.Hkv - 1}):
            r_dk, r_dv = orc.dkv_tail(kh, lo, end)
            check_grad(to_f64(ua.dk[lo:end, kh]), r_dk, "dk")
            check_grad(to_f64(ua.dv[lo:end, kh]), r_dv, "dv")


def test_padded_matches_unpadded_long():
    # S = 32766 pads to 32768 over P = 8; over P = 2 it needs no padding.
    wl8 = WORKLOADS["long32k_pad"]
    inp = make_inputs(wl8, 0, with_do=True)
    q, k, v, do = (to_dev(x) for x in (inp.q, inp.k, inp.v, inp.do))
    outs = []
    for P in (8, 2):
        ua = UlyssesAttention(wl8.S, P, wl8.Hq, wl8.Hkv, wl8.D, rope_base=wl8.rope_base,
                              rope_len=32768)
        dq, dk, dv = ua.step(q, k, v, do)
        ua.check()
        outs.append([t[:wl8.S].clone() for t in (ua.o, dq, dk, dv)])
    for a, b in zip(*outs):
        fa, fb = a.float(), b.float()
        assert (fa - fb).abs().max().item() <= 2e-2 * max(1.0, fb.abs().max().item())


def _first_keys_case(name):
    """(KV heads, first key, end of the longest document) of a workload."""
    wl = WORKLOADS[name]
    if wl.thd:
        from ulysses_sequence_attention_usp_gb300.inputs import cu_seqlens, doc_lengths
        cu = cu_seqlens(doc_lengths(wl.S))
        d = int(np.argmax(np.diff(cu)))
        return wl, [0, wl.Hkv - 1], int(cu[d]), int(cu[d + 1])
    return wl, ([0] if wl.S > 100000 else [0, wl.Hkv - 1]), 0, wl.S


@pytest.mark.parametrize("name", ["long32k_pad", "thd64k",
                                  pytest.param("sp8_120k", marks=pytest.mark.slow)])
def test_full_workload_first_keys(name):
    """dK/dV of the first 48 keys of the longest document: every later query
    row of the document sees them, so the key-stationary pass runs its
    longest loop there (at 120K, 938 query tiles x 4 query heads accumulated
    in TMEM).  The oracle needs each of those rows' LSE and delta, i.e. the
    whole causal forward of the group's query heads, evaluated over row
    chunks in worker processes."""
    wl, kvs, a, e = _first_keys_case(name)
    _, inp, ua, orc = _full_case(name)
    keys = np.arange(a, a + 48)
    for kh in kvs:
        r_dk, r_dv = orc.dkv_keys(kh, keys, np.arange(a, e))
        check_grad(to_f64(ua.dk[a:a + 48, kh]), r_dk, "dk")
        check_grad(to_f64(ua.dv[a:a + 48, kh]), r_dv, "dv")


def test_d64_long_packed_sampled():
    """Head dimension 64 at 16K packed tokens (many tiles, long key-stationary
    loops, documents straddling shards), sampled against the oracle: the
    D = 64 kernels otherwise run only at small sizes."""
    lens = [5000, 129, 1, 7000, 4254]
    wl = custom_workload(16384, 4, 16, 4, 64, base=1.0e4, thd_lens=lens)
    inp = make_inputs(wl, 3, lens=lens)
    orc = SampledOracle(inp.q, inp.k, inp.v, inp.do, inp.cu, wl)
    ua = UlyssesAttention(wl.S, wl.P, wl.Hq, wl.Hkv, wl.D, cu_seqlens=inp.cu,
                          rope_base=wl.rope_base, rope_table=orc.table())
    q, k, v, do = (to_dev(x) for x in (inp.q, inp.k, inp.v, inp.do))
    dq, dk, dv = ua.step(q, k, v, do)
    ua.check()
    check_sampled_full_size(wl, inp, orc, ua.o, ua.lse.reshape(wl.Hq, wl.S_pad), dq, dk, dv,
                            seed=11)
    # dK/dV of the first 48 keys of the longest document (7000 rows)
    a, e = int(inp.cu[3]), int(inp.cu[4])
    keys = np.arange(a, a + 48)
    for kh in (0, wl.Hkv - 1):
        r_dk, r_dv = orc.dkv_keys(kh, keys, np.arange(a, e))
        check_grad(to_f64(dk[a:a + 48, kh]), r_dk, "dk")
        check_grad(to_f64(dv[a:a + 48, kh]), r_dv, "dv")
