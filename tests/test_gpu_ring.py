"""GPU parity of ring attention (SpecForge PR #728 / verl PR #45 Ulysses x
Ring mesh): the forward over a key window (one ring step) against the
oracle's windowed attention, the log-sum-exp merge kernel against the
oracle's merge, and the whole pipeline with R ring steps against
full-sequence attention."""
import math

import numpy as np
import pytest
import torch

from oracle import usp_oracle as O
from ulysses_sequence_attention_usp_gb300 import binding as B
from ulysses_sequence_attention_usp_gb300.inputs import WORKLOADS, make_inputs
from ulysses_sequence_attention_usp_gb300.pipeline import UlyssesAttention

from gpu_util import (SampledOracle, check_grad, check_lse, check_o, check_sampled_full_size,
                      lse_tol_end_to_end, to_dev, to_f64)
from test_gpu_attention import _kernel_inputs, _setup

pytestmark = pytest.mark.gpu

WINDOWS = [(0, 1000), (0, 128), (100, 357), (600, 1000), (1000, 1000), (999, 1000), (0, 0)]


@pytest.mark.parametrize("causal", [True, False])
def test_window_forward_vs_fp64(causal):
    case = (1000, 2, 8, 2, 128, [300, 1, 450, 249])
    wl, inp = _setup(case, seed=7)
    qh, kh, vh, _, doc = _kernel_inputs(wl, inp)
    cu_dev = torch.from_numpy(inp.cu.astype(np.int32)).cuda()
    d = B.make_dims(wl.S, wl.P, wl.Hq, wl.Hkv, wl.D, cu_dev, inp.cu, causal=causal)
    P, Sp, hq, D = wl.P, wl.S_pad, wl.Hq // wl.P, wl.D
    tq, tk, tv = to_dev(qh), to_dev(kh), to_dev(vh)
    tdoc = torch.from_numpy(doc.astype(np.int32)).cuda()
    scale = 1.0 / math.sqrt(D)
    for lo, hi in WINDOWS:
        o = torch.full((P, Sp, hq, D), 9.0, dtype=torch.bfloat16, device="cuda")
        lse = torch.full((P, hq, Sp), 9.0, dtype=torch.float32, device="cuda")
        B.usp_attn_fwd_window(d, tq, tk, tv, tdoc, lo, hi, o, lse)
        B.usp_device_status()
        for g in range(P):
            qf, kf, vf = (O.bf16_to_f64(x[g]) for x in (qh, kh, vh))
            o_ref, lse_ref = O.attention_window(qf, kf, vf, doc, scale, lo, hi, causal)
            check_o(to_f64(o[g]), o_ref)
            got = lse[g].cpu().numpy().astype(np.float64)
            fin = np.isfinite(lse_ref)
            assert np.array_equal(np.isfinite(got), fin), (lo, hi)
            if fin.any():
                check_lse(got[fin], lse_ref[fin])


def test_merge_kernel_vs_fp64():
    S, P, Hq, D = 300, 2, 4, 128
    d = B.make_dims(S, P, Hq, Hq, D)
    hq = Hq // P
    rng = np.random.default_rng(8)
    parts = []
    for i in range(3):
        o = rng.standard_normal((P, S, hq, D)).astype(np.float32)
        lse = (rng.standard_normal((P, hq, S)) * 3).astype(np.float32)
        lse[rng.random((P, hq, S)) < 0.2] = -np.inf       # rows with no key in this part
        o[np.transpose(np.isneginf(lse), (0, 2, 1))] = 0.0
        parts.append((torch.from_numpy(o).to(torch.bfloat16), torch.from_numpy(lse)))
    lse_all = np.stack([p[1].numpy() for p in parts])
    lse_all[0, :, :, :5] = -np.inf                        # rows with no key at all
    lse_all[1, :, :, :5] = -np.inf
    lse_all[2, :, :, :5] = -np.inf
    o_acc = torch.empty((P, S, hq, D), dtype=torch.float32, device="cuda")
    lse_acc = torch.empty((P, hq, S), dtype=torch.float32, device="cuda")
    o_out = torch.empty((P, S, hq, D), dtype=torch.bfloat16, device="cuda")
    ref_o, ref_l = None, None
    for i, (o_p, _) in enumerate(parts):
        l_p = torch.from_numpy(lse_all[i].astype(np.float32))
        B.usp_lse_merge(d, o_acc, lse_acc, o_p.cuda(), l_p.cuda(), i == 0,
                        o_out if i == 2 else None)
        of = o_p.float().numpy().astype(np.float64)
        lf = lse_all[i].astype(np.float64)
        # the oracle's merge works on [T][H][D] / [H][T]; map each group
        if ref_o is None:
            ref_o, ref_l = of, lf
        else:
            mo, ml = [], []
            for g in range(P):
                a, b = O.lse_merge(ref_o[g], ref_l[g], of[g], lf[g])
                mo.append(a)
                ml.append(b)
            ref_o, ref_l = np.stack(mo), np.stack(ml)
    torch.cuda.synchronize()
    got_o = o_acc.cpu().numpy().astype(np.float64)
    got_l = lse_acc.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isfinite(got_l), np.isfinite(ref_l))
    fin = np.isfinite(ref_l)
    assert np.abs(got_l[fin] - ref_l[fin]).max() <= 1e-5 * max(1.0, np.abs(ref_l[fin]).max())
    assert np.abs(got_o - ref_o).max() <= 1e-5 * max(1.0, np.abs(ref_o).max())
    assert not got_o[:, :5].any()
    out = o_out.float().cpu().numpy().astype(np.float64)
    assert np.abs(out - ref_o).max() <= 2.0 ** -8 * max(1.0, np.abs(ref_o).max())


@pytest.mark.parametrize("case,R,causal", [((1000, 2, 8, 2, 128, None), 2, True),
                                           ((1000, 2, 8, 2, 128, None), 3, False),
                                           ((777, 4, 8, 4, 64, [100, 1, 300, 376]), 4, True),
                                           ((777, 4, 8, 4, 64, [100, 1, 300, 376]), 5, False)])
def test_ring_pipeline_vs_full_sequence(case, R, causal):
    wl, inp = _setup(case, seed=9)
    ua = UlyssesAttention(wl.S, wl.P, wl.Hq, wl.Hkv, wl.D, cu_seqlens=inp.cu,
                          rope_base=wl.rope_base, causal=causal, ring=R)
    q, k, v, do = (to_dev(x) for x in (inp.q, inp.k, inp.v, inp.do))
    dq, dk, dv = ua.step(q, k, v, do)
    ua.check()
    cos, sin = O.rope_cos_sin(wl.S_pad, wl.D, wl.rope_base)
    f = O.bf16_to_f64
    ref = O.full_sequence(f(inp.q), f(inp.k), f(inp.v), f(inp.do), inp.cu, cos, sin,
                          1.0 / math.sqrt(wl.D), causal=causal)
    S = wl.S
    check_o(to_f64(ua.o)[:S], ref["o"])
    check_grad(to_f64(dq)[:S], ref["dq"], "dq")
    check_grad(to_f64(dk)[:S], ref["dk"], "dk")
    check_grad(to_f64(dv)[:S], ref["dv"], "dv")
    lse = ua.lse.cpu().numpy().astype(np.float64).reshape(wl.Hq, wl.S_pad)[:, :S]
    nq = np.linalg.norm(f(inp.q), axis=-1).max()
    nk = np.linalg.norm(f(inp.k), axis=-1).max()
    check_lse(lse, ref["lse"], lse_tol_end_to_end(nq, nk, 1.0 / math.sqrt(wl.D)))


def test_ring_120k_sampled():
    """The 120K SP8 workload with four ring steps, as `bench.py --ring 4`
    runs it: sampled rows of O, LSE and dQ and the last 48 keys' dK/dV
    against the oracle (the merged O and LSE feed the backward)."""
    wl = WORKLOADS["sp8_120k"]
    inp = make_inputs(wl, 0)
    orc = SampledOracle(inp.q, inp.k, inp.v, inp.do, inp.cu, wl)
    ua = UlyssesAttention(wl.S, wl.P, wl.Hq, wl.Hkv, wl.D, cu_seqlens=inp.cu,
                          rope_base=wl.rope_base, yarn_factor=wl.yarn_factor,
                          yarn_orig_ctx=wl.yarn_orig_ctx, rope_len=wl.rope_len,
                          rope_table=orc.table(), ring=4)
    q, k, v, do = (to_dev(x) for x in (inp.q, inp.k, inp.v, inp.do))
    dq, dk, dv = ua.step(q, k, v, do)
    ua.check()
    check_sampled_full_size(wl, inp, orc, ua.o, ua.lse.reshape(wl.Hq, wl.S_pad), dq, dk, dv,
                            seed=9)
