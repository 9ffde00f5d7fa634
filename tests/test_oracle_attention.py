"""Pins for the oracle's attention forward/backward and the two pipelines.

References used (none of them is the oracle itself): torch's
scaled_dot_product_attention and autograd in fp64 on the CPU, a pure-Python
brute-force loop, closed forms for special inputs, central finite
differences, and invariants of softmax."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import usp_oracle as O


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _sdpa(q, k, v, causal=True):
    # q [T,Hq,D], k/v [T,Hkv,D] fp64 -> O [T,Hq,D]
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]
    tk = torch.from_numpy(k).permute(1, 0, 2)[None]
    tv = torch.from_numpy(v).permute(1, 0, 2)[None]
    o = F.scaled_dot_product_attention(tq, tk, tv, is_causal=causal,
                                       enable_gqa=q.shape[1] != k.shape[1])
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("T,Hq,Hkv,D", [(33, 4, 2, 8), (64, 8, 8, 16), (17, 6, 2, 4)])
def test_fwd_matches_torch_sdpa_gqa(T, Hq, Hkv, D):
    q, k, v = _rand((T, Hq, D), 1), _rand((T, Hkv, D), 2), _rand((T, Hkv, D), 3)
    doc = np.zeros(T, np.int64)
    o, lse = O.attention_fwd(q, k, v, doc, 1 / math.sqrt(D))
    assert np.allclose(o, _sdpa(q, k, v), atol=1e-12, rtol=0)
    # LSE: recompute the softmax denominator from SDPA on V = e_j one-hot is
    # not available, so pin it through the identity O(V=1) = 1 and the K=0
    # closed form below; here check it is finite and >= the row's own score.
    G = Hq // Hkv
    for h in range(Hq):
        own = (q[:, h] * k[:, h // G]).sum(-1) / math.sqrt(D)
        assert np.all(lse[h] >= own - 1e-12)


def test_fwd_thd_is_concatenation_of_documents():
    lens = [5, 1, 12, 7]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, Hq, Hkv, D = int(cu[-1]), 4, 2, 8
    q, k, v = _rand((T, Hq, D), 4), _rand((T, Hkv, D), 5), _rand((T, Hkv, D), 6)
    _, doc = O.positions_docs(T, 1, cu)
    o, _ = O.attention_fwd(q, k, v, doc, 1 / math.sqrt(D))
    for a, b in zip(cu[:-1], cu[1:]):
        assert np.allclose(o[a:b], _sdpa(q[a:b], k[a:b], v[a:b]), atol=1e-12, rtol=0)


def test_fwd_closed_forms():
    lens = [6, 3, 9]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, Hq, Hkv, D = int(cu[-1]), 2, 1, 4
    q, v = _rand((T, Hq, D), 7), _rand((T, Hkv, D), 8)
    _, doc = O.positions_docs(T, 1, cu)
    # K = 0: uniform weights -> prefix mean of V inside the document, and
    # LSE = ln(number of visible keys)
    o, lse = O.attention_fwd(q, np.zeros((T, Hkv, D)), v, doc, 0.5)
    for a, b in zip(cu[:-1], cu[1:]):
        for t in range(a, b):
            assert np.allclose(o[t, 0], v[a:t + 1, 0].mean(0), atol=1e-14)
            assert lse[1, t] == pytest.approx(math.log(t - a + 1), abs=1e-14)
    # the first row of each document sees only itself
    k = _rand((T, Hkv, D), 9)
    o, lse = O.attention_fwd(q, k, v, doc, 0.5)
    for a in cu[:-1]:
        assert np.array_equal(o[a, 1], v[a, 0])
        assert lse[1, a] == pytest.approx(0.5 * float(q[a, 1] @ k[a, 0]), abs=1e-14)
    # V = 1: softmax rows sum to one
    o, _ = O.attention_fwd(q, k, np.ones((T, Hkv, D)), doc, 0.5)
    assert np.allclose(o, 1.0, atol=1e-14, rtol=0)


def test_fwd_brute_force_python_loops():
    T, D = 6, 3
    q, k, v = _rand((T, 1, D), 10), _rand((T, 1, D), 11), _rand((T, 1, D), 12)
    doc = np.array([0, 0, 0, 1, 1, -1])
    o, lse = O.attention_fwd(q, k, v, doc, 0.7)
    for t in range(T):
        keys = [u for u in range(T) if doc[t] >= 0 and doc[u] == doc[t] and u <= t]
        if not keys:
            assert np.all(o[t, 0] == 0) and lse[0, t] == -math.inf
            continue
        sc = {u: 0.7 * sum(q[t, 0, d] * k[u, 0, d] for d in range(D)) for u in keys}
        z = sum(math.exp(s) for s in sc.values())
        for d in range(D):
            want = sum(math.exp(sc[u]) / z * v[u, 0, d] for u in keys)
            assert o[t, 0, d] == pytest.approx(want, abs=1e-14)
        assert lse[0, t] == pytest.approx(math.log(z), abs=1e-14)


def _torch_grads(q, k, v, do, lens):
    tq, tk, tv = (torch.from_numpy(x).clone().requires_grad_(True) for x in (q, k, v))
    outs = []
    a = 0
    for n in lens:
        qq = tq[a:a + n].permute(1, 0, 2)[None]
        kk = tk[a:a + n].permute(1, 0, 2)[None]
        vv = tv[a:a + n].permute(1, 0, 2)[None]
        outs.append(F.scaled_dot_product_attention(
            qq, kk, vv, is_causal=True, enable_gqa=q.shape[1] != k.shape[1])[0].permute(1, 0, 2))
        a += n
    o = torch.cat(outs, 0)
    (o * torch.from_numpy(do)).sum().backward()
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


@pytest.mark.parametrize("lens,Hq,Hkv,D", [([40], 4, 2, 8), ([9, 1, 14], 8, 2, 4), ([25], 2, 2, 16)])
def test_bwd_matches_torch_autograd(lens, Hq, Hkv, D):
    T = sum(lens)
    q, k, v = _rand((T, Hq, D), 13), _rand((T, Hkv, D), 14), _rand((T, Hkv, D), 15)
    do = _rand((T, Hq, D), 16)
    _, doc = O.positions_docs(T, 1, np.concatenate([[0], np.cumsum(lens)]))
    dq, dk, dv = O.attention_bwd(q, k, v, do, doc, 1 / math.sqrt(D))
    tq, tk, tv = _torch_grads(q, k, v, do, lens)
    for a, b in ((dq, tq), (dk, tk), (dv, tv)):
        assert np.allclose(a, b, atol=1e-12, rtol=0)


def test_bwd_uniform_score_shift_has_zero_gradient():
    # If every key has the same component along a direction w, shifting q
    # along w shifts a whole score row by a constant, which softmax ignores:
    # sum_u dS_tu = 0 makes dQ . w vanish.
    T, Hq, Hkv, D = 20, 2, 1, 6
    q, k, v, do = _rand((T, Hq, D), 17), _rand((T, Hkv, D), 18), _rand((T, Hkv, D), 19), _rand((T, Hq, D), 20)
    k[..., -1] = 2.5
    doc = np.zeros(T, np.int64)
    dq, _, _ = O.attention_bwd(q, k, v, do, doc, 0.4)
    assert np.max(np.abs(dq[..., -1])) < 1e-13


def _loss_pre_rope(q, k, v, do, cu, cos, sin, P):
    r = O.ulysses(q, k, v, do, cu, cos, sin, 0.5, P)
    return r["loss"], r


def test_pipeline_gradients_by_finite_differences():
    # gradients w.r.t. the PRE-RoPE sequence-sharded inputs, through padding,
    # both all-to-alls, RoPE and its inverse
    S, P, Hq, Hkv, D = 7, 2, 2, 2, 4
    cu = np.array([0, 4, 7])
    q, k, v, do = _rand((S, Hq, D), 21), _rand((S, Hkv, D), 22), _rand((S, Hkv, D), 23), _rand((S, Hq, D), 24)
    cos, sin = O.rope_cos_sin(8, D, 100.0)
    _, r = _loss_pre_rope(q, k, v, do, cu, cos, sin, P)
    eps = 1e-6
    for name, x in (("dq", q), ("dk", k), ("dv", v)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + eps
            lp, _ = _loss_pre_rope(q, k, v, do, cu, cos, sin, P)
            x[idx] = old - eps
            lm, _ = _loss_pre_rope(q, k, v, do, cu, cos, sin, P)
            x[idx] = old
            num[idx] = (lp - lm) / (2 * eps)
        err = np.max(np.abs(num - r[name])) / max(1e-300, np.max(np.abs(r[name])))
        assert err <= 1e-6, (name, err)


@pytest.mark.parametrize("S,P,Hq,Hkv,D,lens", [
    (256, 2, 4, 2, 16, None),          # tiny-like, one sequence
    (30, 4, 8, 4, 8, None),            # padded 30 -> 32
    (45, 3, 6, 3, 8, [10, 1, 20, 14]),  # packed documents straddling shards
    (13, 8, 8, 8, 4, [13]),            # fewer rows per shard than one token each
])
def test_ulysses_equals_full_sequence(S, P, Hq, Hkv, D, lens):
    q, k, v, do = _rand((S, Hq, D), 25), _rand((S, Hkv, D), 26), _rand((S, Hkv, D), 27), _rand((S, Hq, D), 28)
    cu = None if lens is None else np.concatenate([[0], np.cumsum(lens)])
    cos, sin = O.rope_cos_sin(O.padded_len(S, P), D, 1.0e4)
    a = O.full_sequence(q, k, v, do, cu, cos, sin, 1 / math.sqrt(D))
    b = O.ulysses(q, k, v, do, cu, cos, sin, 1 / math.sqrt(D), P)
    for key in ("o", "dq", "dk", "dv"):
        assert np.allclose(a[key], b[key], atol=1e-12, rtol=0), key
    assert np.allclose(a["lse"], b["lse"], atol=1e-12, rtol=0)
    assert abs(a["loss"] - b["loss"]) <= 1e-12 * max(1.0, abs(a["loss"]))


def test_padding_has_no_effect_on_valid_rows():
    # S=30 over P=4 pads two rows; over P=2 and P=1 it pads none
    S, Hq, Hkv, D = 30, 4, 4, 8
    q, k, v, do = _rand((S, Hq, D), 29), _rand((S, Hkv, D), 30), _rand((S, Hkv, D), 31), _rand((S, Hq, D), 32)
    cos, sin = O.rope_cos_sin(32, D, 1.0e4)
    r4 = O.ulysses(q, k, v, do, None, cos, sin, 0.3, 4)
    r2 = O.ulysses(q, k, v, do, None, cos, sin, 0.3, 2)
    for key in ("o", "lse", "dq", "dk", "dv"):
        assert np.array_equal(r4[key], r2[key]) or np.allclose(r4[key], r2[key], atol=1e-13, rtol=0), key


def _torch_grads_masked(q, k, v, do, doc, causal):
    # one head, explicit boolean mask (same document, and u <= t if causal)
    tq, tk, tv = (torch.from_numpy(x).clone().requires_grad_(True) for x in (q, k, v))
    T = q.shape[0]
    d = torch.from_numpy(doc)
    mask = (d[:, None] == d[None, :]) & (d[:, None] >= 0)
    if causal:
        mask &= torch.ones(T, T, dtype=torch.bool).tril()
    o = F.scaled_dot_product_attention(tq[None, None], tk[None, None], tv[None, None],
                                       attn_mask=mask[None, None])[0, 0]
    o = torch.where(mask.any(1, keepdim=True), o, torch.zeros_like(o))
    (o * torch.from_numpy(do)).sum().backward()
    return tk.grad.numpy(), tv.grad.numpy()


@pytest.mark.parametrize("causal", [True, False])
def test_bwd_keys_matches_torch_autograd_and_splits_over_row_chunks(causal):
    # dK/dV at a few key rows, summed over all query rows, equal autograd's
    # (documents of lengths 9, 1, 14 and 2 pad rows); the sum over disjoint
    # row chunks equals the sum over all rows.
    lens = [9, 1, 14]
    T, D = sum(lens) + 2, 8
    q, k, v, do = (_rand((T, D), s) for s in (31, 32, 33, 34))
    _, doc = O.positions_docs(sum(lens), 1, np.concatenate([[0], np.cumsum(lens)]), S_pad=T)
    keys = np.array([0, 3, 9, 10, 11, 23, 24])
    dk, dv = O.attention_bwd_keys(q, k, v, do, doc, 1 / math.sqrt(D), keys, causal=causal)
    tk, tv = _torch_grads_masked(q, k, v, do, doc, causal)
    assert np.allclose(dk, tk[keys], atol=1e-12, rtol=0)
    assert np.allclose(dv, tv[keys], atol=1e-12, rtol=0)
    assert not dk[-1].any() and not dv[-1].any()          # a pad row is never a key
    parts = [O.attention_bwd_keys(q, k, v, do, doc, 1 / math.sqrt(D), keys, rows=r,
                                  causal=causal) for r in (np.arange(0, 7), np.arange(7, T))]
    assert np.allclose(parts[0][0] + parts[1][0], dk, atol=1e-13, rtol=0)
    assert np.allclose(parts[0][1] + parts[1][1], dv, atol=1e-13, rtol=0)


def test_parallel_key_gradients_equal_the_direct_oracle():
    # tests/oracle_pool.py (spawned workers over row chunks, used by the
    # full-size GPU checks) against the whole-sequence oracle: pre-RoPE dK/dV
    # of a GQA group's KV head at its first keys.
    from oracle_pool import dkdv_keys
    from ulysses_sequence_attention_usp_gb300.inputs import normal_bf16
    T, G, D = 300, 3, 16
    cu = np.array([0, 120, 300])
    pos, doc = O.positions_docs(T, 1, cu)
    cos, sin = O.rope_cos_sin(T, D, 1.0e4)
    qb = normal_bf16((T, G, D), 7, "q")
    kb, vb = normal_bf16((T, 1, D), 7, "k"), normal_bf16((T, 1, D), 7, "v")
    dob = normal_bf16((T, G, D), 7, "do")
    scale = 1 / math.sqrt(D)
    f = O.bf16_to_f64
    ref = O.full_sequence(f(qb), f(kb), f(vb), f(dob), cu, cos, sin, scale)
    keys = np.arange(120, 130)          # first keys of the second document
    dk, dv = dkdv_keys(qb, kb[:, 0], vb[:, 0], dob, pos, doc, cos, sin, scale, keys,
                       np.arange(120, 300), chunk=64, workers=2)
    assert np.allclose(dk, ref["dk"][keys, 0], atol=1e-12, rtol=0)
    assert np.allclose(dv, ref["dv"][keys, 0], atol=1e-12, rtol=0)
