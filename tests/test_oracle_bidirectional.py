"""Pins for the oracle's bidirectional variant (causal=False): attention
within each document over all of its keys, pad rows never keys (zhtmike/verl
PR #45 "[trainer] feat: support sequence parallel", What does this PR do:
Ulysses SP for the Diffusers SDPA attention with the padding for SP alignment
masked).

References: torch's scaled_dot_product_attention (is_causal=False, and with
an explicit boolean mask for documents) and autograd in fp64, a pure-Python
brute-force loop, the K = 0 closed form, and the Ulysses = full-sequence
identity."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import usp_oracle as O


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _t(x):
    return torch.from_numpy(x).permute(1, 0, 2)[None]      # [1, H, T, D]


def _sdpa(q, k, v, mask=None):
    o = F.scaled_dot_product_attention(_t(q), _t(k), _t(v), attn_mask=mask,
                                       enable_gqa=q.shape[1] != k.shape[1])
    return o[0].permute(1, 0, 2).numpy()


def _doc_mask(doc):
    d = torch.from_numpy(np.asarray(doc))
    return (d[:, None] == d[None, :]) & (d[None, :] >= 0)


@pytest.mark.parametrize("T,Hq,Hkv,D", [(33, 4, 2, 8), (17, 6, 2, 4)])
def test_bidirectional_fwd_matches_sdpa(T, Hq, Hkv, D):
    q, k, v = _rand((T, Hq, D), 11), _rand((T, Hkv, D), 12), _rand((T, Hkv, D), 13)
    o, _ = O.attention_fwd(q, k, v, np.zeros(T, np.int64), 1 / math.sqrt(D), causal=False)
    assert np.allclose(o, _sdpa(q, k, v), atol=1e-12, rtol=0)


def test_bidirectional_documents_and_padding_match_masked_sdpa():
    lens = [5, 1, 12, 7]
    cu = np.concatenate([[0], np.cumsum(lens)])
    S, P = int(cu[-1]), 8                      # 25 -> 32 rows, 7 pad rows
    pos, doc = O.positions_docs(S, P, cu)
    T, Hq, Hkv, D = doc.shape[0], 4, 2, 8
    q, k, v = _rand((T, Hq, D), 14), _rand((T, Hkv, D), 15), _rand((T, Hkv, D), 16)
    o, lse = O.attention_fwd(q, k, v, doc, 1 / math.sqrt(D), causal=False)
    ref = _sdpa(q, k, v, _doc_mask(doc))
    valid = doc >= 0
    assert np.allclose(o[valid], ref[valid], atol=1e-12, rtol=0)
    assert not o[~valid].any() and np.all(np.isneginf(lse[:, ~valid]))
    for a, b in zip(cu[:-1], cu[1:]):           # each document on its own
        assert np.allclose(o[a:b], _sdpa(q[a:b], k[a:b], v[a:b]), atol=1e-12, rtol=0)


def test_bidirectional_closed_form_zero_keys():
    # K = 0: every score is 0, so each row of a document averages the V of
    # the whole document and LSE = ln(document length)
    lens = [6, 3, 9]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, Hq, Hkv, D = int(cu[-1]), 2, 1, 4
    _, doc = O.positions_docs(T, 1, cu)
    q, k, v = _rand((T, Hq, D), 17), np.zeros((T, Hkv, D)), _rand((T, Hkv, D), 18)
    o, lse = O.attention_fwd(q, k, v, doc, 0.5, causal=False)
    for a, b in zip(cu[:-1], cu[1:]):
        mean = v[a:b, 0].mean(axis=0)
        for h in range(Hq):
            assert np.allclose(o[a:b, h], mean[None, :], atol=1e-12)
            assert np.allclose(lse[h, a:b], math.log(b - a), atol=1e-12)


def test_bidirectional_brute_force_loop():
    T, D = 7, 3
    doc = np.array([0, 0, 0, 1, 1, 1, -1])
    q, k, v = _rand((T, D), 19), _rand((T, D), 20), _rand((T, D), 21)
    o, lse = O.attention_rows(q, k, v, doc, np.arange(T), 0.7, causal=False)
    for t in range(T):
        keys = [u for u in range(T) if doc[t] >= 0 and doc[u] == doc[t]]
        if not keys:
            assert not o[t].any() and lse[t] == -np.inf
            continue
        w = [math.exp(0.7 * sum(q[t, i] * k[u, i] for i in range(D))) for u in keys]
        z = sum(w)
        for i in range(D):
            assert abs(o[t, i] - sum(wj * v[u, i] for wj, u in zip(w, keys)) / z) < 1e-12
        assert abs(lse[t] - math.log(z)) < 1e-12


def test_bidirectional_gradients_match_autograd():
    lens = [9, 4, 11]
    cu = np.concatenate([[0], np.cumsum(lens)])
    S, P = int(cu[-1]), 4                       # 24 rows, no pad
    _, doc = O.positions_docs(S, P, cu)
    T, Hq, Hkv, D = doc.shape[0], 4, 2, 8
    q, k, v, do = (_rand((T, Hq, D), 22), _rand((T, Hkv, D), 23), _rand((T, Hkv, D), 24),
                   _rand((T, Hq, D), 25))
    scale = 1 / math.sqrt(D)
    dq, dk, dv = O.attention_bwd(q, k, v, do, doc, scale, causal=False)
    tq, tk, tv = (_t(x).clone().requires_grad_() for x in (q, k, v))
    o = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=_doc_mask(doc), scale=scale,
                                       enable_gqa=True)
    (o * _t(do)).sum().backward()
    back = lambda g: g[0].permute(1, 0, 2).numpy()  # noqa: E731
    assert np.allclose(dq, back(tq.grad), atol=1e-10, rtol=0)
    assert np.allclose(dk, back(tk.grad), atol=1e-10, rtol=0)
    assert np.allclose(dv, back(tv.grad), atol=1e-10, rtol=0)


def test_bidirectional_differs_from_causal_only_before_the_last_row():
    T, D = 10, 4
    doc = np.zeros(T, np.int64)
    q, k, v = _rand((T, D), 26), _rand((T, D), 27), _rand((T, D), 28)
    oc, _ = O.attention_rows(q, k, v, doc, np.arange(T), 0.5, causal=True)
    ob, _ = O.attention_rows(q, k, v, doc, np.arange(T), 0.5, causal=False)
    assert np.allclose(oc[-1], ob[-1], atol=1e-14)      # the last row sees all keys either way
    assert not np.allclose(oc[0], ob[0])


@pytest.mark.parametrize("S,P,lens", [(30, 4, None), (25, 8, [5, 1, 12, 7]), (3, 8, None)])
def test_bidirectional_ulysses_equals_full_sequence(S, P, lens):
    Hq, Hkv, D = 8, 8, 8
    cu = None if lens is None else np.concatenate([[0], np.cumsum(lens)])
    q, k, v, do = (_rand((S, Hq, D), 29), _rand((S, Hkv, D), 30), _rand((S, Hkv, D), 31),
                   _rand((S, Hq, D), 32))
    cos, sin = O.rope_cos_sin(O.padded_len(S, P), D, 1.0e4)
    a = O.full_sequence(q, k, v, do, cu, cos, sin, 1 / math.sqrt(D), causal=False)
    b = O.ulysses(q, k, v, do, cu, cos, sin, 1 / math.sqrt(D), P, causal=False)
    for key in ("o", "dq", "dk", "dv"):
        assert np.allclose(a[key], b[key], atol=1e-12, rtol=0), key
    assert np.allclose(a["lse"], b["lse"], atol=1e-12, rtol=0)
