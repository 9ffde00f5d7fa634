"""Pins for the oracle's ring attention (windowed attention and the
log-sum-exp merge of partial results; SpecForge PR #728 and verl PR #45
configure a Ulysses x Ring mesh).

References: the full attention of the oracle's pinned forward (ring over any
number of chunks must reproduce it), a brute-force loop for a window, merge
identities, and a softmax split in two written out with math.exp."""
import math

import numpy as np
import pytest

from oracle import usp_oracle as O


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("R", [1, 2, 3, 5, 8])
def test_ring_equals_full_attention(R, causal):
    T, Hq, Hkv, D = 37, 4, 2, 8
    q, k, v = _rand((T, Hq, D), 1), _rand((T, Hkv, D), 2), _rand((T, Hkv, D), 3)
    _, doc = O.positions_docs(33, 1, np.array([0, 10, 11, 30, 33]), S_pad=T)   # 4 pad rows
    o, lse = O.attention_fwd(q, k, v, doc, 0.3, causal)
    o2, lse2 = O.ring_fwd(q, k, v, doc, 0.3, R, causal)
    assert np.allclose(o, o2, atol=1e-12, rtol=0)
    fin = np.isfinite(lse)
    assert np.array_equal(fin, np.isfinite(lse2))
    assert np.allclose(lse[fin], lse2[fin], atol=1e-12, rtol=0)


def test_window_brute_force():
    T, D = 9, 3
    doc = np.array([0, 0, 0, 0, 1, 1, 1, 1, -1])
    q, k, v = _rand((T, 1, D), 4), _rand((T, 1, D), 5), _rand((T, 1, D), 6)
    for causal in (True, False):
        o, lse = O.attention_window(q, k, v, doc, 0.7, 2, 6, causal)
        for t in range(T):
            keys = [u for u in range(2, 6)
                    if doc[t] >= 0 and doc[u] == doc[t] and (u <= t or not causal)]
            if not keys:
                assert not o[t, 0].any() and lse[0, t] == -np.inf
                continue
            w = [math.exp(0.7 * sum(q[t, 0, i] * k[u, 0, i] for i in range(D))) for u in keys]
            z = sum(w)
            for i in range(D):
                want = sum(wj * v[u, 0, i] for wj, u in zip(w, keys)) / z
                assert abs(o[t, 0, i] - want) < 1e-12
            assert abs(lse[0, t] - math.log(z)) < 1e-12


def test_full_and_empty_windows():
    T, H, D = 12, 2, 4
    q, k, v = _rand((T, H, D), 7), _rand((T, H, D), 8), _rand((T, H, D), 9)
    doc = np.zeros(T, np.int64)
    o, lse = O.attention_fwd(q, k, v, doc, 0.5)
    ow, lw = O.attention_window(q, k, v, doc, 0.5, 0, T)
    assert np.allclose(o, ow, atol=1e-14) and np.allclose(lse, lw, atol=1e-14)
    oe, le = O.attention_window(q, k, v, doc, 0.5, 5, 5)
    assert not oe.any() and np.all(np.isneginf(le))


def test_merge_identities_and_split_softmax():
    T, H, D = 5, 2, 3
    o_a, l_a = _rand((T, H, D), 10), _rand((H, T), 11)
    empty_o, empty_l = np.zeros((T, H, D)), np.full((H, T), -np.inf)
    o, l = O.lse_merge(o_a, l_a, empty_o, empty_l)
    assert np.allclose(o, o_a, atol=1e-15) and np.allclose(l, l_a, atol=1e-15)
    o_b, l_b = _rand((T, H, D), 12), _rand((H, T), 13)
    o1, l1 = O.lse_merge(o_a, l_a, o_b, l_b)
    o2, l2 = O.lse_merge(o_b, l_b, o_a, l_a)
    assert np.allclose(o1, o2, atol=1e-14) and np.allclose(l1, l2, atol=1e-14)
    # one row, scores s_0..s_5 split {0,1,2} | {3,4,5}, values x_u (scalars)
    s = [0.3, -1.2, 2.0, 0.7, 0.1, -0.4]
    x = [1.0, 2.0, -1.0, 0.5, 3.0, -2.0]
    def part(idx):
        z = sum(math.exp(s[i]) for i in idx)
        return sum(math.exp(s[i]) * x[i] for i in idx) / z, math.log(z)
    (oa, la), (ob, lb) = part([0, 1, 2]), part([3, 4, 5])
    om, lm = O.lse_merge(np.array([[[oa]]]), np.array([[la]]), np.array([[[ob]]]),
                         np.array([[lb]]))
    z = sum(math.exp(v) for v in s)
    assert abs(om[0, 0, 0] - sum(math.exp(si) * xi for si, xi in zip(s, x)) / z) < 1e-14
    assert abs(lm[0, 0] - math.log(z)) < 1e-14
