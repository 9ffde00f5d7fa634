"""Pins for the oracle's zigzag partition (Megatron-LM PR #7 "GLM-5.2 131k
context parallelism", closing comment: upstream's zigzag CP; reading: 2P
equal chunks, rank r holds chunks r and 2P-1-r).

References: a hand-worked layout, the identity at P = 1, equal causal work
per rank (which singles out the r / 2P-1-r pairing), the contiguous
all-to-all applied after undoing the zigzag order, round trips, and the
Ulysses = full-sequence identity."""
import math

import numpy as np
import pytest

from oracle import usp_oracle as O


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_hand_worked_layout():
    # P = 2, S = 8: four chunks of 2 rows; rank 0 holds chunks 0 and 3, rank 1
    # holds chunks 1 and 2
    assert O.zigzag_padded_len(8, 2) == 8
    assert list(O.zigzag_order(8, 2)) == [0, 1, 6, 7, 2, 3, 4, 5]
    # P = 4, S = 8: chunks of 1 row; ranks hold (0,7) (1,6) (2,5) (3,4)
    assert list(O.zigzag_order(8, 4)) == [0, 7, 1, 6, 2, 5, 3, 4]


def test_one_rank_is_identity_and_order_is_a_permutation():
    assert np.array_equal(O.zigzag_order(10, 1), np.arange(10))
    for S_pad, P in ((48, 4), (32, 8), (6, 3)):
        assert np.array_equal(np.sort(O.zigzag_order(S_pad, P)), np.arange(S_pad))


@pytest.mark.parametrize("S_pad,P", [(64, 4), (96, 8), (20, 2)])
def test_every_rank_gets_the_same_causal_work(S_pad, P):
    order = O.zigzag_order(S_pad, P).reshape(P, -1)
    work = (order + 1).sum(axis=1)             # causal keys seen by each rank's rows
    assert np.all(work == work[0])
    contiguous = (np.arange(S_pad).reshape(P, -1) + 1).sum(axis=1)
    assert not np.all(contiguous == contiguous[0])


def test_padding_rows_are_zero_and_at_the_global_tail():
    S, P, H, D = 7, 2, 2, 3
    x = _rand((S, H, D), 1)
    y = O.shard_pad_zigzag(x, P)
    order = O.zigzag_order(8, P)
    assert y.shape[0] == 8
    for i, t in enumerate(order):
        assert np.array_equal(y[i], x[t]) if t < S else not y[i].any()


def test_all_to_all_equals_contiguous_after_reordering():
    S_pad, P, H, D = 24, 4, 8, 2
    x_seq = _rand((S_pad, H, D), 2)
    order = O.zigzag_order(S_pad, P)
    x_global = x_seq[np.argsort(order)]          # row t of the global sequence
    assert np.array_equal(O.seq_to_head_zigzag(x_seq, P), O.seq_to_head(x_global, P))
    assert np.array_equal(O.head_to_seq_zigzag(O.seq_to_head_zigzag(x_seq, P)), x_seq)


def test_positions_with_zigzag_padding_stay_global():
    cu = np.array([0, 5, 11])
    pos, doc = O.positions_docs(11, 2, cu, S_pad=O.zigzag_padded_len(11, 2))
    assert pos.shape[0] == 12
    assert list(pos) == [0, 1, 2, 3, 4, 0, 1, 2, 3, 4, 5, 6]
    assert list(doc) == [0] * 5 + [1] * 6 + [-1]


@pytest.mark.parametrize("S,P,lens,causal", [(30, 4, None, True), (25, 2, [5, 1, 12, 7], True),
                                             (25, 2, [5, 1, 12, 7], False), (3, 2, None, True)])
def test_zigzag_ulysses_equals_full_sequence(S, P, lens, causal):
    Hq, Hkv, D = 8, 4, 8
    cu = None if lens is None else np.concatenate([[0], np.cumsum(lens)])
    q, k, v, do = (_rand((S, Hq, D), 3), _rand((S, Hkv, D), 4), _rand((S, Hkv, D), 5),
                   _rand((S, Hq, D), 6))
    cos, sin = O.rope_cos_sin(O.zigzag_padded_len(S, P), D, 1.0e4)
    a = O.full_sequence(q, k, v, do, cu, cos, sin, 1 / math.sqrt(D), causal=causal)
    b = O.ulysses(q, k, v, do, cu, cos, sin, 1 / math.sqrt(D), P, causal=causal, zigzag=True)
    for key in ("o", "dq", "dk", "dv", "lse"):
        assert np.allclose(a[key], b[key], atol=1e-12, rtol=0), key
