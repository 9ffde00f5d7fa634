"""Pins for the oracle's context parallelism with a K/V all-gather
(basetenlabs/Megatron-LM PR #7 "GLM-5.2 131k context parallelism", Purpose:
all-gather of the KV across CP ranks in the forward, reduce-scatter of dKV
in the backward, contiguous partition, global cu_seqlens positions).

References: the pinned full-sequence computation (every CP degree, with or
without documents and padding, must reproduce it), central finite
differences of the loss on a tiny case, and the causal and document
structure of each rank's partial dK/dV before the reduction."""
import numpy as np
import pytest

from oracle import usp_oracle as O


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _case(S, Hq, Hkv, D, seed=0):
    return (_rand((S, Hq, D), seed + 1), _rand((S, Hkv, D), seed + 2),
            _rand((S, Hkv, D), seed + 3), _rand((S, Hq, D), seed + 4))


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("P", [1, 2, 3, 4])
@pytest.mark.parametrize("heads", [(4, 1), (4, 2), (2, 2)])
def test_allgather_equals_full_sequence(P, heads, causal):
    S, D = 23, 8                                  # 23 rows: padding for P = 2, 3, 4
    Hq, Hkv = heads
    q, k, v, do = _case(S, Hq, Hkv, D)
    cu = np.array([0, 7, 8, 19, 23])             # a single-row document included
    cos, sin = O.rope_cos_sin(64, D, 1.0e4)
    ref = O.full_sequence(q, k, v, do, cu, cos, sin, 0.35, causal)
    got = O.allgather_cp(q, k, v, do, cu, cos, sin, 0.35, P, causal)
    for n in ("o", "dq", "dk", "dv"):
        assert np.allclose(got[n], ref[n], atol=1e-12, rtol=0), n
    assert np.allclose(got["lse"], ref["lse"], atol=1e-12, rtol=0)
    assert abs(got["loss"] - ref["loss"]) <= 1e-12 * max(1.0, abs(ref["loss"]))


def test_fewer_kv_heads_than_ranks():
    # the case the all-to-all cannot shard: Hkv = 1 < P = 4
    S, Hq, Hkv, D, P = 16, 4, 1, 4, 4
    q, k, v, do = _case(S, Hq, Hkv, D, seed=10)
    cos, sin = O.rope_cos_sin(S, D, 1.0e4)
    with pytest.raises(ValueError):
        O.ulysses(q, k, v, do, None, cos, sin, 0.5, P)
    got = O.allgather_cp(q, k, v, do, None, cos, sin, 0.5, P)
    ref = O.full_sequence(q, k, v, do, None, cos, sin, 0.5)
    assert np.allclose(got["dk"], ref["dk"], atol=1e-12, rtol=0)


def test_gradients_by_finite_differences():
    S, Hq, Hkv, D, P = 7, 2, 1, 4, 3
    q, k, v, do = _case(S, Hq, Hkv, D, seed=20)
    cu = np.array([0, 4, 7])
    cos, sin = O.rope_cos_sin(S + 2, D, 1.0e4)
    got = O.allgather_cp(q, k, v, do, cu, cos, sin, 0.6, P)
    eps = 1e-6
    rng = np.random.default_rng(21)
    for name, x in (("dq", q), ("dk", k), ("dv", v)):
        for _ in range(6):
            idx = tuple(int(rng.integers(n)) for n in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args = {"dq": (xp, k, v), "dk": (q, xp, v), "dv": (q, k, xp)}[name]
            argm = {"dq": (xm, k, v), "dk": (q, xm, v), "dv": (q, k, xm)}[name]
            lp = O.allgather_cp(*args, do, cu, cos, sin, 0.6, P)["loss"]
            lm = O.allgather_cp(*argm, do, cu, cos, sin, 0.6, P)["loss"]
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - got[name][idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx)


@pytest.mark.parametrize("causal", [True, False])
def test_rank_partials_follow_the_mask(causal):
    # before the reduction, rank r's partial dK/dV can be non-zero only on the
    # key rows its queries see: none after its last row (causal) and none
    # outside the documents of its rows
    S, Hq, Hkv, D, P = 20, 2, 1, 4, 4
    q, k, v, do = _case(S, Hq, Hkv, D, seed=30)
    cu = np.array([0, 3, 12, 20])
    cos, sin = O.rope_cos_sin(S, D, 1.0e4)
    out = O.allgather_cp(q, k, v, do, cu, cos, sin, 0.4, P, causal, return_partials=True)
    _, doc = O.positions_docs(S, P, cu)
    S_loc = doc.shape[0] // P
    for r in range(P):
        rows = np.arange(r * S_loc, (r + 1) * S_loc)
        seen = set(doc[rows][doc[rows] >= 0].tolist())
        for u in range(doc.shape[0]):
            visible = doc[u] in seen and (not causal or u <= rows[-1])
            if not visible:
                assert not out["dk_part"][r, u].any() and not out["dv_part"][r, u].any()
        # the rank's own last row is a key it sees (itself) in every mode
        assert out["dv_part"][r, rows[-1]].any()
