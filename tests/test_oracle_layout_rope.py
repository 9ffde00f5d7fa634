"""Pins for the oracle's shard/pad, all-to-all and RoPE functions.

Every check compares the oracle with something other than itself: hand-worked
fixtures under tests/golden, closed forms, IEEE rounding facts, brute-force
loops and algebraic invariants of rotations."""
import json
import math
import os
import struct

import numpy as np
import pytest

from oracle import usp_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------- shard/pad

def test_positions_docs_hand_example():
    g = _gold("positions_thd.json")
    pos, doc = O.positions_docs(g["S"], g["P"], np.array(g["cu_seqlens"]))
    assert pos.tolist() == g["pos"]
    assert doc.tolist() == g["doc"]


def test_positions_single_sequence_padded():
    # one sequence of 30 tokens over P=4: pads to 32, positions keep counting
    pos, doc = O.positions_docs(30, 4)
    assert pos.tolist() == list(range(32))
    assert doc.tolist() == [0] * 30 + [-1, -1]


def test_shard_pad_zero_tail_and_identity():
    x = np.arange(7 * 2 * 3, dtype=np.float64).reshape(7, 2, 3) + 1
    y = O.shard_pad(x, 4)
    assert y.shape == (8, 2, 3)
    assert np.array_equal(y[:7], x) and not y[7].any()
    assert np.array_equal(O.shard_pad(x, 7), x)       # already a multiple
    assert np.array_equal(O.shard_pad(x, 1), x)


def test_padded_len_examples():
    assert O.padded_len(32766, 8) == 32768
    assert O.padded_len(120000, 8) == 120000
    assert O.padded_len(1, 8) == 8
    assert O.padded_len(0, 8) == 0


# ---------------------------------------------------------------- all-to-all

def test_a2a_hand_example():
    g = _gold("a2a_hand.json")
    x = np.array(g["x_seq"], dtype=np.float64)[:, :, None]
    want = np.array(g["x_head"], dtype=np.float64)[..., None]
    assert np.array_equal(O.seq_to_head_loops(x, 2), want)
    assert np.array_equal(O.seq_to_head(x, 2), want)
    assert np.array_equal(O.head_to_seq(want), x)


@pytest.mark.parametrize("P,S_pad,H,D", [(2, 8, 4, 3), (4, 12, 8, 2), (1, 5, 3, 2), (3, 9, 6, 1)])
def test_a2a_loops_equal_vectorised_and_inverse(P, S_pad, H, D):
    rng = np.random.default_rng(1)
    x = rng.standard_normal((S_pad, H, D))
    a = O.seq_to_head_loops(x, P)
    b = O.seq_to_head(x, P)
    assert np.array_equal(a, b)
    assert np.array_equal(O.head_to_seq(b), x)
    if P == 1:
        assert np.array_equal(b[0], x)


def test_check_heads():
    O.check_heads(8, 32, 8)
    O.check_heads(2, 4, 2)
    O.check_heads(8, 64, 8)
    for bad in [(8, 32, 4), (3, 32, 8), (0, 4, 2), (2, 4, 3), (4, 6, 2)]:
        with pytest.raises(ValueError):
            O.check_heads(*bad)


# ---------------------------------------------------------------------- RoPE

def test_rope_hand_example_pairing_and_sign():
    # D=4, base b: pairs (0,2) at inv_freq 1 and (1,3) at b^-1/2.  At pos 1 the
    # first pair turns by exactly 1 radian counter-clockwise.
    b = 1.0e4
    cos, sin = O.rope_cos_sin(3, 4, b)
    assert O.rope_inv_freq(4, b)[1] == pytest.approx(0.01, rel=1e-15)
    pos = np.array([1])
    e0 = np.array([[[1.0, 0, 0, 0]]])
    e2 = np.array([[[0.0, 0, 1, 0]]])
    y0 = O.rope_rotate(e0, pos, cos, sin)[0, 0]
    y2 = O.rope_rotate(e2, pos, cos, sin)[0, 0]
    assert y0 == pytest.approx([math.cos(1), 0, math.sin(1), 0], abs=1e-15)
    assert y2 == pytest.approx([-math.sin(1), 0, math.cos(1), 0], abs=1e-15)
    # second pair at pos 2 turns by 2 * 0.01 radians
    e1 = np.array([[[0.0, 1, 0, 0]]])
    y1 = O.rope_rotate(e1, np.array([2]), cos, sin)[0, 0]
    assert y1 == pytest.approx([0, math.cos(0.02), 0, math.sin(0.02)], abs=1e-15)


def test_rope_invariants():
    rng = np.random.default_rng(2)
    D, T = 16, 40
    cos, sin = O.rope_cos_sin(200, D, 1.0e4)
    x = rng.standard_normal((T, 3, D))
    pos = rng.integers(0, 150, T)
    y = O.rope_rotate(x, pos, cos, sin)
    # identity at position 0
    assert np.array_equal(O.rope_rotate(x, np.zeros(T, np.int64), cos, sin), x)
    # each (i, i+D/2) pair keeps its norm
    h = D // 2
    assert np.allclose(x[..., :h] ** 2 + x[..., h:] ** 2, y[..., :h] ** 2 + y[..., h:] ** 2,
                       rtol=1e-13, atol=0)
    # inverse undoes forward
    assert np.allclose(O.rope_rotate(y, pos, cos, sin, inverse=True), x, atol=1e-13)
    # scores depend only on the position difference
    q = rng.standard_normal((1, 1, D))
    k = rng.standard_normal((1, 1, D))
    for m, n, c in [(5, 3, 17), (0, 9, 40), (100, 100, 7)]:
        s1 = (O.rope_rotate(q, np.array([m]), cos, sin) * O.rope_rotate(k, np.array([n]), cos, sin)).sum()
        s2 = (O.rope_rotate(q, np.array([m + c]), cos, sin) * O.rope_rotate(k, np.array([n + c]), cos, sin)).sum()
        assert abs(s1 - s2) <= 1e-12


def test_rope_table_layout_and_norm():
    t = O.rope_table_f32(64, 8, 1.0e4)
    assert t.shape == (64, 4, 2) and t.dtype == np.float32
    assert np.all(t[0, :, 0] == 1.0) and np.all(t[0, :, 1] == 0.0)
    assert np.allclose(t[..., 0].astype(np.float64) ** 2 + t[..., 1].astype(np.float64) ** 2,
                       1.0, atol=2e-7)
    # entry = fp32 rounding of cos/sin of pos * base^(-2i/D)
    assert t[3, 1, 0] == np.float32(math.cos(3 * 1.0e4 ** (-2 / 8)))
    assert t[5, 2, 1] == np.float32(math.sin(5 * 1.0e4 ** (-4 / 8)))


def test_yarn_factor_one_is_plain_rope_bitwise():
    a = O.rope_table_f32(1000, 128, 1.0e6)
    b = O.rope_table_f32(1000, 128, 1.0e6, factor=1.0, orig_ctx=32768)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_yarn_regimes_and_mscale():
    # Peng et al. 2023: pairs that turn many times over the original context
    # keep their frequency; pairs whose wavelength exceeds it are slowed by
    # the scale factor; cos/sin carry mscale = 0.1 ln(s) + 1.
    D, base, s, L = 128, 1.0e6, 4.0, 32768
    plain = O.rope_inv_freq(D, base)
    yarn = O.rope_inv_freq(D, base, s, L)
    turns = L * plain / (2 * math.pi)
    fast = turns >= 64
    slow = turns <= 0.5
    assert fast.sum() > 10 and slow.sum() > 10
    assert np.array_equal(yarn[fast], plain[fast])
    assert np.allclose(yarn[slow], plain[slow] / s, rtol=1e-15)
    assert np.all(yarn <= plain) and np.all(yarn >= plain / s * (1 - 1e-15))
    assert np.all(np.diff(yarn) < 0)                     # still monotone in i
    assert O.rope_mscale(4.0) == pytest.approx(1.1386294361119891, rel=1e-15)
    t = O.rope_table_f32(4, D, base, s, L)
    assert np.all(t[0, :, 0] == np.float32(1.1386294361119891))


def test_yarn_ramp_hand_worked_golden():
    # Correction range and interior ramp values worked out by hand from
    # Peng et al. 2023, sec. 3.2, for the 131,072-token YaRN table of
    # SpecForge PR #728, Accuracy Test (tests/golden/yarn_ramp.json holds the
    # derivation).  An off-by-one in the floor/ceil of the correction range,
    # a wrong ramp denominator or a ramp over the wrong index all move these.
    g = _gold("yarn_ramp.json")
    D, base, L, s = g["D"], g["base"], g["orig_ctx"], g["scale"]
    two_ln_b = 2 * math.log(base)
    assert D * math.log(L / (2 * math.pi * g["beta_fast"])) / two_ln_b == pytest.approx(
        g["corr_dim_fast"], abs=1e-3)
    assert D * math.log(L / (2 * math.pi * g["beta_slow"])) / two_ln_b == pytest.approx(
        g["corr_dim_slow"], abs=1e-3)
    yarn = O.rope_inv_freq(D, base, s, L)
    for i, ratio in g["ratio_to_plain"].items():
        plain = 10.0 ** (-6.0 * 2 * int(i) / D)
        assert yarn[int(i)] == pytest.approx(plain * ratio, rel=1e-13), i
    for i, e in g["inv_freq_exponent_of_10"].items():
        ratio = g["ratio_to_plain"][i]
        assert yarn[int(i)] == pytest.approx(10.0 ** e * ratio, rel=1e-13), i
    # the ramp is linear in i between the two ends: equal steps of f_i * 0.75/17
    lo, hi = g["ramp_lo"], g["ramp_hi"]
    plain = O.rope_inv_freq(D, base)
    steps = np.diff(yarn[lo:hi + 1] / plain[lo:hi + 1])
    assert np.allclose(steps, -0.75 / (hi - lo), rtol=0, atol=1e-14)


# ---------------------------------------------------------- bf16 RoPE recipe

def _f32(v):
    return struct.unpack("<f", struct.pack("<f", v))[0]


def _bits(v):  # bf16 bits of a value exactly representable in bf16
    u = struct.unpack("<I", struct.pack("<f", v))[0]
    assert u & 0xFFFF == 0
    return u >> 16


def _table(c, s):
    t = np.zeros((2, 1, 2), dtype=np.float32)
    t[0, 0] = (1.0, 0.0)
    t[1, 0] = (c, s)
    return t


def _apply(x1, x2, c, s, inverse=False):
    x = np.array([[[_bits(x1), _bits(x2)]]], dtype=np.uint16)
    y = O.rope_recipe_bf16(x, np.array([1]), _table(c, s), inverse)
    return y[0, 0].tolist()


def test_recipe_exact_hand_values():
    # x1=1.5, x2=-2, c=0.5, s=0.75 -> y1 = 0.75 + 1.5 = 2.25, y2 = -1 + 1.125
    assert _apply(1.5, -2.0, 0.5, 0.75) == [_bits(2.25), _bits(0.125)]
    # inverse rotation negates s: y1 = 0.75 - 1.5, y2 = -1 - 1.125
    assert _apply(1.5, -2.0, 0.5, 0.75, inverse=True) == [_bits(-0.75), _bits(-2.125)]


def test_recipe_rounds_to_nearest_even():
    # 1 + 2^-8 lies halfway between bf16 neighbours 1 and 1 + 2^-7: even -> 1
    assert _apply(1.0, 0.0, 1.0 + 2 ** -8, 0.0)[0] == _bits(1.0)
    # 1 + 3*2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6: even -> 1 + 2^-6
    assert _apply(1.0, 0.0, 1.0 + 3 * 2 ** -8, 0.0)[0] == _bits(1.0 + 2 ** -6)
    # just above the tie rounds up
    assert _apply(1.0, 0.0, 1.0 + 2 ** -8 + 2 ** -20, 0.0)[0] == _bits(1.0 + 2 ** -7)


def _bf16_of_f32(v):
    u = struct.unpack("<I", struct.pack("<f", v))[0]
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) & 0xFFFF


def test_recipe_rounds_each_product_to_fp32():
    # Input found by search where rounding each product to fp32 first (the
    # recipe) and rotating exactly then rounding once give different bf16
    # results.  The expected bits follow from IEEE fp32 rounding done here
    # one operation at a time with struct.
    x1 = struct.unpack("<f", bytes.fromhex("0000b73d"))[0]   # bf16 0x3db7
    x2 = struct.unpack("<f", bytes.fromhex("000095bd"))[0]   # bf16 0xbd95
    c = struct.unpack("<f", bytes.fromhex("049eebbe"))[0]
    s = struct.unpack("<f", bytes.fromhex("344863bf"))[0]
    y1 = _f32(_f32(x1 * c) - _f32(x2 * s))
    assert _bf16_of_f32(y1) == 0xBDD8
    assert _bf16_of_f32(_f32(x1 * c - x2 * s)) == 0xBDD9     # one rounding
    assert _apply(x1, x2, c, s)[0] == 0xBDD8


def test_recipe_position_zero_is_identity_and_close_to_exact():
    rng = np.random.default_rng(3)
    T, H, D = 64, 4, 32
    x = O.f32_to_bf16(rng.standard_normal((T, H, D)).astype(np.float32))
    table = O.rope_table_f32(T, D, 1.0e4)
    assert np.array_equal(O.rope_recipe_bf16(x, np.zeros(T, np.int64), table), x)
    pos = np.arange(T)
    y = O.bf16_to_f64(O.rope_recipe_bf16(x, pos, table))
    # exact fp64 rotation with the same fp32 table entries
    c = table[..., 0].astype(np.float64)
    s = table[..., 1].astype(np.float64)
    exact = O.rope_rotate(O.bf16_to_f64(x), pos, c, s)
    # each output is within one bf16 ulp of the exact value (RNE after two
    # fp32 roundings of size 2^-24 relative)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(exact), 1e-30))) - 7)
    assert np.all(np.abs(y - exact) <= ulp)
    assert np.mean(np.abs(y - exact) <= ulp / 2 + 1e-30) > 0.99
