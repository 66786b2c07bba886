"""Pins for the oracle's RoPE, bf16 rounding and fused RoPE append.

"Faster fuzzy minds" ("Recurrent depth — a deep model in a trench coat"): a
token keeps one RoPE position across all T of its banks; depth is not sequence
position.  The pages fix no RoPE variant; the reading taken is the
rotate-half pairing (x[i], x[i + rot_dim/2]) turned by pos * base^(-2i/rot_dim).
These pins check the oracle against properties of rotations and against
library routines (numpy power, cos, sin), not against a retyped formula.
"""
import math

import numpy as np
import pytest

import oracle


def bf16_to_float(bits):
    return np.asarray(bits, np.uint32).astype(np.uint32).__lshift__(16).view(np.float32).astype(np.float64)


# ------------------------------------------------------------ bf16 rounding

def test_bf16_round_is_nearest_with_ties_to_even():
    rng = np.random.default_rng(0)
    xs = np.concatenate([rng.normal(size=3000) * 10.0 ** rng.integers(-30, 30, size=3000),
                         rng.uniform(-4, 4, size=3000)])
    for x in xs:
        b = oracle.bf16_round(float(x))
        v = float(bf16_to_float(b))
        # neighbours of the chosen pattern in the direction of x
        for nb in (b - 1, b + 1):
            if (nb & 0x7F80) == 0x7F80 or nb < 0 or nb > 0xFFFF or (nb ^ b) & 0x8000:
                continue
            w = float(bf16_to_float(nb))
            assert abs(x - v) <= abs(x - w), (x, hex(b), hex(nb))
            if abs(x - v) == abs(x - w):
                assert b % 2 == 0                       # tie: the even mantissa wins


def test_bf16_round_special_values():
    assert oracle.bf16_round(0.0) == 0x0000
    assert oracle.bf16_round(-0.0) == 0x8000
    assert oracle.bf16_round(float("nan")) == 0x7FC0
    assert oracle.bf16_round(1e39) == 0x7F80
    assert oracle.bf16_round(-1e39) == 0xFF80
    assert oracle.bf16_round(1.0 + 2 ** -8) == 0x3F80        # halfway, to even
    assert oracle.bf16_round(1.0 + 3 * 2 ** -8) == 0x3F82    # halfway, to even (up)
    assert oracle.bf16_round(2.0 ** -133) == 0x0001          # smallest subnormal
    assert oracle.bf16_round(2.0 ** -135) == 0x0000          # below half of it
    # every bf16 value is its own rounding
    for b in range(0, 0x7F80, 97):
        assert oracle.bf16_round(float(bf16_to_float(b))) == b


# ------------------------------------------------------------------- RoPE

D, BASE = 128, 10000.0


def test_rope_position_zero_is_identity():
    x = np.random.default_rng(1).normal(size=D)
    assert np.array_equal(oracle.rope(x, 0, D, BASE), x)


def test_rope_unit_vectors_turn_by_the_pair_frequency():
    half = D // 2
    theta = np.power(BASE, -2.0 * np.arange(half) / D)
    for i in (0, 1, 17, half - 1):
        for pos in (1, 7, 1000, 131071):
            e = np.zeros(D)
            e[i] = 1.0
            y = oracle.rope(e, pos, D, BASE)
            a = pos * theta[i]
            assert abs(y[i] - math.cos(a)) < 1e-12 and abs(y[i + half] - math.sin(a)) < 1e-12
            y[i] = y[i + half] = 0.0
            assert np.all(y == 0)                       # rotate-half: only dims i and i + D/2 move


def test_rope_preserves_pair_norms_and_is_a_rotation_group():
    rng = np.random.default_rng(2)
    half = D // 2
    for _ in range(20):
        x = rng.normal(size=D)
        a, b = (int(v) for v in rng.integers(0, 200000, size=2))
        y = oracle.rope(x, a, D, BASE)
        n0 = np.hypot(x[:half], x[half:])
        n1 = np.hypot(y[:half], y[half:])
        assert np.allclose(n0, n1, rtol=1e-12, atol=1e-12)
        # two turns add their positions
        z = oracle.rope(y, b, D, BASE)
        assert np.allclose(z, oracle.rope(x, a + b, D, BASE), rtol=1e-9, atol=1e-9)


def test_rope_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(3)
    q, k = rng.normal(size=D), rng.normal(size=D)
    for m, n in ((5, 3), (4096, 17), (131000, 130000), (9, 9)):
        lhs = oracle.rope(q, m, D, BASE) @ oracle.rope(k, n, D, BASE)
        rhs = oracle.rope(q, m - n, D, BASE) @ k
        assert abs(lhs - rhs) < 1e-9 * (1 + abs(rhs))


@pytest.mark.parametrize("rot_dim", [32, 64])
def test_partial_rotary_leaves_the_rest(rot_dim):
    x = np.random.default_rng(4).normal(size=D)
    y = oracle.rope(x, 12345, rot_dim, BASE)
    assert np.array_equal(y[rot_dim:], x[rot_dim:])
    assert not np.allclose(y[:rot_dim], x[:rot_dim])
    # the rotated block is the full rotation of a rot_dim-wide head
    assert np.array_equal(y[:rot_dim], oracle.rope(x[:rot_dim], 12345, rot_dim, BASE))


# --------------------------------------------------------- fused append

def test_append_rope_rotates_keys_copies_values_and_skips():
    rng = np.random.default_rng(5)
    P, Hkv, ps, Dh = 9, 2, 16, 64
    kp = rng.integers(0, 2 ** 16, size=(P, Hkv, ps, Dh), dtype=np.uint16) & 0x7F7F   # finite patterns
    vp = rng.integers(0, 2 ** 16, size=(P, Hkv, ps, Dh), dtype=np.uint16) & 0x7F7F
    kn = np.array([oracle.bf16_round(v) for v in rng.normal(size=4 * Hkv * Dh)], np.uint16).reshape(4, Hkv, Dh)
    vn = np.array([oracle.bf16_round(v) for v in rng.normal(size=4 * Hkv * Dh)], np.uint16).reshape(4, Hkv, Dh)
    pos = np.array([0, 15, 77, 100000], np.int64)
    loc = np.array([3, -1, 70, 143], np.int64)
    k2, v2 = kp.copy(), vp.copy()
    oracle.kv_append_rope(k2, v2, kn, vn, pos, loc, 48, 500000.0)
    for i, s in enumerate(loc):
        if s < 0:
            continue
        page, off = divmod(int(s), ps)
        assert np.array_equal(v2[page, :, off], vn[i])
        for g in range(Hkv):
            want = [oracle.bf16_round(v) for v in
                    oracle.rope(bf16_to_float(kn[i, g]), int(pos[i]), 48, 500000.0)]
            assert np.array_equal(k2[page, g, off], np.array(want, np.uint16))
        k2[page, :, off] = kp[page, :, off]
        v2[page, :, off] = vp[page, :, off]
    assert np.array_equal(k2, kp) and np.array_equal(v2, vp)   # nothing else changed


def test_append_rope_at_position_zero_stores_the_key_unchanged():
    rng = np.random.default_rng(6)
    kn = np.array([oracle.bf16_round(v) for v in rng.normal(size=2 * 64)], np.uint16).reshape(1, 2, 64)
    k = np.zeros((1, 2, 1, 64), np.uint16)
    v = np.zeros_like(k)
    oracle.kv_append_rope(k, v, kn, kn, [0], [0], 64, 10000.0)
    assert np.array_equal(k[0, :, 0], kn[0]) and np.array_equal(v[0, :, 0], kn[0])
