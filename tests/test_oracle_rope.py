"""Pins of the RoPE oracle and of its bfloat16 rounding (no GPU)."""
import math
import random
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle


def exact_bf16(x: float) -> float:
    """Brute-force nearest bfloat16 (8 significant bits, ties to even) with exact
    rational arithmetic, searching the two neighbouring candidates."""
    if x == 0.0 or not math.isfinite(x):
        return x
    fx = Fraction(x)
    e = math.frexp(abs(x))[1]                    # |x| in [2^(e-1), 2^e)
    qe = max(e - 8, -133)
    quantum = Fraction(2) ** qe
    lo = (fx / quantum).__floor__()
    cands = [lo, lo + 1]
    best = None
    for c in cands:
        err = abs(fx - c * quantum)
        if best is None or err < best[0] or (err == best[0] and c % 2 == 0):
            best = (err, c)
    r = best[1] * quantum
    if abs(r) >= Fraction(2) ** 128:
        return math.copysign(math.inf, x)
    return float(r)


def test_round_bf16_matches_exact_rounding():
    rng = random.Random(0)
    vals = [rng.gauss(0, 1) * 10 ** rng.uniform(-3, 3) for _ in range(3000)]
    # exact ties between two bfloat16 neighbours must go to the even one
    for m in range(128, 256):
        for e in (-3, 0, 5):
            vals.append((m + 0.5) * 2.0 ** (e - 7))
            vals.append(-(m + 0.5) * 2.0 ** (e - 7))
    vals += [1e-39, 3e-40, -2.5e-41, 3.3e38, 3.4e38, 1.0, -1.0]
    for x in vals:
        assert oracle.round_bf16(x) == exact_bf16(x), x


def test_round_bf16_values_are_bf16():
    rng = random.Random(1)
    for _ in range(500):
        y = oracle.round_bf16(rng.gauss(0, 3))
        bits = struct.unpack("<I", struct.pack("<f", y))[0]
        assert bits & 0xFFFF == 0


def test_position_zero_is_identity():
    x = np.random.default_rng(0).standard_normal((2, 1, 16)).astype(np.float32)
    y = oracle.rope(x, positions=[0], round_to="f32")
    assert np.array_equal(x, y)


def test_two_dim_closed_form():
    """d=2: theta_0 = base^0 = 1, so position m rotates (1, 0) to (cos m, sin m)."""
    x = np.tile(np.array([1.0, 0.0], np.float32), (5, 1))
    pos = [0, 1, 2, 7, 100]
    y = oracle.rope(x, base=10000.0, positions=pos, round_to=None)
    for t, m in enumerate(pos):
        assert y[t, 0] == pytest.approx(math.cos(m), abs=1e-15)
        assert y[t, 1] == pytest.approx(math.sin(m), abs=1e-15)
    # second pair of a d=4 vector turns by base^(-1/2) per position: 0.01 rad for 10000
    x4 = np.array([[0.0, 0.0, 1.0, 0.0]], np.float32)
    y4 = oracle.rope(x4, base=10000.0, positions=[100], round_to=None)
    assert np.allclose(y4[0], [0.0, 0.0, math.cos(1.0), math.sin(1.0)], atol=1e-14)


def test_relative_position_property():
    """The rotated q_m . k_n depends on m - n only."""
    rng = np.random.default_rng(2)
    d = 16
    q = rng.standard_normal((1, d)).astype(np.float32)
    k = rng.standard_normal((1, d)).astype(np.float32)
    for m, n in [(5, 2), (100, 40), (7, 7), (3, 90)]:
        dots = []
        for shift in (0, 13, 1000, 65000):
            qm = oracle.rope(q, positions=[m + shift], round_to=None)[0]
            kn = oracle.rope(k, positions=[n + shift], round_to=None)[0]
            dots.append(float(qm @ kn))
        assert np.allclose(dots, dots[0], atol=1e-10), (m, n, dots)


def test_pair_norms_preserved_and_rotations_compose():
    rng = np.random.default_rng(3)
    T, d = 40, 8
    x = rng.standard_normal((T, d)).astype(np.float32)
    y = oracle.rope(x, round_to=None)
    nx = (x.astype(np.float64).reshape(T, d // 2, 2) ** 2).sum(-1)
    ny = (y.reshape(T, d // 2, 2) ** 2).sum(-1)
    assert np.allclose(nx, ny, atol=1e-12)
    # rotating by position m and then by n equals rotating by m + n
    pos_a = rng.integers(0, 500, T)
    pos_b = rng.integers(0, 500, T)
    once = oracle.rope(x, positions=pos_a + pos_b, round_to=None)
    mid = oracle.rope(x, positions=pos_a, round_to=None)
    # second rotation applied to the fp64 intermediate, one coordinate pair at a time
    base = 10000.0
    twice = np.empty_like(mid)
    for t in range(T):
        for c in range(d // 2):
            ang = pos_b[t] * base ** (-2 * c / d)
            a, b = mid[t, 2 * c], mid[t, 2 * c + 1]
            twice[t, 2 * c] = a * math.cos(ang) - b * math.sin(ang)
            twice[t, 2 * c + 1] = a * math.sin(ang) + b * math.cos(ang)
    assert np.allclose(once, twice, atol=1e-11)


def test_rounded_output_is_rounding_of_fp64_result():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((3, 50, 8)) * 0.5).astype(np.float32)
    y64 = oracle.rope(x, round_to=None)
    yb = oracle.rope(x, round_to="bf16")
    yf = oracle.rope(x, round_to="f32")
    flat = y64.reshape(-1)
    assert np.array_equal(yf.reshape(-1), flat.astype(np.float32))
    for i in range(0, flat.size, 7):
        assert yb.reshape(-1)[i] == exact_bf16(float(flat[i]))


def test_odd_dimension_rejected():
    with pytest.raises(ValueError):
        oracle.rope(np.zeros((2, 3), np.float32))


def test_position_interpolation_rescales_the_index():
    """Position Interpolation ("Extending Context Window of Large Language Models
    via Position Interpolation" summary): positions are rescaled into the
    original range before rotating.  Scale 1/4 at positions 4m is plain RoPE at
    positions m, bit for bit (4m * 1/4 = m exactly); scale 1 is plain RoPE."""
    rng = np.random.default_rng(21)
    x = rng.standard_normal((2, 50, 16)).astype(np.float32)
    m = np.arange(50, dtype=np.int64) * 3 + 1
    plain = oracle.rope(x, base=10000.0, positions=m, round_to=None)
    pi = oracle.rope(x, base=10000.0, positions=4 * m, round_to=None, pos_scale=0.25)
    assert np.array_equal(plain, pi)
    assert np.array_equal(oracle.rope(x, positions=m, round_to=None, pos_scale=1.0), plain)
    assert not np.array_equal(oracle.rope(x, positions=m, round_to=None, pos_scale=0.5), plain)


def test_position_interpolation_keeps_relative_positions():
    """With scale s, the dot product of a rotated query at m and key at n depends
    only on (m - n) s: shifting both positions leaves it unchanged."""
    rng = np.random.default_rng(22)
    d = 8
    q = rng.standard_normal((1, 1, d)).astype(np.float32)
    k = rng.standard_normal((1, 1, d)).astype(np.float32)
    s = 0.375
    def dot(mq, nk):
        a = oracle.rope(q, positions=np.array([mq]), round_to=None, pos_scale=s)
        b = oracle.rope(k, positions=np.array([nk]), round_to=None, pos_scale=s)
        return float(np.sum(a * b))
    base_dot = dot(40, 11)
    for shift in (1, 17, 1000):
        assert abs(dot(40 + shift, 11 + shift) - base_dot) <= 1e-12
