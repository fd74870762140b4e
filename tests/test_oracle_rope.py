"""Pins for the oracle's rotary position embedding.

The rotation follows the two RoPE equations of "手写LLM推理引擎：Tokenizer、
Transformer与Detokenizer三段式实现" section 3.2 with rotate-half pairing
(j, j + D/2) and inverse frequency base^(-2j/D). Each pin checks it against
something other than itself: closed forms, the complex-number form of the
rotation, a hand example evaluated in 40-digit arithmetic, and the invariants
that define a rotary embedding.
"""
import math

import numpy as np
import pytest

import oracle
from tests.golden.figures import page_figures


def test_inv_freq_closed_forms():
    figs = page_figures()
    base, dim = figs["rope_table_base"], figs["rope_table_dim"]
    inv = oracle.rope_inv_freq(float(base), dim)
    assert inv.shape == (dim // 2,)
    assert inv[0] == 1.0
    # j = D/4: base^(-1/2). For the page's table (base 10000, dim 128) that is 1/100.
    assert inv[dim // 4] == pytest.approx(0.01, rel=1e-15)
    # inv_j * inv_{D/2 - j} = base^(-1) for every j
    for j in range(1, dim // 2):
        assert inv[j] * inv[dim // 2 - j] == pytest.approx(1 / base, rel=1e-14)
    # geometric: consecutive ratio is base^(-2/D)
    np.testing.assert_allclose(inv[1:] / inv[:-1], base ** (-2.0 / dim), rtol=1e-14)


def test_position_zero_is_identity():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 64))
    y = oracle.rope_rotate(x, np.zeros(5, np.int32), 500000.0)
    assert np.array_equal(x, y)


def _complex_form(x, pos, theta):
    """RoPE as multiplication of z_j = x_j + i x_{j+D/2} by exp(i pos theta_j)."""
    n, d = x.shape
    half = d // 2
    freqs = theta ** (-np.arange(half) * 2.0 / d)
    z = x[:, :half] + 1j * x[:, half:]
    w = z * np.exp(1j * (pos[:, None].astype(np.float64) * freqs[None, :]))
    return np.concatenate([w.real, w.imag], axis=1)


@pytest.mark.parametrize("theta", [10000.0, 500000.0, 1e6])
def test_matches_complex_form(theta):
    rng = np.random.default_rng(1)
    x = rng.standard_normal((200, 64))
    pos = rng.integers(0, 4097, 200).astype(np.int32)
    y = oracle.rope_rotate(x, pos, theta)
    # numpy's power and the C library's pow may differ by an ulp in the inverse
    # frequency; at angles up to 4096 rad that moves cos/sin by ~1e-12.
    np.testing.assert_allclose(y, _complex_form(x, pos, theta), rtol=0, atol=1e-11)


def test_hand_example_high_precision():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 40
    # D = 4, base 100, position 3: pairs (x0, x2) at angle 3 and (x1, x3) at
    # angle 3 * 100^(-1/2) = 0.3.
    x = np.array([[1.0, 2.0, 3.0, 4.0]])
    y = oracle.rope_rotate(x, np.array([3], np.int32), 100.0)[0]
    a0, a1 = mp.mpf(3), mp.mpf(3) * mp.power(100, mp.mpf(-0.5))
    want = [1 * mp.cos(a0) - 3 * mp.sin(a0),
            2 * mp.cos(a1) - 4 * mp.sin(a1),
            3 * mp.cos(a0) + 1 * mp.sin(a0),
            4 * mp.cos(a1) + 2 * mp.sin(a1)]
    for got, w in zip(y, want):
        assert got == pytest.approx(float(w), rel=0, abs=4e-16)


def test_pair_norms_preserved():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((100, 64))
    pos = rng.integers(0, 100000, 100).astype(np.int32)
    y = oracle.rope_rotate(x, pos, 500000.0)
    nx = np.hypot(x[:, :32], x[:, 32:])
    ny = np.hypot(y[:, :32], y[:, 32:])
    np.testing.assert_allclose(ny, nx, rtol=1e-13)


def test_relative_position_property():
    # <R_m q, R_n k> depends only on m - n.
    rng = np.random.default_rng(3)
    q = rng.standard_normal((50, 64))
    k = rng.standard_normal((50, 64))
    m = rng.integers(0, 3000, 50).astype(np.int32)
    n = rng.integers(0, 3000, 50).astype(np.int32)
    delta = rng.integers(0, 1000, 50).astype(np.int32)
    for theta in (500000.0, 1e6):
        d0 = np.sum(oracle.rope_rotate(q, m, theta) * oracle.rope_rotate(k, n, theta), axis=1)
        d1 = np.sum(oracle.rope_rotate(q, m + delta, theta) * oracle.rope_rotate(k, n + delta, theta), axis=1)
        np.testing.assert_allclose(d1, d0, rtol=0, atol=1e-9 * 64)


def test_rotation_direction():
    # Position 1 of base-1 RoPE (all frequencies 1) rotates (1, 0) to (cos 1, sin 1):
    # counter-clockwise, the sign convention of the equations.
    x = np.zeros((1, 8))
    x[0, 0] = 1.0
    y = oracle.rope_rotate(x, np.array([1], np.int32), 1.0)[0]
    assert y[0] == pytest.approx(math.cos(1.0), abs=1e-16)
    assert y[4] == pytest.approx(math.sin(1.0), abs=1e-16)
    assert np.count_nonzero(y) == 2


def _cr_reference(angles):
    """cos and sin of each fp64 angle in 200-bit arithmetic, rounded to the
    nearest fp64 value (mpmath; an independent evaluation)."""
    mpmath = pytest.importorskip("mpmath")
    from mpmath.libmp import round_nearest, to_float
    c, s = [], []
    with mpmath.workprec(200):
        for a in angles:
            x = mpmath.mpf(float(a))
            c.append(to_float(mpmath.cos(x)._mpf_, rnd=round_nearest))
            s.append(to_float(mpmath.sin(x)._mpf_, rnd=round_nearest))
    return np.array(c), np.array(s)


def _rope_sample_angles():
    """RoPE angles fl(pos * inv_j) at the three bases in use: every frequency
    at a spread of positions (small, page-sized, the context caps, far beyond
    them, up to the largest int32), plus random doubles and the doubles
    nearest to multiples of pi/2 (the reductions with most cancellation)."""
    rng = np.random.default_rng(5)
    pos = np.unique(np.concatenate([np.arange(0, 40), [63, 64, 1000, 2047, 2048, 4095, 4096,
                                                       65535, 131071, 1 << 20, 12345678,
                                                       2**31 - 1],
                                    rng.integers(0, 1 << 17, 150)]))
    ang = [oracle.rope_angles(pos, th).reshape(-1) for th in (1e4, 5e5, 1e6)]
    k = np.arange(1, 4000, dtype=np.float64)
    near = k * (math.pi / 2)
    return np.concatenate(ang + [rng.uniform(0, 2**17, 3000), near, np.nextafter(near, 0)])


def test_cos_sin_are_correctly_rounded():
    """The oracle's fp64 cos and sin are the fp64 values nearest to the true
    ones (checked against a 200-bit evaluation), and every rounding was
    decided."""
    a = _rope_sample_angles()
    c, s, undecided = oracle.cos_sin(a)
    assert undecided == 0
    want_c, want_s = _cr_reference(a)
    assert np.array_equal(c, want_c), int((c != want_c).sum())
    assert np.array_equal(s, want_s), int((s != want_s).sum())


def test_cos_sin_special_values_and_symmetry():
    c, s, bad = oracle.cos_sin(np.array([0.0, -0.0]))
    assert bad == 0 and np.all(c == 1.0) and np.all(s == 0.0)
    assert not np.signbit(s[0]) and np.signbit(s[1])       # sin(+0) = +0, sin(-0) = -0
    rng = np.random.default_rng(6)
    a = rng.uniform(0, 1e5, 2000)
    c1, s1, _ = oracle.cos_sin(a)
    c2, s2, _ = oracle.cos_sin(-a)
    assert np.array_equal(c1, c2) and np.array_equal(s1, -s2)  # cos even, sin odd


def test_cos_sin_within_one_ulp_of_the_c_library():
    """The C library's cos and sin are not correctly rounded everywhere but
    are within one ulp: a sanity bound on the oracle's values."""
    a = _rope_sample_angles()
    c, s, _ = oracle.cos_sin(a)
    lc = np.array([math.cos(x) for x in a])
    ls = np.array([math.sin(x) for x in a])
    for got, ref in ((c, lc), (s, ls)):
        ulp = np.spacing(np.abs(ref))
        assert np.all(np.abs(got - ref) <= ulp)


def test_cos_sin_decided_over_the_whole_rope_domain():
    """Every angle fl(pos * inv_j) for positions below 2^17 and every
    frequency at bases 1e4, 5e5 and 1e6 (12.6 million values each of cos and
    sin) is decided by the oracle's rounding test, so the pool's bit-exact key
    bytes are defined everywhere the workloads reach."""
    for th in (1e4, 5e5, 1e6):
        _, _, undecided = oracle.cos_sin(oracle.rope_angles(np.arange(1 << 17), th))
        assert undecided == 0, th
