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
