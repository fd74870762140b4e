"""Pins for the oracle's double -> bf16 rounding (round to nearest, ties to even).

The rounding decides the pool bytes the append writes, which must match bit
for bit, so it is pinned three independent ways: encodings fixed by the format
itself, torch's float32 -> bf16 conversion on float32-exact inputs, and a
brute-force nearest search over the whole bf16 codebook with exact rationals.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

# (value, bf16 encoding) fixed by the format: 1 sign, 8 exponent (bias 127),
# 7 fraction bits; subnormal spacing 2^-133.
FORMAT_CASES = [
    (1.0, 0x3F80),
    (-2.0, 0xC000),
    (0.1, 0x3DCD),                      # 1.6 * 2^-4, fraction 0.6*128 = 76.8 -> 77
    (1 + 2**-8, 0x3F80),                # exact tie, even neighbour is 1.0
    (1 + 3 * 2**-8, 0x3F82),            # exact tie, even neighbour is 1 + 2^-6
    (1 + 2**-8 + 2**-40, 0x3F81),       # just above the tie
    (1 + 2**-8 - 2**-40, 0x3F80),       # just below the tie
    ((2 - 2**-7) * 2.0**127, 0x7F7F),   # largest finite bf16
    ((2 - 2**-8) * 2.0**127, 0x7F80),   # tie between largest finite and 2^128: rounds to inf
    ((2 - 2**-8) * 2.0**127 * (1 - 2**-50), 0x7F7F),
    (2.0**-126, 0x0080),                # smallest normal
    (2.0**-133, 0x0001),                # smallest subnormal
    (2.0**-134, 0x0000),                # tie between 0 and 2^-133: even is 0
    (3 * 2.0**-134, 0x0002),            # tie between 1 and 2 quanta: even is 2
    (2.0**-134 * 1.0000001, 0x0001),
    (1e-300, 0x0000),
    (-1e-300, 0x8000),
    (1e300, 0x7F80),
    (-1e300, 0xFF80),
    (math.inf, 0x7F80),
    (-math.inf, 0xFF80),
    (0.0, 0x0000),
    (-0.0, 0x8000),
    (math.nan, 0x7FC0),
]


@pytest.mark.parametrize("value,bits", FORMAT_CASES)
def test_format_cases(value, bits):
    got = int(oracle.bf16_from_double(np.array([value]))[0])
    assert got == bits, f"{value!r}: got {got:#06x}, want {bits:#06x}"


def test_bf16_to_double_roundtrip_all_finite():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bf16_to_double(bits)
    finite = np.isfinite(vals)
    back = oracle.bf16_from_double(vals[finite])
    # -0.0 and +0.0 keep their sign; every finite encoding round-trips.
    assert np.array_equal(back, bits[finite])


def test_matches_torch_on_float32_exact_inputs():
    # For a double that is exactly a float32, one rounding from double equals
    # torch's float32 -> bf16 round-to-nearest-even.
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000),
        rng.standard_normal(5000) * 1e-39,        # float32 subnormal range
        rng.standard_normal(5000) * 1e37,
        rng.uniform(-4, 4, 5000),
    ]).astype(np.float32)
    # add exact ties: float32 values whose low 16 bits are 0x8000
    ties = (rng.integers(0, 1 << 15, 4000).astype(np.uint32) << 16 | 0x8000).view(np.float32)
    x = np.concatenate([x, ties[np.isfinite(ties)]])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_from_double(x.astype(np.float64))
    assert np.array_equal(got, want)


def _codebook():
    bits = np.arange(0, 0x7F80, dtype=np.uint32).astype(np.uint16)  # +0 .. largest finite
    vals = oracle.bf16_to_double(bits)
    return bits, vals


def _nearest_by_search(x: float, bits, vals) -> int:
    """Nearest bf16 to x by searching the sorted codebook, ties to the even encoding."""
    sign = 0x8000 if math.copysign(1.0, x) < 0 else 0
    a = abs(x)
    fa = Fraction(a)
    i = int(np.searchsorted(vals, a))
    if i < len(vals) and vals[i] == a:
        return sign | int(bits[i])
    lo_bits, lo = int(bits[i - 1]), Fraction(float(vals[i - 1]))
    if i < len(vals):
        hi_bits, hi = int(bits[i]), Fraction(float(vals[i]))
    else:  # above the largest finite value: the next grid point is 2^128 (inf)
        hi_bits, hi = 0x7F80, Fraction(2) ** 128
    dlo, dhi = fa - lo, hi - fa
    if dlo < dhi:
        return sign | lo_bits
    if dhi < dlo:
        return sign | hi_bits
    return sign | (lo_bits if lo_bits % 2 == 0 else hi_bits)


def test_brute_force_codebook_search():
    bits, vals = _codebook()
    rng = np.random.default_rng(7)
    xs = list(rng.standard_normal(1500))
    xs += list(rng.standard_normal(300) * 2.0**-128)          # subnormal region
    xs += list(rng.uniform(0.99, 1.01, 300))
    xs += [float(v) + float(d) for v, d in zip(vals[rng.integers(1, len(vals) - 1, 300)],
                                               rng.standard_normal(300) * 1e-12)]
    xs += [-x for x in xs[:200]]
    xs = np.array(xs, dtype=np.float64)
    got = oracle.bf16_from_double(xs)
    for x, g in zip(xs, got):
        assert int(g) == _nearest_by_search(float(x), bits, vals), x
