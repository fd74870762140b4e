"""The new key's rotation at bf16 rounding boundaries, both step paths.

Each rotated key element is stored as the bf16 round-to-nearest-even of an
fp64 rotation (RoPE equations of "手写LLM推理引擎…" section 3.2; fp64 products
and sum, as the oracle computes them). The fused step gets there without
fp64 arithmetic when it can certify the rounding from an fp32 double-word
estimate and falls back to fp64 otherwise; the append kernel uses fp64.
Random keys almost never land close to a rounding boundary, so this test
searches, with the oracle's own rotation, for bf16 pairs whose rotated value
lies within about 2^-24 (relative) of a bf16 midpoint -- where an fp32-only
estimate would misround about half the time -- and plants them, plus pairs
of zeros (which take the fp64 route), in the new keys. The pool bytes must
equal the oracle's.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import DeviceWorkload, oracle_layer, u16

pytestmark = pytest.mark.gpu

HALF = 32


def _random_bf16_bits(rng, shape):
    """bf16 bit patterns, both signs, magnitudes in [2^-4, 2^5)."""
    sign = rng.integers(0, 2, shape, dtype=np.uint16) << 15
    expo = rng.integers(127 - 4, 127 + 5, shape, dtype=np.uint16) << 7
    mant = rng.integers(0, 128, shape, dtype=np.uint16)
    return (sign | expo | mant).astype(np.uint16)


def _midpoint_distance(y):
    """|y - nearest midpoint between neighbouring bf16 values| (inf for y == 0)."""
    ay = np.abs(y)
    m, e = np.frexp(ay)  # ay = m 2^e, m in [0.5, 1): bf16 spacing 2^(e-8)
    ulp = np.ldexp(1.0, e - 8)
    t = ay / ulp
    d = np.abs(t - np.floor(t) - 0.5) * ulp
    return np.where(ay > 0, d, np.inf)


def near_tie_keys(pos, theta, rows, n_cand, seed):
    """``rows`` key rows of bf16 bits [rows, 64] for one position: for every
    frequency j the pairs (j, j+32) are the candidates (out of n_cand random
    ones) whose rotation by the oracle lands closest, relative to the pair's
    magnitude, to a bf16 midpoint. Also returns the planted pairs' relative
    distances [rows, 32]. (Where the angle is tiny -- high frequencies at small
    positions -- the rotation barely moves x and no candidate comes close.)"""
    rng = np.random.default_rng(seed)
    bits = _random_bf16_bits(rng, (n_cand, 2 * HALF))
    x = oracle.bf16_to_double(bits).reshape(n_cand, 2 * HALF)
    y = oracle.rope_rotate(x, np.full(n_cand, pos, dtype=np.int32), theta)
    scale = np.maximum(np.abs(x[:, :HALF]), np.abs(x[:, HALF:]))
    d = np.minimum(_midpoint_distance(y[:, :HALF]), _midpoint_distance(y[:, HALF:])) / scale
    out = np.empty((rows, 2 * HALF), dtype=np.uint16)
    planted = np.empty((rows, HALF))
    for j in range(HALF):
        best = np.argsort(d[:, j], kind="stable")[:rows]
        out[:, j] = bits[best, j]
        out[:, j + HALF] = bits[best, j + HALF]
        planted[:, j] = d[best, j]
    return out, planted


def test_rotation_rounds_like_fp64_at_midpoints():
    cached = [0, 5, 16, 40, 200, 1000, 4095, 33000]  # position 0 (cos 1, sin 0) included
    wl = workloads.build("ties", batch=len(cached), num_layers=1, num_q_heads=32, num_kv_heads=8,
                         cached_lens=cached, rope_theta=500000.0, seed=11, sentinel=True)
    k = u16(wl.k).copy()  # [1, B, Hkv, 64]
    close = 0
    for b in range(wl.batch):
        rows, planted = near_tie_keys(int(wl.positions[b]), wl.rope_theta, wl.num_kv_heads,
                                      1 << 16, seed=100 + b)
        k[0, b] = rows
        close += int((planted < 2.0 ** -21).sum())
    assert close >= 512, close  # the search really found near-ties
    # zero pairs: both zero (every sign combination) and one zero
    z = np.uint16(0x8000)
    k[0, 0, 0, [0, 1, 2, 3]] = [0, z, 0, z]
    k[0, 0, 0, [HALF, HALF + 1, HALF + 2, HALF + 3]] = [0, 0, z, z]
    k[0, 0, 0, 4], k[0, 0, 0, HALF + 5] = 0, z
    wl.k = torch.from_numpy(k.view(np.int16)).view(torch.bfloat16)

    for fused in (True, False):
        dw = DeviceWorkload(wl)
        dw.run(fused=fused)
        assert dw.step.error_bits() == 0
        pool_host = u16(wl.pool).reshape(-1).copy()
        oracle_layer(pool_host, wl, 0, u16(wl.q)[0], k[0], u16(wl.v)[0])
        got = u16(dw.pool).reshape(-1)
        mism = np.flatnonzero(got != pool_host)
        assert mism.size == 0, f"fused={fused}: {mism.size} pool elements differ, first at {mism[:5]}"
        dw.step.close()
