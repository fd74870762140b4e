"""The RoPE cos/sin table the decode step and the prefill build on the GPU.

Its fp64 values are the correctly rounded cos and sin of the angles
fl(pos * inv_freq_j) ("手写LLM推理引擎…" section 3.2; the stored key is the
bf16 rounding of an fp64 rotation by them, so they must agree bit for bit
with the oracle's, which are pinned against a 200-bit evaluation). Checked
for every position below 2^17 and every frequency at the three bases in use
(12.6 million angles), at positions up to the largest int32, and for the
position table the decode step and the prefill read (row p = position p). The fp32 pairs must be the fp32 rounding
of each value and the fp32 rounding of the remainder.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_rope_gb300 as pkv

pytestmark = pytest.mark.gpu


def _split_table(table, n):
    raw = table.cpu().numpy()
    pairs = raw[:n * 512].view(np.float32).reshape(n, 32, 4)
    full = raw[n * 512:n * 1024].view(np.float64).reshape(n, 32, 2)
    return pairs, full


def _check_against_oracle(pos, theta, pairs, full):
    c, s, undecided = oracle.cos_sin(oracle.rope_angles(pos, theta))
    assert undecided == 0
    for got, want, what in ((full[..., 0], c, "cos"), (full[..., 1], s, "sin")):
        bad = got != want
        assert not bad.any(), (f"theta {theta}: {int(bad.sum())} fp64 {what} values differ from "
                               f"the correctly rounded ones, first at {np.argwhere(bad)[:3].tolist()}")
    for k, v in ((0, c), (2, s)):
        hi = v.astype(np.float32)
        lo = (v - hi.astype(np.float64)).astype(np.float32)
        assert np.array_equal(pairs[..., k], hi) and np.array_equal(pairs[..., k + 1], lo)
    return c


@pytest.mark.parametrize("theta", [1e4, 5e5, 1e6])
def test_table_is_correctly_rounded_for_every_position_below_2_17(theta):
    n = 1 << 17
    pos = torch.arange(n, dtype=torch.int32, device="cuda")
    table = pkv.alloc_rope_table(n)
    pkv.paged_rope_cos_sin(pos, theta, table)
    torch.cuda.synchronize()
    pairs, full = _split_table(table, n)
    c = _check_against_oracle(np.arange(n), theta, pairs, full)
    # for the record: how often the C library's cos is not the correctly rounded one
    sample = oracle.rope_angles(np.arange(0, n, 97), theta)
    libm = np.vectorize(math.cos)(sample)
    print(f"theta {theta}: C library cos differs from the correctly rounded value on "
          f"{int((libm != c[::97]).sum())} of {sample.size} sampled angles")


def test_table_at_large_positions():
    rng = np.random.default_rng(3)
    p = np.concatenate([[131072, 1 << 20, (1 << 21) - 1, 12345678, 2**31 - 1],
                        rng.integers(1 << 17, 2**31 - 1, 4091)]).astype(np.int32)
    pos = torch.from_numpy(p).cuda()
    for theta in (1e4, 5e5, 1e6):
        table = pkv.alloc_rope_table(p.size)
        pkv.paged_rope_cos_sin(pos, theta, table)
        torch.cuda.synchronize()
        pairs, full = _split_table(table, p.size)
        _check_against_oracle(p, theta, pairs, full)


def test_position_table_build_equals_the_gather():
    """paged_rope_table_build (row p = position p) gives the same bytes as
    paged_rope_cos_sin over positions 0..n-1, and the oracle's values."""
    n = 3000
    built = pkv.build_rope_table(1e6, n)
    gathered = pkv.alloc_rope_table(n)
    pkv.paged_rope_cos_sin(torch.arange(n, dtype=torch.int32, device="cuda"), 1e6, gathered)
    torch.cuda.synchronize()
    assert torch.equal(built, gathered)
    pairs, full = _split_table(built, n)
    _check_against_oracle(np.arange(n), 1e6, pairs, full)
