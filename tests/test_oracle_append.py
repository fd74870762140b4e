"""Pins for the oracle's append of the new token into the page pool.

Per the shared BF16 KV page pool item of "Hours of YouTube and 85 handtyped
pages of notes on LLM Inference – Start here", decode writes the new token's
K and V at its absolute position. The pins check where the bytes land (only
the slot of cache index seq_len - 1 changes), that V is copied verbatim, that
the stored key is a correctly rounded bf16 of the rotated key (the rotation
checked against the complex-number form), and that the rotated query is kept
unrounded.
"""
import numpy as np
import pytest

import oracle

D, P = 64, 16


def _complex_rot(x, pos, theta):
    half = x.shape[-1] // 2
    freqs = theta ** (-np.arange(half) * 2.0 / x.shape[-1])
    z = (x[..., :half] + 1j * x[..., half:]) * np.exp(1j * pos * freqs)
    return np.concatenate([z.real, z.imag], axis=-1)


def _case(rng, bsz=3, hkv=2, g=4, num_pages=12, seq_lens=(17, 16, 1), theta=500000.0):
    pool = np.full(num_pages * hkv * 2 * P * D, 0x7FC1, dtype=np.uint16)
    max_blocks = 3
    bt = np.full((bsz, max_blocks), -1, np.int32)
    free = rng.permutation(num_pages)
    cur = 0
    for b, n in enumerate(seq_lens):
        npg = -(-n // P)
        bt[b, :npg] = free[cur:cur + npg]
        cur += npg
    q = oracle.bf16_from_double(rng.standard_normal((bsz, hkv * g, D)))
    k = oracle.bf16_from_double(rng.standard_normal((bsz, hkv, D)))
    v = oracle.bf16_from_double(rng.standard_normal((bsz, hkv, D)))
    seq = np.array(seq_lens, np.int32)
    pos = seq - 1 + np.array([0, 100, 3000][:bsz], np.int32)  # positions need not equal the index
    return pool, bt, q, k, v, seq, pos, max_blocks, theta


def _append(pool, bt, q, k, v, seq, pos, max_blocks, theta, hkv=2):
    bsz, hq, _ = q.shape
    return oracle.append_rope(pool, num_kv_heads=hkv, q=q, k=k, v=v, block_tables=bt,
                              max_blocks=max_blocks, seq_lens=seq, positions=pos, batch=bsz,
                              num_q_heads=hq, theta=theta)


def test_only_the_new_slot_changes_and_values_are_right():
    rng = np.random.default_rng(0)
    pool, bt, q, k, v, seq, pos, mb, theta = _case(rng)
    before = pool.copy()
    q_rot = _append(pool, bt, q, k, v, seq, pos, mb, theta)
    view = pool.reshape(-1, 2, 2, P, D)
    changed = np.argwhere((pool != before).reshape(view.shape).any(axis=(1, 2, 4)))
    want = {(int(bt[b, (seq[b] - 1) // P]), int((seq[b] - 1) % P)) for b in range(3)}
    assert {(int(p), int(s)) for p, s in changed} == want
    for b in range(3):
        t = seq[b] - 1
        page, slot = bt[b, t // P], t % P
        for h in range(2):
            # V verbatim
            assert np.array_equal(view[page, h, 1, slot], v[b, h])
            # K is the rotated key rounded to bf16: within half a bf16 ulp of the
            # exact rotation, and equal to the oracle's own rounding of it.
            exact = _complex_rot(oracle.bf16_to_double(k[b, h]), float(pos[b]), theta)
            stored = oracle.bf16_to_double(view[page, h, 0, slot])
            half_ulp = np.ldexp(1.0, np.frexp(np.abs(exact))[1] - 9)
            assert np.all(np.abs(stored - exact) <= half_ulp * (1 + 1e-9) + 1e-300)
            assert np.array_equal(view[page, h, 0, slot],
                                  oracle.bf16_from_double(oracle.rope_rotate(
                                      oracle.bf16_to_double(k[b, h])[None], pos[b:b + 1], theta)[0]))
    # q_rot is the unrounded fp64 rotation of q
    for b in range(3):
        np.testing.assert_allclose(q_rot[b], _complex_rot(oracle.bf16_to_double(q[b]), float(pos[b]), theta),
                                   rtol=0, atol=1e-11)


def test_page_boundaries():
    # seq_len 16 -> index 15: last slot of the first page; 17 -> first slot of the second page.
    rng = np.random.default_rng(1)
    pool, bt, q, k, v, seq, pos, mb, theta = _case(rng, seq_lens=(16, 17, 33))
    before = pool.copy()
    _append(pool, bt, q, k, v, seq, pos, mb, theta)
    view = (pool != before).reshape(-1, 2, 2, P, D).any(axis=(1, 2, 4))
    assert view[bt[0, 0], 15] and view[bt[1, 1], 0] and view[bt[2, 2], 0]
    assert view.sum() == 3


def test_position_zero_stores_key_unchanged():
    rng = np.random.default_rng(2)
    pool, bt, q, k, v, seq, pos, mb, theta = _case(rng, bsz=1, seq_lens=(1,))
    pos[:] = 0
    q_rot = _append(pool, bt, q, k, v, seq, pos, mb, theta)
    view = pool.reshape(-1, 2, 2, P, D)
    assert np.array_equal(view[bt[0, 0], :, 0, 0], k[0])
    assert np.array_equal(q_rot[0], oracle.bf16_to_double(q[0]))


def test_errors():
    rng = np.random.default_rng(3)
    pool, bt, q, k, v, seq, pos, mb, theta = _case(rng)
    with pytest.raises(ValueError, match="-1"):
        _append(pool, bt, q, k, v, np.array([0, 1, 1], np.int32), pos, mb, theta)
    bad = bt.copy()
    bad[0, 1] = 999
    with pytest.raises(ValueError, match="-2"):
        _append(pool, bad, q, k, v, seq, pos, mb, theta)
