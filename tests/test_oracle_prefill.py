"""Pins for the oracle's chunked causal prefill.

Prefill ("Hours of YouTube …": prefill fills prompt pages; dense causal
prefill) is pinned to things other than itself: a one-token chunk is exactly
one decode step; splitting a chunk in two gives the same pool and outputs;
a token's output ignores later tokens (causality); sequences are independent;
and on a tiny case the outputs equal a brute-force causal attention written
with numpy from the pinned RoPE and bf16 primitives.
"""
import math

import numpy as np

import oracle

HQ, HKV, D, P = 4, 2, 64, 16
THETA, SCALE = 10000.0, 1.0 / 8.0


def _bits(rng, shape):
    x = rng.standard_normal(shape)
    return oracle.bf16_from_double(x).reshape(shape)


def _case(seed, starts, lens, num_pages=16, max_blocks=4):
    rng = np.random.default_rng(seed)
    total = int(sum(lens))
    pool = _bits(rng, (num_pages * 2 * HKV * P * D,))
    q = _bits(rng, (total, HQ, D))
    k = _bits(rng, (total, HKV, D))
    v = _bits(rng, (total, HKV, D))
    bt = np.stack([rng.permutation(num_pages)[:max_blocks] for _ in starts]).astype(np.int32)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return pool, q, k, v, bt, cu, np.asarray(starts, dtype=np.int32), max_blocks


def _prefill(pool, q, k, v, bt, cu, starts, max_blocks):
    return oracle.prefill(pool, num_kv_heads=HKV, q=q, k=k, v=v, block_tables=bt,
                          max_blocks=max_blocks, cu_tokens=cu, start_pos=starts,
                          num_q_heads=HQ, theta=THETA, scale=SCALE)


def test_one_token_chunk_is_one_decode_step():
    pool, q, k, v, bt, cu, starts, mb = _case(1, [37], [1])
    p1 = pool.copy()
    qr, out = _prefill(p1, q, k, v, bt, cu, starts, mb)
    p2 = pool.copy()
    qr2 = oracle.append_rope(p2, num_kv_heads=HKV, q=q, k=k, v=v, block_tables=bt, max_blocks=mb,
                             seq_lens=[38], positions=[37], batch=1, num_q_heads=HQ, theta=THETA)
    out2 = oracle.gqa_decode(p2, num_kv_heads=HKV, q_rot=qr2, block_tables=bt, max_blocks=mb,
                             seq_lens=[38], batch=1, num_q_heads=HQ, scale=SCALE)
    assert np.array_equal(p1, p2) and np.array_equal(qr, qr2) and np.array_equal(out, out2)


def test_splitting_a_chunk_changes_nothing():
    pool, q, k, v, bt, cu, starts, mb = _case(2, [5], [30])
    p1 = pool.copy()
    qr1, out1 = _prefill(p1, q, k, v, bt, cu, starts, mb)
    p2 = pool.copy()
    qa, oa = _prefill(p2, q[:12], k[:12], v[:12], bt, np.array([0, 12], np.int32), starts, mb)
    qb, ob = _prefill(p2, q[12:], k[12:], v[12:], bt, np.array([0, 18], np.int32),
                      np.array([17], np.int32), mb)
    assert np.array_equal(p1, p2)
    assert np.array_equal(out1, np.concatenate([oa, ob])) and np.array_equal(qr1, np.concatenate([qa, qb]))


def test_causality_later_tokens_do_not_matter():
    pool, q, k, v, bt, cu, starts, mb = _case(3, [9], [20])
    _, out1 = _prefill(pool.copy(), q, k, v, bt, cu, starts, mb)
    k2, v2 = k.copy(), v.copy()
    k2[-1] ^= 0x0101  # perturb the last token's key and value bits
    v2[-1] ^= 0x0101
    _, out2 = _prefill(pool.copy(), q, k2, v2, bt, cu, starts, mb)
    assert np.array_equal(out1[:-1], out2[:-1])
    assert not np.array_equal(out1[-1], out2[-1])


def test_sequences_are_independent():
    pool, q, k, v, bt, cu, starts, mb = _case(4, [0, 40], [17, 9], num_pages=32)
    p1 = pool.copy()
    _, out = _prefill(p1, q, k, v, bt, cu, starts, mb)
    p2 = pool.copy()
    _, o0 = _prefill(p2, q[:17], k[:17], v[:17], bt[:1], np.array([0, 17], np.int32), starts[:1], mb)
    _, o1 = _prefill(p2, q[17:], k[17:], v[17:], bt[1:], np.array([0, 9], np.int32), starts[1:], mb)
    assert np.array_equal(p1, p2) and np.array_equal(out, np.concatenate([o0, o1]))


def test_tiny_case_equals_brute_force_causal_attention():
    """One sequence, no cached tokens, 5 prompt tokens: numpy softmax attention
    over the rotated, bf16-rounded keys of tokens 0..t for query t."""
    pool, q, k, v, bt, cu, starts, mb = _case(5, [0], [5])
    _, out = _prefill(pool.copy(), q, k, v, bt, cu, starts, mb)
    pos = np.arange(5)
    qf = oracle.bf16_to_double(q).reshape(5, HQ, D)
    kf = oracle.bf16_to_double(k).reshape(5, HKV, D)
    vf = oracle.bf16_to_double(v).reshape(5, HKV, D)
    g = HQ // HKV
    for t in range(5):
        for i in range(HQ):
            h = i // g
            qr = oracle.rope_rotate(qf[t, i][None], [t], THETA)[0]
            keys = np.stack([oracle.bf16_to_double(oracle.bf16_from_double(
                oracle.rope_rotate(kf[s, h][None], [pos[s]], THETA)[0])) for s in range(t + 1)])
            sc = SCALE * keys @ qr
            w = np.exp(sc - sc.max())
            want = (w / w.sum()) @ vf[: t + 1, h]
            assert np.allclose(out[t, i], want, rtol=1e-12, atol=1e-12), (t, i)
    assert math.isfinite(out.sum())
