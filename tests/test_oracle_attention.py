"""Pins for the oracle's paged GQA decode attention and its split/LSE merge.

The attention follows the direct paged decode attention item of "Hours of
YouTube and 85 handtyped pages of notes on LLM Inference – Start here": every
query head attends over the cached pages of its own sequence. Pins: closed
forms (one token, identical keys, zero scale, two tokens, GQA head mapping),
the invariance to where pages sit in the pool, brute force on dense
contiguous K/V with scipy's softmax, and the closed form of the LSE merge.
"""
import numpy as np
import pytest
from scipy.special import expit, softmax

import oracle

D, P = 64, 16


def _scatter_pool(kdense, vdense, num_pages, rng):
    """Place dense per-(b, h) K/V [B][Hkv][N_b][D] (lists) into a fresh pool.

    Returns (pool_u16, block_tables [B][max_blocks], seq_lens). The pool layout
    is [page][kv_head][K|V][slot][dim]; pages are drawn from a random permutation.
    """
    bsz = len(kdense)
    hkv = kdense[0].shape[0]
    lens = np.array([kd.shape[1] for kd in kdense], dtype=np.int32)
    max_blocks = int(-(-lens.max() // P))
    pool = np.full((num_pages, hkv, 2, P, D), 0x7FC1, dtype=np.uint16)
    free = rng.permutation(num_pages)
    bt = np.full((bsz, max_blocks), -1, dtype=np.int32)
    cur = 0
    for b in range(bsz):
        npg = -(-int(lens[b]) // P)
        bt[b, :npg] = free[cur:cur + npg]
        cur += npg
        for t in range(int(lens[b])):
            pool[bt[b, t // P], :, 0, t % P, :] = kdense[b][:, t, :]
            pool[bt[b, t // P], :, 1, t % P, :] = vdense[b][:, t, :]
    return pool.reshape(-1), bt, lens


def _bf16_bits(x):
    return oracle.bf16_from_double(x)


def _decode(pool, bt, lens, q_rot, hkv, scale=1 / 8):
    bsz, hq, _ = q_rot.shape
    return oracle.gqa_decode(pool, num_kv_heads=hkv, q_rot=q_rot, block_tables=bt,
                             max_blocks=bt.shape[1], seq_lens=lens, batch=bsz,
                             num_q_heads=hq, scale=scale)


def _random_case(rng, lens, hkv, g):
    kd = [_bf16_bits(rng.standard_normal((hkv, n, D))) for n in lens]
    vd = [_bf16_bits(rng.standard_normal((hkv, n, D))) for n in lens]
    q = rng.standard_normal((len(lens), hkv * g, D))
    return kd, vd, q


def test_one_token_returns_v_exactly():
    rng = np.random.default_rng(0)
    kd, vd, q = _random_case(rng, [1, 1], hkv=2, g=3)
    pool, bt, lens = _scatter_pool(kd, vd, 8, rng)
    out = _decode(pool, bt, lens, q, 2)
    for b in range(2):
        for i in range(6):
            assert np.array_equal(out[b, i], oracle.bf16_to_double(vd[b][i // 3, 0]))


def test_identical_keys_give_mean_of_v():
    rng = np.random.default_rng(1)
    kd, vd, q = _random_case(rng, [37, 5], hkv=2, g=4)
    for b in range(2):
        kd[b][:] = kd[b][:, :1, :]          # every token shares one key
    pool, bt, lens = _scatter_pool(kd, vd, 16, rng)
    out = _decode(pool, bt, lens, q, 2)
    for b in range(2):
        for i in range(8):
            mean = oracle.bf16_to_double(vd[b][i // 4]).mean(axis=0)
            np.testing.assert_allclose(out[b, i], mean, rtol=0, atol=1e-14)


def test_zero_scale_gives_mean_of_v():
    rng = np.random.default_rng(2)
    kd, vd, q = _random_case(rng, [50], hkv=1, g=2)
    pool, bt, lens = _scatter_pool(kd, vd, 8, rng)
    out = _decode(pool, bt, lens, q, 1, scale=0.0)
    mean = oracle.bf16_to_double(vd[0][0]).mean(axis=0)
    np.testing.assert_allclose(out[0, 0], mean, rtol=0, atol=1e-14)
    np.testing.assert_allclose(out[0, 1], mean, rtol=0, atol=1e-14)


def test_two_tokens_closed_form():
    rng = np.random.default_rng(3)
    kd, vd, q = _random_case(rng, [2], hkv=1, g=1)
    pool, bt, lens = _scatter_pool(kd, vd, 4, rng)
    out = _decode(pool, bt, lens, q, 1)[0, 0]
    k = oracle.bf16_to_double(kd[0][0])
    v = oracle.bf16_to_double(vd[0][0])
    s0, s1 = (q[0, 0] @ k[0]) / 8, (q[0, 0] @ k[1]) / 8
    want = expit(s0 - s1) * v[0] + expit(s1 - s0) * v[1]
    np.testing.assert_allclose(out, want, rtol=1e-13, atol=1e-15)


def test_gqa_head_mapping():
    # Every V of KV head h equals h + 1, so query head i must return i // g + 1.
    rng = np.random.default_rng(4)
    hkv, g = 4, 3
    kd, vd, q = _random_case(rng, [21, 40], hkv=hkv, g=g)
    for b in range(2):
        for h in range(hkv):
            vd[b][h] = _bf16_bits(np.full(vd[b][h].shape, h + 1.0))
    pool, bt, lens = _scatter_pool(kd, vd, 16, rng)
    out = _decode(pool, bt, lens, q, hkv)
    for i in range(hkv * g):
        np.testing.assert_allclose(out[:, i], i // g + 1.0, rtol=1e-14)


def test_page_permutation_invariance_bitwise():
    rng = np.random.default_rng(5)
    kd, vd, q = _random_case(rng, [70, 33, 16], hkv=2, g=4)
    pool, bt, lens = _scatter_pool(kd, vd, 24, rng)
    out = _decode(pool, bt, lens, q, 2)
    # move every physical page somewhere else and remap the block table
    perm = rng.permutation(24)
    pool2 = np.empty_like(pool.reshape(24, -1))
    pool2[perm] = pool.reshape(24, -1)
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    out2 = _decode(pool2.reshape(-1), bt2, lens, q, 2)
    assert np.array_equal(out, out2)


@pytest.mark.parametrize("g", [1, 4, 7])
def test_brute_force_dense(g):
    rng = np.random.default_rng(10 + g)
    hkv = 2
    lens = rng.integers(1, 41, 3)
    kd, vd, q = _random_case(rng, lens, hkv=hkv, g=g)
    pool, bt, seq = _scatter_pool(kd, vd, 16, rng)
    out = _decode(pool, bt, seq, q, hkv)
    for b in range(3):
        for i in range(hkv * g):
            k = oracle.bf16_to_double(kd[b][i // g])
            v = oracle.bf16_to_double(vd[b][i // g])
            p = softmax(k @ q[b, i] / 8.0)
            np.testing.assert_allclose(out[b, i], p @ v, rtol=1e-12, atol=1e-14)


def test_large_scores_stay_finite_and_pick_argmax():
    rng = np.random.default_rng(6)
    kd, vd, q = _random_case(rng, [90], hkv=1, g=1)
    pool, bt, lens = _scatter_pool(kd, vd, 8, rng)
    out = _decode(pool, bt, lens, q * 1e4, 1)[0, 0]
    k = oracle.bf16_to_double(kd[0][0])
    v = oracle.bf16_to_double(vd[0][0])
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(out, v[np.argmax(k @ q[0, 0])], rtol=0, atol=1e-12)


@pytest.mark.parametrize("tps", [1, 7, 16, 100])
def test_split_then_combine_equals_unsplit(tps):
    rng = np.random.default_rng(20 + tps)
    kd, vd, q = _random_case(rng, [1, 45, 16, 130], hkv=2, g=4)
    pool, bt, lens = _scatter_pool(kd, vd, 24, rng)
    full = _decode(pool, bt, lens, q, 2)
    o, lse, ns = oracle.gqa_decode_split(pool, num_kv_heads=2, q_rot=q, block_tables=bt,
                                         max_blocks=bt.shape[1], seq_lens=lens, batch=4,
                                         num_q_heads=8, scale=1 / 8, tokens_per_split=tps)
    assert list(ns.reshape(4, 8)[:, 0]) == [-(-int(n) // tps) for n in lens]
    merged = oracle.lse_combine(o, lse, ns).reshape(full.shape)
    np.testing.assert_allclose(merged, full, rtol=1e-12, atol=1e-14)


def test_split_lse_is_log_partition():
    # lse of a one-split row is log(sum_t exp(s_t)) of that row's scores.
    rng = np.random.default_rng(30)
    kd, vd, q = _random_case(rng, [23], hkv=1, g=1)
    pool, bt, lens = _scatter_pool(kd, vd, 4, rng)
    o, lse, ns = oracle.gqa_decode_split(pool, num_kv_heads=1, q_rot=q, block_tables=bt,
                                         max_blocks=bt.shape[1], seq_lens=lens, batch=1,
                                         num_q_heads=1, scale=1 / 8, tokens_per_split=64)
    s = oracle.bf16_to_double(kd[0][0]) @ q[0, 0] / 8
    assert ns[0] == 1
    assert lse[0, 0] == pytest.approx(np.log(np.sum(np.exp(s))), rel=1e-14)


def test_combine_hand_example():
    # Two splits with lse 0 and ln 3: weights 1/4 and 3/4.
    a = np.arange(4, dtype=np.float64)
    b = np.ones(4) * 10
    o = np.stack([a, b])[None]                       # [1 row, 2 splits, D=4]
    lse = np.array([[0.0, np.log(3.0)]])
    out = oracle.lse_combine(o, lse, np.array([2], np.int32))
    np.testing.assert_allclose(out[0], a / 4 + 3 * b / 4, rtol=1e-15)
    # a single split comes back unchanged; unused slots are ignored
    out1 = oracle.lse_combine(o, np.array([[5.0, np.nan]]), np.array([1], np.int32))
    assert np.array_equal(out1[0], a)
