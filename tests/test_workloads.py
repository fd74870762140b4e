"""The input recipe (workloads.py) against what the workloads are stated to be:
shapes, length distributions, pool sizes, page assignment and the key-row
scaling. Host structure only for the full-size workloads (no pool tensor)."""
import math

import numpy as np
import pytest
import torch

import workloads

SHAPES = {
    "llama1b_b1_l1_len37": (1, 1, 32, 8, 500000.0),
    "llama1b_b8_l16_u512": (8, 16, 32, 8, 500000.0),
    "llama1b_b64_l16_u2048": (64, 16, 32, 8, 500000.0),
    "llama1b_b64_l16_u2048_contig": (64, 16, 32, 8, 500000.0),
    "qwen05b_b32_l24_u1024_4096": (32, 24, 14, 2, 1e6),
    "llama1b_b256_l16_skew": (256, 16, 32, 8, 500000.0),
}


def _pages_needed(wl):
    return (wl.seq_lens.astype(np.int64) + 15) // 16


@pytest.mark.parametrize("name", workloads.WORKLOADS)
@pytest.mark.parametrize("seed", [0, 3])
def test_named_workload_structure(name, seed):
    wl = workloads.make(name, seed=seed, materialize=False)
    batch, layers, hq, hkv, theta = SHAPES[name]
    assert (wl.batch, wl.num_layers, wl.num_q_heads, wl.num_kv_heads) == (batch, layers, hq, hkv)
    assert wl.rope_theta == theta and wl.scale == 1.0 / 8.0
    assert np.array_equal(wl.seq_lens, wl.cached_lens + 1)
    assert np.array_equal(wl.positions, wl.cached_lens)
    npg = _pages_needed(wl)
    assert wl.max_blocks >= npg.max()
    bt = wl.block_tables
    assert bt.shape == (layers, batch, wl.max_blocks)
    used = []
    for layer in range(layers):
        for b in range(batch):
            row = bt[layer, b]
            assert (row[:npg[b]] >= 0).all()
            if name != "llama1b_b1_l1_len37":  # that table is a full permutation on purpose
                assert (row[npg[b]:] == -1).all()
            used.append(row[:npg[b]])
    used = np.concatenate(used)
    assert used.max() < wl.num_pages
    assert np.unique(used).size == used.size, "a page is shared between (layer, sequence) rows"


def test_length_distributions():
    c = workloads.make("llama1b_b1_l1_len37", materialize=False).cached_lens
    assert c.tolist() == [37]
    for seed in range(4):
        c = workloads.make("llama1b_b8_l16_u512", seed=seed, materialize=False).cached_lens
        assert c.min() >= 1 and c.max() <= 512
        c = workloads.make("llama1b_b64_l16_u2048", seed=seed, materialize=False).cached_lens
        assert c.min() >= 1 and c.max() <= 2048
        c = workloads.make("qwen05b_b32_l24_u1024_4096", seed=seed, materialize=False).cached_lens
        assert c.min() >= 1024 and c.max() <= 4096
        c = workloads.make("llama1b_b256_l16_skew", seed=seed, materialize=False).cached_lens
        long_ = c >= 1024
        assert long_.sum() == 26 and (c[long_] <= 2048).all()
        assert ((c[~long_] >= 16) & (c[~long_] <= 256)).all()
        # interleaved, not 230 short then 26 long
        assert not (np.flatnonzero(long_) == np.arange(230, 256)).all()


def test_pool_sizes():
    assert workloads.make("llama1b_b1_l1_len37", materialize=False).num_pages == 64
    assert workloads.make("llama1b_b8_l16_u512", materialize=False).num_pages == 4096       # 128 MiB
    wl = workloads.make("llama1b_b64_l16_u2048", materialize=False)
    assert wl.num_pages == 81920 and wl.num_pages * 2 * 8 * 16 * 64 * 2 == 2.5 * 2**30  # 2.5 GiB
    for name in ("qwen05b_b32_l24_u1024_4096", "llama1b_b256_l16_skew"):
        wl = workloads.make(name, materialize=False)
        need = int(_pages_needed(wl).sum()) * wl.num_layers
        assert wl.num_pages == math.ceil(1.1 * need)


def test_block_table_of_the_single_sequence_is_a_permutation():
    wl = workloads.make("llama1b_b1_l1_len37", seed=5, materialize=False)
    assert sorted(wl.block_tables[0, 0].tolist()) == list(range(64))


def test_scattered_and_contiguous_placement():
    wl = workloads.make("llama1b_b64_l16_u2048", materialize=False)
    wc = workloads.make("llama1b_b64_l16_u2048_contig", materialize=False)
    assert np.array_equal(wl.cached_lens, wc.cached_lens)
    npg = _pages_needed(wc)
    runs_scattered = 0
    for layer in range(wc.num_layers):
        for b in range(wc.batch):
            row = wc.block_tables[layer, b, :npg[b]]
            assert (np.diff(row) == 1).all()
            runs_scattered += int((np.diff(wl.block_tables[layer, b, :npg[b]]) == 1).all())
    assert runs_scattered < wc.num_layers * wc.batch // 10  # the shuffled free list scatters pages


def test_profiling_copy_keeps_lengths_with_fewer_layers():
    full = workloads.make("llama1b_b64_l16_u2048", materialize=False)
    two = workloads.make("llama1b_b64_l16_u2048", layers=2, materialize=False)
    assert two.num_layers == 2 and np.array_equal(two.cached_lens, full.cached_lens)
    assert two.kv_bytes_per_layer() == full.kv_bytes_per_layer()
    assert two.num_pages == math.ceil(1.1 * int(_pages_needed(two).sum()) * 2)


def test_key_rows_scaled_by_eight():
    """About 10% of cached key rows and new key rows are exactly 8x the draw;
    values and queries are untouched."""
    kw = dict(batch=4, num_layers=2, num_q_heads=8, num_kv_heads=2, cached_lens=[300, 40, 511, 1],
              rope_theta=1e4, num_pages=400, seed=11)
    base = workloads.build("plain", **kw)
    big = workloads.build("big", big_key_frac=0.1, **kw)
    assert torch.equal(base.q, big.q) and torch.equal(base.v, big.v)
    pv = base.pool.view(400, 2, 2, 16, 64).float()
    bv = big.pool.view(400, 2, 2, 16, 64).float()
    assert torch.equal(pv[:, :, 1], bv[:, :, 1])                   # V untouched
    rows_same = (pv[:, :, 0] == bv[:, :, 0]).all(-1)
    rows_x8 = (pv[:, :, 0] * 8 == bv[:, :, 0]).all(-1)
    assert (rows_same | rows_x8).all()                             # every key row: as drawn or x8
    frac = (rows_x8 & ~rows_same).float().mean().item()
    assert 0.08 < frac < 0.12
    k_x8 = (base.k.float() * 8 == big.k.float()).all(-1) & ~(base.k == big.k).all(-1)
    assert ((base.k == big.k).all(-1) | k_x8).all()


def test_sentinel_marks_exactly_the_slots_without_a_cached_token():
    wl = workloads.build("s", batch=2, num_layers=1, num_q_heads=4, num_kv_heads=1,
                         cached_lens=[17, 3], rope_theta=1e4, num_pages=6, seed=2, sentinel=True)
    bits = wl.pool.view(torch.int16).view(6, 1, 2, 16, 64).numpy().view(np.uint16)
    is_sent = (bits == workloads.SENTINEL_BF16).all(axis=(1, 2, 4))  # [page][slot]
    assert torch.isnan(wl.pool.view(6, 1, 2, 16, 64).float()).all(dim=(1, 2, 4)).numpy().tolist() \
        == is_sent.tolist()                                          # the sentinel reads as NaN
    want = np.ones((6, 16), dtype=bool)
    for b, n in enumerate([17, 3]):
        for t in range(n):
            want[wl.block_tables[0, b, t // 16], t % 16] = False
    assert np.array_equal(is_sent, want)
