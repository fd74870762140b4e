"""GPU path vs the fp64 oracle, element by element, on small workloads.

Pool bytes after the append must match bit for bit; q_rot and the attention
output must match within the stated tolerances (atol 2e-4 + rtol 2e-3 for the
output). Cases span several pages and ragged tails, every group size the
decode supports, the page boundaries, a single long sequence split over many
warps, and a batch larger than one launch serves.
"""
import numpy as np
import pytest
import torch

import workloads
from tests.parity import DeviceWorkload, assert_close, oracle_layer, u16

pytestmark = pytest.mark.gpu

QROT_ATOL = 2e-5


def full_check(wl, pages_per_split=0, fused=True):
    """Both paths: the fused step (one call per layer) and append + decode."""
    if fused:
        full_check(wl, pages_per_split, fused=False)
    dw = DeviceWorkload(wl, pages_per_split)
    out = dw.run(fused=fused).cpu().numpy()
    assert dw.step.error_bits() == 0
    # the partials of segments split between CTAs are put back to zero: the
    # workspace holds nothing but what the step's plan alone writes there
    after = dw.step.workspace.clone()
    dw.step.workspace.zero_()
    dw.step.plan(fused)
    torch.cuda.synchronize()
    assert torch.equal(after, dw.step.workspace), "decode left workspace words set"
    pool_host = u16(wl.pool).reshape(-1).copy()
    q, k, v = u16(wl.q), u16(wl.k), u16(wl.v)
    q_rot_gpu = dw.step.q_rot.cpu().numpy()
    worst = 0.0
    for layer in range(wl.num_layers):
        q_rot, want = oracle_layer(pool_host, wl, layer, q[layer], k[layer], v[layer])
        np.testing.assert_allclose(q_rot_gpu[layer], q_rot, rtol=1e-5, atol=QROT_ATOL)
        worst = max(worst, assert_close(out[layer], want, f"{wl.name} layer {layer}"))
    got_pool = u16(dw.pool).reshape(-1)
    mism = np.flatnonzero(got_pool != pool_host)
    assert mism.size == 0, f"{mism.size} pool elements differ, first at {mism[:5]}"
    dw.step.close()
    return worst


@pytest.mark.parametrize("name", ["llama1b_b1_l1_len37", "llama1b_b8_l16_u512"])
@pytest.mark.parametrize("seed", [0, 1])
def test_named_small_workloads(name, seed):
    full_check(workloads.make(name, seed=seed, sentinel=True))


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (6, 2), (32, 8), (10, 2), (12, 2), (14, 2), (16, 2)])
def test_every_group_size(hq, hkv):
    cached = [0, 15, 16, 17, 31, 32, 100, 257]
    wl = workloads.build(f"g{hq // hkv}", batch=len(cached), num_layers=2, num_q_heads=hq,
                         num_kv_heads=hkv, cached_lens=cached, rope_theta=1e6, seed=hq,
                         sentinel=True)
    full_check(wl)


def test_page_boundaries_llama():
    cached = [0, 1, 14, 15, 16, 17, 47, 48, 49, 63, 64, 65]
    wl = workloads.build("bounds", batch=len(cached), num_layers=3, num_q_heads=32, num_kv_heads=8,
                         cached_lens=cached, rope_theta=500000.0, seed=3, sentinel=True)
    full_check(wl)


def test_single_long_sequence_split_many_ways():
    # one sequence of 5001 tokens: auto partitioning cuts each head's 313 pages
    # over many warps, so the merge combines dozens of pieces.
    wl = workloads.build("long", batch=1, num_layers=1, num_q_heads=32, num_kv_heads=8,
                         cached_lens=[5000], rope_theta=500000.0, seed=4, sentinel=True)
    full_check(wl)


def test_qwen_shape_long_context():
    wl = workloads.build("qwen", batch=3, num_layers=2, num_q_heads=14, num_kv_heads=2,
                         cached_lens=[1024, 4096, 2500], rope_theta=1e6, seed=5, sentinel=True)
    full_check(wl)


@pytest.mark.parametrize("hq,hkv", [(32, 8), (10, 2), (14, 2), (16, 2)])
def test_segment_over_many_ctas(hq, hkv):
    # one-page ranges: each head's 188 pages span about 19 CTAs, so the CTA of
    # the last one waits for 18 partials (for 5-8 heads staged in shared
    # memory in several batches, more than its page ring holds at once)
    wl = workloads.build("span", batch=2, num_layers=1, num_q_heads=hq, num_kv_heads=hkv,
                         cached_lens=[2999, 40], rope_theta=1e6, seed=hq + 7, sentinel=True)
    full_check(wl, pages_per_split=1)


@pytest.mark.parametrize("pps", [1, 2, 7, 64])
def test_split_invariance(pps):
    wl = workloads.make("llama1b_b8_l16_u512", seed=2, sentinel=True)
    full_check(wl, pages_per_split=pps)


def test_batch_larger_than_one_launch():
    rng = np.random.default_rng(6)
    cached = rng.integers(0, 40, 2100)
    wl = workloads.build("b2100", batch=2100, num_layers=1, num_q_heads=4, num_kv_heads=1,
                         cached_lens=cached, rope_theta=1e4, seed=6, sentinel=True)
    full_check(wl)
    full_check(wl, pages_per_split=1)


def test_many_tiny_sequences_repeat_deterministic():
    rng = np.random.default_rng(7)
    cached = rng.integers(0, 3, 300)
    wl = workloads.build("tiny", batch=300, num_layers=2, num_q_heads=32, num_kv_heads=8,
                         cached_lens=cached, rope_theta=500000.0, seed=7, sentinel=True)
    full_check(wl)
    # running the same step twice gives the same bytes (append is idempotent;
    # the decode's reduction order does not depend on timing)
    dw = DeviceWorkload(wl)
    a = dw.run().clone()
    b = dw.run().clone()
    assert torch.equal(a, b)
    dw.step.close()


def test_contiguous_page_placement():
    # every (layer, sequence) on consecutive pages: the contiguous-cache baseline's layout
    cached = [0, 15, 16, 100, 700, 1500]
    wl = workloads.build("contig", batch=len(cached), num_layers=3, num_q_heads=32, num_kv_heads=8,
                         cached_lens=cached, rope_theta=500000.0, seed=21, sentinel=True,
                         contiguous=True)
    assert (wl.block_tables[0, 4, 1:44] - wl.block_tables[0, 4, :43] == 1).all()
    full_check(wl)
