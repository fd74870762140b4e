"""The named full-size workloads, in the launch configuration the benchmark
times (automatic balancing over the persistent grid, the fused step without
the optional rotated-query output), checked against the fp64 oracle in full.

For every layer the oracle takes that layer's pages as they were before the
step, appends every sequence's new token and attends over every sequence;
then
* pool: every page of that layer equals the oracle's bit for bit (the new
  slots and everything around them), and pages no layer uses are untouched;
* output: every (sequence, query head) row of that layer is within
  atol 2e-4 + rtol 2e-3 of the oracle, element by element.
The oracle stays single-threaded per call; the layers run in a thread pool
(the oracle's C calls release the interpreter lock).
"""
import concurrent.futures
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import DeviceWorkload, assert_close, u16

pytestmark = pytest.mark.gpu

FULL = ["llama1b_b8_l16_u512", "llama1b_b64_l16_u2048", "qwen05b_b32_l24_u1024_4096",
        "llama1b_b256_l16_skew"]


def _layer_check(wl, layer, before_pages, after_pages, used, q, k, v, out_layer):
    """Oracle append + decode of every sequence of one layer on a compact copy
    of its pages; returns (pool bytes equal, max |err|) or raises."""
    remap = np.full(wl.num_pages, -1, dtype=np.int64)
    remap[used] = np.arange(len(used))
    bt = wl.block_tables[layer]
    bt2 = np.where(bt >= 0, remap[np.maximum(bt, 0)], -1).astype(np.int32)
    mini = before_pages.reshape(-1).copy()
    q_rot = oracle.append_rope(mini, num_kv_heads=wl.num_kv_heads, q=q, k=k, v=v, block_tables=bt2,
                               max_blocks=wl.max_blocks, seq_lens=wl.seq_lens,
                               positions=wl.positions, batch=wl.batch, num_q_heads=wl.num_q_heads,
                               theta=wl.rope_theta)
    want = oracle.gqa_decode(mini, num_kv_heads=wl.num_kv_heads, q_rot=q_rot, block_tables=bt2,
                             max_blocks=wl.max_blocks, seq_lens=wl.seq_lens, batch=wl.batch,
                             num_q_heads=wl.num_q_heads, scale=wl.scale)
    same = np.array_equal(mini, after_pages.reshape(-1))
    err = assert_close(out_layer, want, f"{wl.name} layer {layer}")
    return same, err


@pytest.mark.parametrize("name", FULL)
def test_full_size_every_row(name):
    wl = workloads.make(name, seed=0, device="cuda")
    dw = DeviceWorkload(wl, fused_q_rot=False)
    before = wl.pool  # the generator's tensor stays untouched; dw.pool is a copy
    out = dw.run()
    assert dw.step.error_bits() == 0
    out_h = out.cpu().numpy()
    assert np.all(np.isfinite(out_h))
    nl = wl.num_layers
    pages_before = before.view(wl.num_pages, -1)
    pages_after = dw.pool.view(wl.num_pages, -1)

    # pages that no layer uses are untouched
    used_any = np.zeros(wl.num_pages, dtype=bool)
    bt_all = wl.block_tables
    used_any[bt_all[bt_all >= 0]] = True
    idle = torch.from_numpy(np.flatnonzero(~used_any)).cuda()
    if idle.numel():
        assert torch.equal(pages_before[idle], pages_after[idle]), "a page no layer uses changed"

    q_all, k_all, v_all = u16(wl.q), u16(wl.k), u16(wl.v)
    jobs = []
    workers = max(1, min(16, os.cpu_count() or 1))
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
        for layer in range(nl):
            bt = wl.block_tables[layer]
            used = np.unique(bt[bt >= 0])
            idx = torch.from_numpy(used).cuda()
            jobs.append((layer, ex.submit(_layer_check, wl, layer, u16(pages_before[idx]),
                                          u16(pages_after[idx]), used, q_all[layer], k_all[layer],
                                          v_all[layer], out_h[layer])))
        worst = 0.0
        for layer, fut in jobs:
            same, err = fut.result()
            assert same, f"{name} layer {layer}: pool pages differ from the oracle's append"
            worst = max(worst, err)
    print(f"{name}: {nl} layers x {wl.batch} sequences x {wl.num_q_heads} heads, "
          f"max |err| {worst:.3g}")
    dw.step.close()
