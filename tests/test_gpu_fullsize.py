"""The named full-size workloads, in the launch configuration the benchmark
times (automatic balancing over the persistent grid), checked against the
oracle on samples the oracle can compute one by one.

* Pool after the step: every element that changed lies in a new token's slot,
  and every new token's K/V row equals the oracle's bytes exactly.
* Output: sampled (layer, sequence) rows, including the longest and shortest
  sequence, match the oracle within atol 2e-4 + rtol 2e-3; every output is
  finite.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import DeviceWorkload, assert_close, gather_pages, u16

pytestmark = pytest.mark.gpu

FULL = ["llama1b_b8_l16_u512", "llama1b_b64_l16_u2048", "qwen05b_b32_l24_u1024_4096",
        "llama1b_b256_l16_skew"]


def _new_slot_rows(wl):
    """(layer, b) -> (page, slot) of the appended token."""
    t = wl.seq_lens - 1
    pages = wl.block_tables[:, np.arange(wl.batch), t // 16]  # [NL, B]
    return pages, t % 16


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(name):
    wl = workloads.make(name, seed=0, device="cuda")
    dw = DeviceWorkload(wl)
    before = wl.pool  # the generator's tensor stays untouched; dw.pool is a copy
    out = dw.run()
    assert dw.step.error_bits() == 0
    assert bool(torch.isfinite(out).all())
    hkv, nl, bsz = wl.num_kv_heads, wl.num_layers, wl.batch
    pool5 = dw.pool.view(wl.num_pages, hkv, 2, 16, 64)
    before5 = before.view(wl.num_pages, hkv, 2, 16, 64)

    # 1. only the new slots changed
    pages, slots = _new_slot_rows(wl)
    changed = (pool5 != before5).any(dim=-1).any(dim=2).any(dim=1)  # [pages, 16]
    expected = torch.zeros_like(changed)
    expected[torch.from_numpy(pages.reshape(-1)).cuda(),
             torch.from_numpy(np.tile(slots, nl)).cuda()] = True
    assert not bool((changed & ~expected).any()), "append wrote outside the new tokens' slots"

    # 2. the new rows equal the oracle's append, bit for bit
    q_all, k_all, v_all = u16(wl.q), u16(wl.k), u16(wl.v)
    for layer in range(nl):
        used = np.unique(pages[layer])
        remap = {int(p): i for i, p in enumerate(used)}
        mini = u16(before.view(wl.num_pages, -1)[torch.from_numpy(used).cuda()]).reshape(-1).copy()
        bt = np.full((bsz, wl.max_blocks), -1, np.int32)
        for b in range(bsz):
            bt[b, (wl.seq_lens[b] - 1) // 16] = remap[int(pages[layer, b])]
        oracle.append_rope(mini, num_kv_heads=hkv, q=q_all[layer], k=k_all[layer], v=v_all[layer],
                           block_tables=bt, max_blocks=wl.max_blocks, seq_lens=wl.seq_lens,
                           positions=wl.positions, batch=bsz, num_q_heads=wl.num_q_heads,
                           theta=wl.rope_theta)
        got = u16(pool5[torch.from_numpy(used).cuda()]).reshape(len(used), hkv, 2, 16, 64)
        want = mini.reshape(len(used), hkv, 2, 16, 64)
        for b in range(bsz):
            i, s = remap[int(pages[layer, b])], slots[b]
            assert np.array_equal(got[i, :, :, s], want[i, :, :, s]), f"layer {layer} seq {b}"

    # 3. sampled outputs: oracle append + decode from the pool as it was before the step
    rng = np.random.default_rng(1)
    layers = sorted({0, nl // 2, nl - 1})
    seqs = sorted({int(np.argmax(wl.seq_lens)), int(np.argmin(wl.seq_lens)),
                   *rng.choice(bsz, size=min(6, bsz), replace=False).tolist()})
    out_h = out.cpu().numpy()
    for layer in layers:
        mini, bt = gather_pages(before, wl, layer, seqs)
        sel = np.asarray(seqs)
        q_rot = oracle.append_rope(mini, num_kv_heads=hkv, q=q_all[layer][sel], k=k_all[layer][sel],
                                   v=v_all[layer][sel], block_tables=bt, max_blocks=wl.max_blocks,
                                   seq_lens=wl.seq_lens[sel], positions=wl.positions[sel],
                                   batch=len(sel), num_q_heads=wl.num_q_heads, theta=wl.rope_theta)
        want = oracle.gqa_decode(mini, num_kv_heads=hkv, q_rot=q_rot, block_tables=bt,
                                 max_blocks=wl.max_blocks, seq_lens=wl.seq_lens[sel], batch=len(sel),
                                 num_q_heads=wl.num_q_heads, scale=wl.scale)
        assert_close(out_h[layer][sel], want, f"{name} layer {layer}")
    dw.step.close()
