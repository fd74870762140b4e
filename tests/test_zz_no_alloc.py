"""paged_gqa_decode_no_alloc: the decode for callers that cannot allocate.

Some callers may not call cudaMalloc: code under a host framework whose
memory manager owns all device memory, or a plugin that is handed only its
inputs and outputs. This entry point takes no workspace; its scratch is a
fixed array inside the library, shared by every call. The tests check that
its output matches the fp64 oracle and the workspace entry point
(paged_gqa_decode) within the parity tolerance on two calls in a row (the
array keeps what the previous call left in it); that a call which timed out
and left partials in the array does not spoil the next one; and that sizes
beyond the array are rejected. The workload has long sequences, so split
pieces and their tagged partial slots go through the array.

This file is collected last so that a run stopping at its first failure has
already run every other test.
"""
import numpy as np
import pytest
import torch

import workloads
import paged_kv_decode_rope_gb300 as pkv
from tests.parity import ATOL, RTOL, DeviceWorkload, assert_close, oracle_layer, u16

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 8 << 20  # PKV_NO_ALLOC_SCRATCH_BYTES


def _long_workload(name, seed):
    return workloads.build(name, batch=5, num_layers=1, num_q_heads=32, num_kv_heads=8,
                           cached_lens=[3000, 17, 1500, 4000, 260], rope_theta=500000.0, seed=seed)


def _expected(wl):
    pool = u16(wl.pool).reshape(-1).copy()
    _, want = oracle_layer(pool, wl, 0, u16(wl.q)[0], u16(wl.k)[0], u16(wl.v)[0])
    return want


def test_no_alloc_matches_oracle_and_workspace_decode_twice():
    wl = _long_workload("noalloc", 11)
    want = _expected(wl)
    dw = DeviceWorkload(wl)
    st = dw.step
    st.append(0, dw.q, dw.k, dw.v)
    ref = torch.empty_like(st.out[0])
    pkv.paged_gqa_decode(st.pool, st.q_rot[0], ref, st.block_tables[0], st.seq_lens, wl.scale,
                         st.workspace)
    for call in range(2):
        got = torch.full_like(ref, float("nan"))
        pkv.paged_gqa_decode_no_alloc(st.pool, st.q_rot[0], got, st.block_tables[0], st.seq_lens,
                                      wl.scale)
        torch.cuda.synchronize()
        g, r = got.cpu().numpy(), ref.cpu().numpy()
        assert_close(g, want, f"call {call} against the oracle")
        bad = np.abs(g - r) > ATOL + RTOL * np.abs(r)
        assert not bad.any(), f"call {call}: {int(bad.sum())} elements differ from paged_gqa_decode"
    assert st.error_bits() == 0
    st.close()


def test_no_alloc_recovers_after_a_call_that_timed_out():
    """A merger that gives up (wait bound 0 looks: no waiting at all) leaves
    its partials in the array; the next call clears what it uses first."""
    wl = _long_workload("noalloc_dirty", 13)
    want = _expected(wl)
    dw = DeviceWorkload(wl)
    st = dw.step
    st.append(0, dw.q, dw.k, dw.v)
    prev = pkv.kv_pool_set_merge_wait_limit(st.pool, 0)
    out = torch.full_like(st.out[0], float("nan"))
    pkv.paged_gqa_decode_no_alloc(st.pool, st.q_rot[0], out, st.block_tables[0], st.seq_lens,
                                  wl.scale)
    torch.cuda.synchronize()
    assert st.error_bits(reset=True) == pkv.ERR_TIMEOUT  # the array now holds stale partials
    pkv.kv_pool_set_merge_wait_limit(st.pool, prev)
    for call in range(2):
        out.fill_(float("nan"))
        pkv.paged_gqa_decode_no_alloc(st.pool, st.q_rot[0], out, st.block_tables[0], st.seq_lens,
                                      wl.scale)
        torch.cuda.synchronize()
        assert st.error_bits() == 0
        assert_close(out.cpu().numpy(), want, f"call {call} after the timed-out one")
    st.close()


def test_no_alloc_scratch_covers_automatic_splits_at_any_batch():
    """With automatic splitting the scratch a call needs is the partial slots
    (two per warp of the grid: the GPU's SMs and the group size) plus a plan
    area of a few KB per thousand sequences: it fits the array for every
    group size and batch on this GPU."""
    for g, hkv in ((1, 8), (4, 8), (7, 2), (8, 4)):
        for b in (1, 64, 2048, 5000):
            need = pkv.paged_gqa_decode_workspace_bytes(b, g * hkv, hkv, 129)
            assert 0 < need <= SCRATCH_BYTES, f"group {g}, batch {b}: {need}"


def test_no_alloc_rejects_sizes_beyond_the_array():
    wl = workloads.build("noalloc_big", batch=2, num_layers=1, num_q_heads=8, num_kv_heads=8,
                         cached_lens=[20, 20], rope_theta=1e4, seed=12)
    dw = DeviceWorkload(wl)
    st = dw.step
    # one page per range over a huge block table needs more scratch than the array holds
    big_bt = torch.zeros(2, 1 << 16, dtype=torch.int32, device="cuda")
    need = pkv.paged_gqa_decode_workspace_bytes(2, 8, 8, 1 << 16, 1)
    assert need > SCRATCH_BYTES
    with pytest.raises(pkv.PkvError, match="E2BIG"):
        pkv.paged_gqa_decode_no_alloc(st.pool, st.q_rot[0], st.out[0], big_bt, st.seq_lens,
                                      wl.scale, pages_per_split=1)
    st.close()
