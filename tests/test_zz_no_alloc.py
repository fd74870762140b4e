"""paged_gqa_decode_no_alloc: the decode for callers that cannot allocate.

Some callers may not call cudaMalloc (a host framework whose memory manager
owns all device memory, a plugin handed only its inputs and outputs); this
entry point uses a fixed scratch array inside the library instead of a caller
workspace. Its results must equal paged_gqa_decode's, within the tolerance the
parity tests use, on two calls in a row (the array keeps the previous call's
contents). The workload has long sequences, so the split pieces, their
counters and their merges all go through the fixed array.

This file is collected last so that a run stopping at its first failure has
already run every other test.
"""
import numpy as np
import pytest
import torch

import workloads
import paged_kv_decode_rope_gb300 as pkv
from tests.parity import ATOL, RTOL, DeviceWorkload

pytestmark = pytest.mark.gpu


def test_no_alloc_matches_workspace_decode_twice():
    wl = workloads.build("noalloc", batch=5, num_layers=1, num_q_heads=32, num_kv_heads=8,
                         cached_lens=[3000, 17, 1500, 4000, 260], rope_theta=500000.0, seed=11)
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
        assert np.all(np.isfinite(g)), f"call {call}: non-finite output"
        bad = np.abs(g - r) > ATOL + RTOL * np.abs(r)
        assert not bad.any(), f"call {call}: {int(bad.sum())} elements differ from paged_gqa_decode"
    assert st.error_bits() == 0
    st.close()


def test_no_alloc_rejects_sizes_beyond_the_array():
    wl = workloads.build("noalloc_big", batch=2, num_layers=1, num_q_heads=8, num_kv_heads=8,
                         cached_lens=[20, 20], rope_theta=1e4, seed=12)
    dw = DeviceWorkload(wl)
    st = dw.step
    # one page per range over a huge block table needs more scratch than the array holds
    big_bt = torch.zeros(2, 1 << 16, dtype=torch.int32, device="cuda")
    need = pkv.paged_gqa_decode_workspace_bytes(2, 8, 8, 1 << 16, 1)
    assert need > (8 << 20)
    with pytest.raises(pkv.PkvError, match="E2BIG"):
        pkv.paged_gqa_decode_no_alloc(st.pool, st.q_rot[0], st.out[0], big_bt, st.seq_lens,
                                      wl.scale, pages_per_split=1)
    st.close()
