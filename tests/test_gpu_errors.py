"""Device-side argument checks: bad lengths and page ids are caught by the
kernels before any access, reported in the pool's error word, and leave the
rest of the batch correct. Every bad value here is rejected by an explicit
range check before it could index memory; no GPU fault is involved.
"""
import numpy as np
import pytest
import torch

import workloads
import paged_kv_decode_rope_gb300 as pkv
from tests.parity import DeviceWorkload, assert_close, oracle_layer, u16

pytestmark = pytest.mark.gpu


def _wl(seed=0):
    return workloads.build("err", batch=4, num_layers=1, num_q_heads=32, num_kv_heads=8,
                           cached_lens=[40, 70, 5, 100], rope_theta=500000.0, seed=seed,
                           sentinel=True)


def test_bad_sequence_length_is_flagged_and_zeroed():
    wl = _wl()
    dw = DeviceWorkload(wl)
    want_pool = u16(wl.pool).reshape(-1).copy()
    q, k, v = u16(wl.q)[0], u16(wl.k)[0], u16(wl.v)[0]
    good = np.array([0, 1, 3])
    _, want = oracle_layer(want_pool, wl, 0, q, k, v, seqs=good)
    bad_lens = wl.seq_lens.copy()
    bad_lens[2] = 0
    dw.step.seq_lens.copy_(torch.from_numpy(bad_lens))
    out = dw.run()[0].cpu().numpy()
    bits = dw.step.error_bits(reset=True)
    assert bits & pkv.ERR_SEQ_LEN
    assert np.all(out[2] == 0.0)
    assert_close(out[good], want, "good rows")
    # too long for the block table
    bad_lens[2] = wl.max_blocks * 16 + 1
    dw.step.seq_lens.copy_(torch.from_numpy(bad_lens))
    out = dw.run()[0].cpu().numpy()
    assert dw.step.error_bits(reset=True) & pkv.ERR_SEQ_LEN
    assert np.all(out[2] == 0.0)
    assert dw.step.error_bits() == 0
    dw.step.close()


def test_bad_page_id_is_flagged_and_skipped():
    wl = _wl(1)
    dw = DeviceWorkload(wl)
    bt = wl.block_tables.copy()
    bt[0, 1, 0] = wl.num_pages + 7      # first page of sequence 1
    bt[0, 3, 1] = -5                    # second page of sequence 3
    dw.step.block_tables.copy_(torch.from_numpy(bt))
    out = dw.run()[0]
    torch.cuda.synchronize()
    assert dw.step.error_bits(reset=True) & pkv.ERR_PAGE_ID
    assert bool(torch.isfinite(out).all())
    # untouched sequences still match the oracle
    want_pool = u16(wl.pool).reshape(-1).copy()
    _, want = oracle_layer(want_pool, wl, 0, u16(wl.q)[0], u16(wl.k)[0], u16(wl.v)[0],
                           seqs=np.array([0, 2]))
    assert_close(out.cpu().numpy()[[0, 2]], want, "sequences with valid pages")
    dw.step.close()


def test_bad_append_page_writes_nothing():
    wl = _wl(2)
    dw = DeviceWorkload(wl)
    bt = wl.block_tables.copy()
    t = wl.seq_lens[0] - 1
    bt[0, 0, t // 16] = -1
    dw.step.block_tables.copy_(torch.from_numpy(bt))
    before = dw.pool.clone()
    dw.step.append(0, dw.q, dw.k, dw.v)
    torch.cuda.synchronize()
    assert dw.step.error_bits(reset=True) & pkv.ERR_PAGE_ID
    # sequences 1..3 appended, sequence 0 wrote nothing: compare with the oracle on 1..3
    want_pool = u16(wl.pool).reshape(-1).copy()
    oracle_layer(want_pool, wl, 0, u16(wl.q)[0], u16(wl.k)[0], u16(wl.v)[0], seqs=np.array([1, 2, 3]))
    assert np.array_equal(u16(dw.pool).reshape(-1), want_pool)
    assert not torch.equal(before, dw.pool)
    dw.step.close()


def test_host_side_rejections():
    wl = _wl(3)
    dw = DeviceWorkload(wl)
    st = dw.step
    with pytest.raises(pkv.PkvError, match="EINVAL"):   # workspace too small
        pkv.paged_gqa_decode(st.pool, st.q_rot[0], st.out[0], st.block_tables[0], st.seq_lens,
                             0.125, st.workspace[:64])
    with pytest.raises(pkv.PkvError, match="EINVAL"):   # group 16 > 8
        q16 = torch.zeros(st.seq_lens.shape[0], 128, 64, device="cuda")
        pkv.paged_gqa_decode(st.pool, q16, q16.clone(), st.block_tables[0], st.seq_lens, 0.125,
                             st.workspace)
    with pytest.raises(pkv.PkvError, match="EINVAL"):   # theta
        pkv.paged_kv_append_rope(st.pool, dw.q[0], dw.k[0], dw.v[0], st.q_rot[0], st.block_tables[0],
                                 st.seq_lens, st.positions, -1.0)
    with pytest.raises(pkv.PkvError, match="ENOSPC"):
        pkv.kv_pool_create(torch.empty(100, dtype=torch.uint8, device="cuda"), 8)
    with pytest.raises(pkv.PkvError, match="EINVAL"):   # misaligned storage
        pkv.kv_pool_create(torch.empty(1 << 20, dtype=torch.uint8, device="cuda")[8:], 8)
    st.close()


def test_merge_wait_timeout_is_reported_and_recoverable():
    """The one wait on another CTA (a merger looking for the partials of a
    segment split across CTAs) is bounded. With the bound set to 0 looks every
    such merger gives up at once, so nothing waits: the error word gets
    ERR_TIMEOUT, those segments' rows stay unwritten, every other row is
    correct, and after the workspace is zeroed again a normal call is correct
    everywhere and leaves the workspace zero."""
    wl = workloads.build("timeout", batch=5, num_layers=1, num_q_heads=32, num_kv_heads=8,
                         cached_lens=[3000, 17, 1500, 4000, 260], rope_theta=500000.0, seed=21)
    dw = DeviceWorkload(wl)
    st = dw.step
    st.append(0, dw.q, dw.k, dw.v)
    want_pool = u16(wl.pool).reshape(-1).copy()
    _, want = oracle_layer(want_pool, wl, 0, u16(wl.q)[0], u16(wl.k)[0], u16(wl.v)[0])
    assert st.error_bits(reset=True) == 0

    prev = pkv.kv_pool_set_merge_wait_limit(st.pool, 0)
    assert prev == pkv.DEFAULT_MERGE_WAIT_LOOKS
    out = torch.full_like(st.out[0], float("nan"))
    pkv.paged_gqa_decode(st.pool, st.q_rot[0], out, st.block_tables[0], st.seq_lens, wl.scale,
                         st.workspace)
    torch.cuda.synchronize()
    assert st.error_bits(reset=True) == pkv.ERR_TIMEOUT
    got = out.cpu().numpy()
    unwritten = np.isnan(got).all(axis=-1)                     # [B, Hq]
    assert unwritten.any(), "no segment crossed CTAs: the timeout path did not run"
    assert not unwritten.all()
    # a row is written in full or not at all; the written ones are right
    assert not (np.isnan(got).any(axis=-1) & ~unwritten).any()
    assert_close(got[~unwritten], want[~unwritten], "rows whose merge did not time out")
    # rows of one (sequence, kv head) segment go together
    g = wl.num_q_heads // wl.num_kv_heads
    seg = unwritten.reshape(wl.batch, wl.num_kv_heads, g)
    assert (seg.all(axis=-1) | ~seg.any(axis=-1)).all()
    assert bool(st.workspace.any()), "the given-up merges left their partials behind"

    assert pkv.kv_pool_set_merge_wait_limit(st.pool, prev) == 0
    st.workspace.zero_()
    out.fill_(float("nan"))
    pkv.paged_gqa_decode(st.pool, st.q_rot[0], out, st.block_tables[0], st.seq_lens, wl.scale,
                         st.workspace)
    torch.cuda.synchronize()
    assert st.error_bits() == 0
    assert_close(out.cpu().numpy(), want, "after the workspace was zeroed again")
    assert not bool(st.workspace.any()), "a completed call leaves the workspace zero"
    st.close()


def test_position_past_the_rope_table_is_flagged_and_zeroed():
    """The fused step reads each new token's cos/sin from the row of its
    position in the RoPE table. A position the table has no row for skips
    the sequence: nothing appended, its output rows zeroed, ERR_POSITION set;
    the other sequences are correct."""
    wl = _wl(4)  # cached lengths 40, 70, 5, 100: positions 40, 70, 5, 100
    dw = DeviceWorkload(wl, rope_positions=80)  # no row for position 100
    before = dw.pool.clone()
    out = dw.run()[0].cpu().numpy()
    assert dw.step.error_bits(reset=True) == pkv.ERR_POSITION
    assert np.all(out[3] == 0.0)
    good = np.array([0, 1, 2])
    want_pool = u16(wl.pool).reshape(-1).copy()
    _, want = oracle_layer(want_pool, wl, 0, u16(wl.q)[0], u16(wl.k)[0], u16(wl.v)[0], seqs=good)
    assert_close(out[good], want, "sequences with a table row")
    assert np.array_equal(u16(dw.pool).reshape(-1), want_pool), "only sequences 0-2 appended"
    assert not torch.equal(before, dw.pool)
    dw.step.close()
