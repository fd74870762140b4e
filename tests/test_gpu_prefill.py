"""GPU chunked causal prefill (paged_prefill) against the oracle's prefill.

Chunks of new tokens after cached prefixes (start 0: a fresh prompt), across
page boundaries, several sequences per call, both model shapes; the pool must
match bit for bit, q_rot and the outputs within the decode tolerances.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_rope_gb300 as pkv
from tests.parity import assert_close, u16

pytestmark = pytest.mark.gpu


def _run(starts, lens, hq=32, hkv=8, theta=500000.0, seed=0, max_blocks=None, rows=None):
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    ends = [s + n for s, n in zip(starts, lens)]
    mb = max_blocks or max(1, -(-max(ends) // 16))
    need = sum(-(-e // 16) for e in ends)
    num_pages = need + 7
    page_elems = 2 * hkv * 16 * 64
    pool = torch.randn(num_pages * page_elems, generator=gen).to(torch.bfloat16)
    perm = rng.permutation(num_pages).astype(np.int32)
    bt = np.full((len(starts), mb), -1, np.int32)
    cur = 0
    for b, e in enumerate(ends):
        n = -(-e // 16)
        bt[b, :n] = perm[cur:cur + n]
        cur += n
    total = int(sum(lens))
    q = torch.randn(total, hq, 64, generator=gen).to(torch.bfloat16)
    k = torch.randn(total, hkv, 64, generator=gen).to(torch.bfloat16)
    v = torch.randn(total, hkv, 64, generator=gen).to(torch.bfloat16)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    st = np.asarray(starts, np.int32)
    scale = 1.0 / 8.0

    host = u16(pool).copy()
    want_qrot, want = oracle.prefill(host, num_kv_heads=hkv, q=u16(q), k=u16(k), v=u16(v),
                                     block_tables=bt, max_blocks=mb, cu_tokens=cu, start_pos=st,
                                     num_q_heads=hq, theta=theta, scale=scale)

    dev = torch.device("cuda")
    dpool = pool.to(dev)
    kp = pkv.kv_pool_create(dpool, hkv)
    q_rot = torch.empty(total, hq, 64, device=dev)
    out = torch.empty(total, hq, 64, device=dev)
    ws = pkv.alloc_prefill_workspace(total, len(starts), mb, device=dev)
    d_cu, d_st = torch.from_numpy(cu).to(dev), torch.from_numpy(st).to(dev)
    # the position table, built once (default: every position the block tables hold)
    rope = pkv.build_rope_table(theta, rows or mb * 16, device=dev)
    pkv.paged_prefill(kp, q.to(dev), k.to(dev), v.to(dev), q_rot, out, torch.from_numpy(bt).to(dev),
                      d_cu, d_st, rope, scale, ws)
    torch.cuda.synchronize()
    assert pkv.pkv_get_error(kp) == 0
    got_pool = u16(dpool)
    mism = np.flatnonzero(got_pool != host)
    assert mism.size == 0, f"{mism.size} pool elements differ, first at {mism[:5]}"
    np.testing.assert_allclose(q_rot.cpu().numpy(), want_qrot, rtol=1e-5, atol=2e-5)
    assert_close(out.cpu().numpy(), want, f"prefill starts={starts} lens={lens}")
    kp.close()


def test_fresh_prompt():
    _run([0], [37])


def test_chunk_after_cached_prefix_across_pages():
    _run([100], [50], seed=1)


def test_several_sequences_one_token_chunk_included():
    _run([0, 17, 300, 64], [16, 1, 45, 33], seed=2)


def test_qwen_shape():
    _run([5, 0], [40, 70], hq=14, hkv=2, theta=1e6, seed=3)


def test_long_prompt_many_tiles():
    _run([0], [600], seed=4)


def test_tiles_after_a_prefix_ending_mid_page():
    _run([100, 7], [70, 33], seed=6)


def test_rope_table_exactly_as_long_as_the_positions():
    _run([0, 17, 300, 64], [16, 1, 45, 33], seed=10, rows=345)
    _run([5, 0], [40, 70], hq=14, hkv=2, theta=1e6, seed=11, rows=70)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (12, 4), (10, 2), (12, 2), (64, 8)])
def test_every_group_size(hq, hkv):
    _run([3, 40], [35, 20], hq=hq, hkv=hkv, seed=7 + hq)


def test_malformed_chunk_is_flagged_and_zeroed():
    dev = torch.device("cuda")
    hkv, hq = 8, 32
    pool = torch.zeros(8 * 2 * hkv * 16 * 64, dtype=torch.bfloat16, device=dev)
    kp = pkv.kv_pool_create(pool, hkv)
    q = torch.randn(4, hq, 64, device=dev).to(torch.bfloat16)
    k = torch.randn(4, hkv, 64, device=dev).to(torch.bfloat16)
    v = torch.randn(4, hkv, 64, device=dev).to(torch.bfloat16)
    bt = torch.arange(2, dtype=torch.int32, device=dev).view(1, 2)
    q_rot = torch.empty(4, hq, 64, device=dev)
    out = torch.full((4, hq, 64), 7.0, device=dev)
    ws = pkv.alloc_prefill_workspace(4, 1, 2, device=dev)
    rope = pkv.build_rope_table(500000.0, 64, device=dev)
    # start 30 + 4 tokens needs positions up to 33 > 2 pages * 16: the last two are malformed
    pkv.paged_prefill(kp, q, k, v, q_rot, out, bt, torch.tensor([0, 4], dtype=torch.int32, device=dev),
                      torch.tensor([30], dtype=torch.int32, device=dev), rope, 0.125, ws)
    torch.cuda.synchronize()
    assert pkv.pkv_get_error(kp, reset=True) == pkv.ERR_SEQ_LEN
    assert (out[2:] == 0).all() and torch.isfinite(out[:2]).all() and (out[:2] != 7.0).any()
    kp.close()


def test_position_past_the_rope_table_is_flagged_and_zeroed():
    """Tokens at positions the RoPE table has no row for are not stored, their
    rows are zeroed and ERR_POSITION is set; the earlier tokens are right."""
    dev = torch.device("cuda")
    hkv, hq, theta = 8, 32, 500000.0
    gen = torch.Generator().manual_seed(8)
    pool = torch.randn(4 * 2 * hkv * 16 * 64, generator=gen).to(torch.bfloat16)
    t = 20
    q = torch.randn(t, hq, 64, generator=gen).to(torch.bfloat16)
    k = torch.randn(t, hkv, 64, generator=gen).to(torch.bfloat16)
    v = torch.randn(t, hkv, 64, generator=gen).to(torch.bfloat16)
    bt = np.array([[2, 0]], np.int32)
    cu, st = np.array([0, t], np.int32), np.array([0], np.int32)
    rows = 15  # positions 0..14 have a row; tokens 15..19 do not
    host = u16(pool).copy()
    _, want = oracle.prefill(host, num_kv_heads=hkv, q=u16(q)[:rows], k=u16(k)[:rows],
                             v=u16(v)[:rows], block_tables=bt, max_blocks=2,
                             cu_tokens=np.array([0, rows], np.int32), start_pos=st, num_q_heads=hq,
                             theta=theta, scale=0.125)
    dpool = pool.to(dev)
    kp = pkv.kv_pool_create(dpool, hkv)
    q_rot = torch.empty(t, hq, 64, device=dev)
    out = torch.full((t, hq, 64), 7.0, device=dev)
    ws = pkv.alloc_prefill_workspace(t, 1, 2, device=dev)
    pkv.paged_prefill(kp, q.to(dev), k.to(dev), v.to(dev), q_rot, out, torch.from_numpy(bt).to(dev),
                      torch.from_numpy(cu).to(dev), torch.from_numpy(st).to(dev),
                      pkv.build_rope_table(theta, rows, device=dev), 0.125, ws)
    torch.cuda.synchronize()
    assert pkv.pkv_get_error(kp, reset=True) == pkv.ERR_POSITION
    got = out.cpu().numpy()
    assert np.all(got[rows:] == 0.0)
    assert_close(got[:rows], want, "tokens with a table row")
    assert np.array_equal(u16(dpool), host), "only the tokens with a table row are stored"
    kp.close()


def test_bad_page_id_is_flagged_and_masked():
    """A block-table entry outside the pool: the page is neither written nor
    read (its keys get no weight), the error bit is set, outputs stay finite."""
    dev = torch.device("cuda")
    hkv, hq = 8, 32
    gen = torch.Generator().manual_seed(9)
    pool = torch.randn(16 * 2 * hkv * 16 * 64, generator=gen).to(torch.bfloat16).to(dev)
    kp = pkv.kv_pool_create(pool, hkv)
    t = 70
    q = torch.randn(t, hq, 64, generator=gen).to(torch.bfloat16).to(dev)
    k = torch.randn(t, hkv, 64, generator=gen).to(torch.bfloat16).to(dev)
    v = torch.randn(t, hkv, 64, generator=gen).to(torch.bfloat16).to(dev)
    bt = torch.tensor([[3, 7, 99, 1, 5]], dtype=torch.int32, device=dev)  # page 2 of 5 is bad
    q_rot = torch.empty(t, hq, 64, device=dev)
    out = torch.empty(t, hq, 64, device=dev)
    ws = pkv.alloc_prefill_workspace(t, 1, 5, device=dev)
    pkv.paged_prefill(kp, q, k, v, q_rot, out, bt, torch.tensor([0, t], dtype=torch.int32, device=dev),
                      torch.tensor([0], dtype=torch.int32, device=dev),
                      pkv.build_rope_table(500000.0, 80, device=dev), 0.125, ws)
    torch.cuda.synchronize()
    assert pkv.pkv_get_error(kp, reset=True) & pkv.ERR_PAGE_ID
    assert torch.isfinite(out).all()
    kp.close()


def _oracle_prefill_threaded(host, bt, cu, starts, q, k, v, hq, hkv, theta, scale, workers=16):
    """The oracle's prefill by its definition, spread over threads: every chunk
    token is appended exactly as a one-token decode append at its position
    (one oracle append call over all tokens as one-token sequences), then
    token t of sequence b attends, like one decode, over the sequence's first
    start + t + 1 tokens; the causal prefixes only read slots that earlier
    tokens wrote, so the decodes run in parallel batches. (That a prefill
    equals this composition is pinned in tests/test_oracle_prefill.py.)"""
    import concurrent.futures
    total = int(cu[-1])
    seq_of = np.repeat(np.arange(len(starts)), np.diff(cu))
    pos = (np.asarray(starts)[seq_of] + np.arange(total) - cu[seq_of]).astype(np.int32)
    tbt = np.ascontiguousarray(bt[seq_of])
    q_rot = oracle.append_rope(host, num_kv_heads=hkv, q=q, k=k, v=v, block_tables=tbt,
                               max_blocks=bt.shape[1], seq_lens=pos + 1, positions=pos,
                               batch=total, num_q_heads=hq, theta=theta)
    out = np.empty_like(q_rot)

    def part(lo, hi):
        out[lo:hi] = oracle.gqa_decode(host, num_kv_heads=hkv, q_rot=q_rot[lo:hi],
                                       block_tables=tbt[lo:hi], max_blocks=bt.shape[1],
                                       seq_lens=pos[lo:hi] + 1, batch=hi - lo, num_q_heads=hq,
                                       scale=scale)

    # longer prefixes cost more: interleave the token ranges over the threads
    edges = np.linspace(0, total, 8 * workers + 1).astype(int)
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(lambda i: part(edges[i], edges[i + 1]), range(len(edges) - 1)))
    return q_rot, out


@pytest.mark.parametrize("nb,t", [(4, 2048), (1, 8192)])
def test_measured_prefill_sizes_every_row(nb, t):
    """The prompt sizes the benchmark measures (Llama-3.2-1B shape, fresh
    prompts, one layer): the whole pool bit for bit, q_rot and every output
    row of every token and head within the decode tolerances."""
    hq, hkv, theta, scale = 32, 8, 500000.0, 0.125
    gen = torch.Generator().manual_seed(40 + nb)
    rng = np.random.default_rng(40 + nb)
    mb = -(-t // 16)
    num_pages = nb * mb + 5
    pool = torch.randn(num_pages * 2 * hkv * 16 * 64, generator=gen).to(torch.bfloat16)
    bt = rng.permutation(num_pages)[:nb * mb].astype(np.int32).reshape(nb, mb)
    total = nb * t
    q = torch.randn(total, hq, 64, generator=gen).to(torch.bfloat16)
    k = torch.randn(total, hkv, 64, generator=gen).to(torch.bfloat16)
    v = torch.randn(total, hkv, 64, generator=gen).to(torch.bfloat16)
    cu = np.arange(0, total + 1, t, dtype=np.int32)
    starts = np.zeros(nb, np.int32)

    dev = torch.device("cuda")
    dpool = pool.to(dev)
    kp = pkv.kv_pool_create(dpool, hkv)
    q_rot = torch.empty(total, hq, 64, device=dev)
    out = torch.empty(total, hq, 64, device=dev)
    ws = pkv.alloc_prefill_workspace(total, nb, mb, device=dev)
    d_cu, d_st = torch.from_numpy(cu).to(dev), torch.from_numpy(starts).to(dev)
    rope = pkv.build_rope_table(theta, t, device=dev)
    pkv.paged_prefill(kp, q.to(dev), k.to(dev), v.to(dev), q_rot, out, torch.from_numpy(bt).to(dev),
                      d_cu, d_st, rope, scale, ws)
    torch.cuda.synchronize()
    assert pkv.pkv_get_error(kp) == 0

    host = u16(pool).copy()
    want_qrot, want = _oracle_prefill_threaded(host, bt, cu, starts, u16(q), u16(k), u16(v), hq,
                                               hkv, theta, scale)
    mism = np.flatnonzero(u16(dpool) != host)
    assert mism.size == 0, f"{mism.size} pool elements differ, first at {mism[:5]}"
    np.testing.assert_allclose(q_rot.cpu().numpy(), want_qrot, rtol=1e-5, atol=2e-5)
    assert_close(out.cpu().numpy(), want, f"prefill {nb} x {t}")
    kp.close()


def test_misaligned_query_is_rejected():
    """The append reads the queries in 8-byte pieces: a q that does not start
    on a 16-byte boundary is refused with EINVAL before any launch."""
    dev = torch.device("cuda")
    hkv, hq, t = 8, 32, 4
    pool = torch.zeros(8 * 2 * hkv * 16 * 64, dtype=torch.bfloat16, device=dev)
    kp = pkv.kv_pool_create(pool, hkv)
    flat = torch.zeros(t * hq * 64 + 1, dtype=torch.bfloat16, device=dev)
    q = flat[1:].view(t, hq, 64)  # contiguous, 2 bytes past a 16-byte boundary
    k = torch.zeros(t, hkv, 64, dtype=torch.bfloat16, device=dev)
    v = torch.zeros(t, hkv, 64, dtype=torch.bfloat16, device=dev)
    q_rot = torch.empty(t, hq, 64, device=dev)
    out = torch.full((t, hq, 64), 5.0, device=dev)
    ws = pkv.alloc_prefill_workspace(t, 1, 1, device=dev)
    with pytest.raises(pkv.PkvError) as ei:
        pkv.paged_prefill(kp, q, k, v, q_rot, out, torch.zeros(1, 1, dtype=torch.int32, device=dev),
                          torch.tensor([0, t], dtype=torch.int32, device=dev),
                          torch.zeros(1, dtype=torch.int32, device=dev),
                          pkv.build_rope_table(500000.0, 16, device=dev), 0.125, ws)
    assert ei.value.rc == -22
    torch.cuda.synchronize()
    assert torch.all(out == 5.0), "nothing ran"
    kp.close()
