"""The split-KV partial results and the standalone log-sum-exp merge.

``paged_gqa_decode_partials`` leaves every (sequence, head) row's pieces for
``paged_kv_split_combine``. The piece count of each row is index work and must
match the partition exactly; each piece's normalised output and log-sum-exp
must match the oracle over that piece's tokens; the merged result must match
the oracle's unsplit attention. The merge kernel is also checked alone against
the oracle's closed-form merge, including empty and single-split rows.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import paged_kv_decode_rope_gb300 as pkv
from tests.parity import ATOL, RTOL, DeviceWorkload, assert_close, u16

pytestmark = pytest.mark.gpu


def _expected_pieces(wl, pps):
    """Piece ranges of every (b, h): list of (range index, first page, end page)."""
    np_b = (wl.seq_lens + 15) // 16
    pre = np.concatenate([[0], np.cumsum(np_b)])
    out = {}
    for b in range(wl.batch):
        for h in range(wl.num_kv_heads):
            s = wl.num_kv_heads * pre[b] + h * np_b[b]
            e = s + np_b[b]
            pieces = []
            for r in range(s // pps, (e - 1) // pps + 1):
                lo, hi = max(s, r * pps), min(e, (r + 1) * pps)
                pieces.append((lo - s, hi - s))
            out[(b, h)] = pieces
    return out


@pytest.mark.parametrize("pps", [1, 3, 16])
def test_partials_then_combine(pps):
    wl = workloads.make("llama1b_b8_l16_u512", seed=3, sentinel=True)
    wl.num_layers = 1
    wl.q, wl.k, wl.v = wl.q[:1], wl.k[:1], wl.v[:1]
    wl.block_tables = wl.block_tables[:1]
    dw = DeviceWorkload(wl)
    st = dw.step
    st.append(0, dw.q, dw.k, dw.v)
    rows = wl.batch * wl.num_q_heads
    ms = pkv.decode_max_splits(wl.max_blocks, pps)
    o_part = torch.full((rows, ms, 64), float("nan"), device="cuda")
    lse_part = torch.full((rows, ms), float("nan"), device="cuda")
    nsp = torch.full((rows,), -1, dtype=torch.int32, device="cuda")
    pkv.paged_gqa_decode_partials(st.pool, st.q_rot[0], st.block_tables[0], st.seq_lens, wl.scale,
                                  pps, o_part, lse_part, nsp)
    out = torch.empty(rows, 64, device="cuda")
    pkv.paged_kv_split_combine(o_part, lse_part, nsp, out)
    torch.cuda.synchronize()
    assert st.error_bits() == 0

    pool_host = u16(dw.pool).reshape(-1).copy()  # after the GPU append (bit-exact, checked elsewhere)
    q_rot = st.q_rot[0].double().cpu().numpy()
    want = oracle.gqa_decode(pool_host, num_kv_heads=wl.num_kv_heads, q_rot=q_rot,
                             block_tables=wl.block_tables[0], max_blocks=wl.max_blocks,
                             seq_lens=wl.seq_lens, batch=wl.batch, num_q_heads=wl.num_q_heads,
                             scale=wl.scale)
    assert_close(out.cpu().numpy().reshape(want.shape), want, f"combined pps={pps}")

    pieces = _expected_pieces(wl, pps)
    nsp_h = nsp.cpu().numpy().reshape(wl.batch, wl.num_q_heads)
    o_h, lse_h = o_part.cpu().numpy(), lse_part.cpu().numpy()
    g = wl.group
    for b in range(wl.batch):
        for h in range(wl.num_kv_heads):
            pl = pieces[(b, h)]
            assert np.all(nsp_h[b, h * g:(h + 1) * g] == len(pl))
            for j, (p0, p1) in enumerate(pl):
                # oracle over tokens [16 p0, min(16 p1, N)): a shifted view of the block table
                n_tok = min(16 * p1, int(wl.seq_lens[b])) - 16 * p0
                bt = np.full((1, wl.max_blocks), -1, np.int32)
                bt[0, :p1 - p0] = wl.block_tables[0, b, p0:p1]
                qr = q_rot[b:b + 1, h * g:(h + 1) * g]
                o_w, lse_w, _ = oracle.gqa_decode_split(
                    pool_host, num_kv_heads=wl.num_kv_heads,
                    q_rot=np.ascontiguousarray(np.tile(qr, (1, wl.num_kv_heads, 1))),
                    block_tables=bt, max_blocks=wl.max_blocks, seq_lens=np.array([n_tok], np.int32),
                    batch=1, num_q_heads=g * wl.num_kv_heads, scale=wl.scale,
                    tokens_per_split=wl.max_blocks * 16)
                # the tiled q puts query i of the group at row h*g + i, which reads kv head h
                for i in range(g):
                    row = b * wl.num_q_heads + h * g + i
                    assert_close(o_h[row, j], o_w[h * g + i, 0], f"piece o b={b} h={h} j={j}")
                    assert abs(lse_h[row, j] - lse_w[h * g + i, 0]) <= ATOL + RTOL * abs(lse_w[h * g + i, 0])
    st.close()


def test_combine_kernel_alone():
    rng = np.random.default_rng(0)
    rows, ms, d = 300, 9, 64
    o = rng.standard_normal((rows, ms, d)).astype(np.float32)
    lse = (rng.standard_normal((rows, ms)) * 20).astype(np.float32)
    ns = rng.integers(1, ms + 1, rows).astype(np.int32)
    ns[:5] = [0, ms + 1, -3, 1, ms]           # invalid counts -> zeros; single split; all splits
    lse[5, :] = -np.inf                         # every split empty -> zeros
    ns[5] = 3
    lse[6, 1] = -np.inf                         # one empty split among others
    ns[6] = 3
    out = torch.empty(rows, d, device="cuda")
    pkv.paged_kv_split_combine(torch.from_numpy(o).cuda(), torch.from_numpy(lse).cuda(),
                               torch.from_numpy(ns).cuda(), out)
    got = out.cpu().numpy()
    valid = (ns >= 1) & (ns <= ms)
    valid[5] = False
    want = oracle.lse_combine(o[valid].astype(np.float64), lse[valid].astype(np.float64), ns[valid])
    assert_close(got[valid], want, "combine")
    assert np.all(got[~valid] == 0.0)
    assert np.array_equal(got[3], o[3, 0])  # one split: returned as is


def test_combine_other_head_dims():
    rng = np.random.default_rng(1)
    for d in (1, 33, 128):
        o = rng.standard_normal((17, 4, d)).astype(np.float32)
        lse = rng.standard_normal((17, 4)).astype(np.float32)
        ns = rng.integers(1, 5, 17).astype(np.int32)
        out = torch.empty(17, d, device="cuda")
        pkv.paged_kv_split_combine(torch.from_numpy(o).cuda(), torch.from_numpy(lse).cuda(),
                                   torch.from_numpy(ns).cuda(), out)
        assert_close(out.cpu().numpy(), oracle.lse_combine(o.astype(np.float64),
                                                           lse.astype(np.float64), ns), f"d={d}")
