"""A multi-step continuous-batching decode trace against the oracle.

The page scheduler admits requests under their budgets (a small pool forces
waits) and hands out pages lazily; the admitted prompts are prefilled through
the C ABI (in calls of a bounded token count, long prompts split into chunks
over several calls), then every decode step runs the fused step for the
active batch, whose sequences cross page boundaries. The test mirrors the
trace on a host copy of the pool with the oracle (each prefill call, then each
step's append and decode), checks every prefill and step output within the
tolerance, and the whole pool bit for bit at the end (pages reused after
release included).
"""
import numpy as np
import pytest

import oracle
import workloads
from tests.parity import assert_close, u16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("static,prefill_tokens", [(False, 8192), (True, 8192), (False, 48)])
def test_trace_matches_oracle_step_by_step(static, prefill_tokens):
    from paged_kv_decode_rope_gb300.trace import DecodeTrace
    hq, hkv, nl, theta, seed = 32, 8, 2, 500000.0, 4
    reqs = [workloads.TraceRequest(p, m, s) for p, m, s in
            [(5, 40, 40), (100, 20, 7), (16, 33, 33), (47, 18, 18), (31, 2, 2), (1, 25, 25),
             (64, 1, 1), (200, 30, 12)]]
    # 64 pages = 2 layers x 32: budgets of 4..15 pages per layer, so requests wait
    tr = DecodeTrace(reqs, num_pages=64, num_layers=nl, num_q_heads=hq, num_kv_heads=hkv,
                     rope_theta=theta, seed=seed, static_batching=static, max_batch=8,
                     prefill_tokens=prefill_tokens,
                     prompt_qkv=lambda r, n: workloads.trace_prompt_qkv(seed, r, nl, hq, hkv, n),
                     step_qkv=lambda r, s: workloads.trace_step_qkv(seed, r, s, nl, hq, hkv))
    page_elems = 2 * hkv * 16 * 64
    host = np.zeros(64 * page_elems, dtype=np.uint16)
    checked = {"steps": 0, "worst": 0.0, "calls": 0, "split": 0}

    def on_prefill(chunks, inputs, q_rot, out):
        cu, start, bt, q, k, v = inputs
        checked["split"] += sum(1 for c in chunks if c[1] > 0)
        got_qrot, got = q_rot.cpu().numpy(), out.cpu().numpy()
        for layer in range(nl):
            want_qrot, want = oracle.prefill(host, num_kv_heads=hkv, q=u16(q[layer]), k=u16(k[layer]),
                                             v=u16(v[layer]), block_tables=bt[layer],
                                             max_blocks=bt.shape[-1], cu_tokens=cu, start_pos=start,
                                             num_q_heads=hq, theta=theta, scale=1.0 / 8.0)
            np.testing.assert_allclose(got_qrot[layer], want_qrot, rtol=1e-5, atol=2e-5)
            checked["worst"] = max(checked["worst"],
                                   assert_close(got[layer], want, f"prefill {checked['calls']} layer {layer}"))
        checked["calls"] += 1

    def on_step(batch, inputs, out):
        pos, seq_lens, bt, q, k, v = inputs
        got = out.cpu().numpy()
        for layer in range(nl):
            q_rot = oracle.append_rope(host, num_kv_heads=hkv, q=u16(q[layer]), k=u16(k[layer]),
                                       v=u16(v[layer]), block_tables=bt[layer], max_blocks=bt.shape[-1],
                                       seq_lens=seq_lens, positions=pos, batch=len(batch),
                                       num_q_heads=hq, theta=theta)
            want = oracle.gqa_decode(host, num_kv_heads=hkv, q_rot=q_rot, block_tables=bt[layer],
                                     max_blocks=bt.shape[-1], seq_lens=seq_lens, batch=len(batch),
                                     num_q_heads=hq, scale=1.0 / 8.0)
            checked["worst"] = max(checked["worst"],
                                   assert_close(got[layer], want, f"step {checked['steps']} layer {layer}"))
        checked["steps"] += 1

    stats = tr.run(on_step=on_step, on_prefill=on_prefill)
    assert stats["completed"] == len(reqs)
    sched = stats["sched"]
    assert sched["admission_waits"] > 0 and sched["free_pages"] == 64 and sched["active"] == 0
    assert sched["largest_batch"] <= 8 and sched["peak_assigned_pages"] <= 64
    # every decode step processed one token of every active request
    assert stats["decode_tokens"] == sum(r.stop_after - 1 for r in reqs)
    assert stats["prompt_tokens"] == sum(r.prompt_len for r in reqs)
    assert stats["prefill_calls"] == checked["calls"] >= 1
    if prefill_tokens < max(r.prompt_len for r in reqs):
        assert checked["split"] > 0  # some prompt continued in a later call
    got_pool = u16(tr.pool)
    mism = np.flatnonzero(got_pool != host)
    assert mism.size == 0, f"{mism.size} pool elements differ, first at {mism[:5]}"
    tr.close()
