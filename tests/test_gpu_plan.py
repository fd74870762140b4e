"""The step's work plan (paged_decode_plan).

The plan only carries the decode's partition (page prefix sums and range
bounds), worked out once per step instead of in every CTA of every layer, so
a decode that takes it must give exactly the same result as one that works
the partition out itself: the tests compare the two bit for bit, and both
with the oracle. A plan made for other lengths, or for the other kind of
launch, must be ignored (the decode falls back to its own partition and is
still correct).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import paged_kv_decode_rope_gb300 as pkv
from tests.parity import DeviceWorkload, assert_close, oracle_layer, u16

pytestmark = pytest.mark.gpu

CASES = [
    dict(name="plan_llama", batch=64, num_q_heads=32, num_kv_heads=8, seed=31, lo=1, hi=2048),
    dict(name="plan_qwen", batch=32, num_q_heads=14, num_kv_heads=2, seed=32, lo=1024, hi=4096),
    dict(name="plan_small", batch=5, num_q_heads=32, num_kv_heads=8, seed=33, lo=1, hi=60),
]


def _wl(c):
    rng = np.random.default_rng(c["seed"])
    lens = rng.integers(c["lo"], c["hi"], size=c["batch"], endpoint=True)
    return workloads.build(c["name"], batch=c["batch"], num_layers=1, num_q_heads=c["num_q_heads"],
                           num_kv_heads=c["num_kv_heads"], cached_lens=lens,
                           rope_theta=1e6 if c["num_kv_heads"] == 2 else 500000.0, seed=c["seed"])


def _step(dw, out, plan: bool):
    st = dw.step
    st.workspace.zero_()  # no plan left from an earlier call
    if plan:
        pkv.paged_decode_plan(st.pool, st.seq_lens, st.block_tables[0], st.num_q_heads, st.workspace,
                              positions=st.positions, rope_table=st.rope)
    pkv.paged_decode_step(st.pool, dw.q[0], dw.k[0], dw.v[0], st.rope, st.positions, out,
                          st.block_tables[0], st.seq_lens, st.scale, st.workspace)
    torch.cuda.synchronize()


@pytest.mark.parametrize("c", CASES, ids=[c["name"] for c in CASES])
def test_planned_step_equals_unplanned_and_oracle(c):
    wl = _wl(c)
    want_pool = u16(wl.pool).reshape(-1).copy()
    _, want = oracle_layer(want_pool, wl, 0, u16(wl.q)[0], u16(wl.k)[0], u16(wl.v)[0])
    dw = DeviceWorkload(wl)
    outs = []
    for plan in (False, True, True):  # the planned call twice: the plan is read, not consumed
        out = torch.full_like(dw.step.out[0], float("nan"))
        _step(dw, out, plan)
        assert dw.step.error_bits() == 0
        outs.append(out.cpu().numpy())
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])
    assert_close(outs[1], want, f"{c['name']} planned")
    assert np.array_equal(u16(dw.pool).reshape(-1), want_pool)
    dw.step.close()


def test_planned_decode_from_q_rot_equals_unplanned():
    wl = _wl(CASES[0])
    dw = DeviceWorkload(wl)
    st = dw.step
    st.append(0, dw.q, dw.k, dw.v)
    outs = []
    for plan in (False, True):
        st.workspace.zero_()
        if plan:
            pkv.paged_decode_plan(st.pool, st.seq_lens, st.block_tables[0], st.num_q_heads, st.workspace)
        out = torch.full_like(st.out[0], float("nan"))
        pkv.paged_gqa_decode(st.pool, st.q_rot[0], out, st.block_tables[0], st.seq_lens, wl.scale,
                             st.workspace)
        torch.cuda.synchronize()
        outs.append(out.cpu().numpy())
    assert st.error_bits() == 0
    assert np.array_equal(outs[0], outs[1])
    st.close()


def test_stale_or_mismatched_plan_is_ignored():
    """A plan made for other lengths (the step before), or for the decode
    from q_rot, is not taken: the step is still exactly right."""
    wl = _wl(CASES[0])
    want_pool = u16(wl.pool).reshape(-1).copy()
    _, want = oracle_layer(want_pool, wl, 0, u16(wl.q)[0], u16(wl.k)[0], u16(wl.v)[0])
    dw = DeviceWorkload(wl)
    st = dw.step
    ref = torch.empty_like(st.out[0])
    _step(dw, ref, plan=False)
    other = st.seq_lens.clone()
    other[3] -= 1  # the lengths of another step
    for kind in ("stale", "decode"):
        st.workspace.zero_()
        if kind == "stale":
            pkv.paged_decode_plan(st.pool, other, st.block_tables[0], st.num_q_heads, st.workspace,
                                  positions=st.positions, rope_table=st.rope)
        else:
            pkv.paged_decode_plan(st.pool, st.seq_lens, st.block_tables[0], st.num_q_heads, st.workspace)
        out = torch.full_like(ref, float("nan"))
        pkv.paged_decode_step(st.pool, dw.q[0], dw.k[0], dw.v[0], st.rope, st.positions, out,
                              st.block_tables[0], st.seq_lens, st.scale, st.workspace)
        torch.cuda.synchronize()
        assert st.error_bits() == 0
        g = out.cpu().numpy()
        assert np.array_equal(g, ref.cpu().numpy()), kind
        assert_close(g, want, kind)
    assert np.array_equal(u16(dw.pool).reshape(-1), want_pool)
    st.close()
