"""Host page allocator and page-budget admission (include/pkv_sched.h), on CPU.

The policy under test is the one "Hours of YouTube and 85 handtyped pages of
notes on LLM Inference – Start here" states for its continuous batching:
budget = prompt + allowed new tokens - 1, rounded up to 16-token pages, in
every layer, with the new tokens clamped to the context; pages assigned
lazily; FIFO admission when budgets fit (static batching: only as a new group);
rejection of a budget larger than the pool; pages and credits returned on
completion.
"""
import math

import numpy as np
import pytest

import paged_kv_decode_rope_gb300 as pkv
from paged_kv_decode_rope_gb300 import PageScheduler, PkvError

L = 16  # layers of the Llama-3.2-1B shape


def test_budget_is_processed_prefix_in_pages_per_layer():
    s = PageScheduler(num_pages=4096, num_layers=L, context_len=2048)
    # 10 prompt tokens, 64 new: 73 processed tokens -> 5 pages in each of 16 layers
    assert s.budget(10, 64) == 5 * L
    # exactly on a page boundary: 16 + 1 - 1 = 16 tokens -> 1 page per layer
    assert s.budget(16, 1) == 1 * L
    assert s.budget(16, 2) == 2 * L
    # the new tokens are clamped to the context: 2000 + 48 - 1 = 2047 tokens -> 128 pages
    assert s.budget(2000, 128) == 128 * L == s.budget(2000, 48)
    with pytest.raises(PkvError):
        s.budget(2048, 1)  # no room for even one new token
    s.close()


def test_request_larger_than_pool_is_rejected():
    s = PageScheduler(num_pages=100, num_layers=L)
    with pytest.raises(PkvError, match="ENOSPC"):
        s.submit(100, 10)  # ceil(109 / 16) * 16 = 112 > 100 pages
    rid = s.submit(40, 9)  # ceil(48 / 16) * 16 = 48 pages
    assert rid == 0
    st = s.stats()
    assert st["rejected"] == 1 and st["waiting"] == 1
    s.close()


def test_fifo_admission_does_not_skip_the_head():
    s = PageScheduler(num_pages=100, num_layers=L)
    a = s.submit(40, 9)   # 48 pages
    b = s.submit(60, 5)   # 64 pages: does not fit next to a
    c = s.submit(1, 1)    # 16 pages: would fit, but waits behind b
    assert s.admit() == [a]
    st = s.stats()
    assert st["active"] == 1 and st["waiting"] == 2 and st["admission_waits"] == 2
    assert s.admit() == []  # nothing changed
    assert s.stats()["admission_waits"] == 2  # each request counted once
    s.finish(a)
    assert s.admit() == [b, c]  # 64 + 16 <= 100
    st = s.stats()
    assert st["reserved_credits"] == 80 and st["peak_active"] == 2 and st["completed"] == 1
    s.close()


def test_static_batching_admits_only_whole_groups():
    s = PageScheduler(num_pages=100, num_layers=L, static_batching=True)
    a = s.submit(1, 1)   # 16
    b = s.submit(1, 1)   # 16
    assert s.admit() == [a, b]
    c = s.submit(1, 1)
    assert s.admit() == []  # room for c, but the group is still running
    s.finish(a)
    assert s.admit() == []
    s.finish(b)
    assert s.admit() == [c]
    s.close()


def test_lazy_page_assignment_and_release():
    s = PageScheduler(num_pages=200, num_layers=2)
    rid = s.submit(20, 30)  # 49 tokens -> 4 pages per layer, 8 credits
    assert s.admit() == [rid]
    assert s.stats()["assigned_pages"] == 0  # credits only, no pages yet
    s.grow(rid, 20)  # the prompt: 2 pages per layer
    rows = s.block_rows(rid, 8)
    assert (rows[:, :2] >= 0).all() and (rows[:, 2:] == -1).all()
    assert s.stats()["assigned_pages"] == 4
    s.grow(rid, 32)  # still 2 pages
    assert s.stats()["assigned_pages"] == 4
    s.grow(rid, 33)  # crosses into the third page of each layer
    assert s.stats()["assigned_pages"] == 6
    with pytest.raises(PkvError):
        s.grow(rid, 50)  # beyond the budget of 49 processed tokens
    s.grow(rid, 49)
    st = s.stats()
    assert st["assigned_pages"] == 8 and st["free_pages"] == 192 and st["peak_assigned_pages"] == 8
    s.finish(rid)
    st = s.stats()
    assert st["assigned_pages"] == 0 and st["free_pages"] == 200 and st["reserved_credits"] == 0
    with pytest.raises(PkvError):
        s.grow(rid, 1)  # no longer active
    s.close()


def test_free_list_order_is_seeded_and_deterministic():
    def pages(seed):
        s = PageScheduler(num_pages=64, num_layers=1, seed=seed)
        rid = s.submit(64, 1)
        s.admit()
        s.grow(rid, 64)
        row = s.block_row(rid, 0, 4)
        s.close()
        return row.tolist()
    assert pages(0) == [0, 1, 2, 3]
    assert pages(7) == pages(7)
    assert pages(7) != pages(8)
    assert sorted(set(pages(7))) == sorted(pages(7))


def test_random_traffic_keeps_the_invariants():
    """Random submissions, growth and completions: pages are never shared, never
    exceed a request's credits, and free + assigned always equals the pool."""
    rng = np.random.default_rng(5)
    num_pages, layers, ctx = 300, 4, 256
    s = PageScheduler(num_pages=num_pages, num_layers=layers, context_len=ctx, seed=3)
    state = {}  # rid -> [prompt, budget_tokens, kv_len]
    for _ in range(600):
        op = rng.integers(0, 4)
        if op == 0:
            p, m = int(rng.integers(1, ctx)), int(rng.integers(1, 200))
            try:
                rid = s.submit(p, m)
                state[rid] = [p, p + min(m, ctx - p) - 1, 0]
            except PkvError:
                assert math.ceil((p + min(m, ctx - p) - 1) / 16) * layers > num_pages
        elif op == 1:
            for rid in s.admit():
                state[rid][2] = state[rid][0]
                s.grow(rid, state[rid][2])
        elif op == 2:
            active = [r for r, v in state.items() if v[2] > 0]
            if active:
                rid = active[int(rng.integers(len(active)))]
                state[rid][2] = min(state[rid][1], state[rid][2] + int(rng.integers(1, 40)))
                s.grow(rid, state[rid][2])
        else:
            active = [r for r, v in state.items() if v[2] > 0]
            if active:
                rid = active[int(rng.integers(len(active)))]
                s.finish(rid)
                del state[rid]
        st = s.stats()
        assert st["free_pages"] + st["assigned_pages"] == num_pages
        assert st["reserved_credits"] <= num_pages
        seen = []
        for rid, (p, budget, kv) in state.items():
            if kv == 0:
                continue
            rows = s.block_rows(rid, 16)
            need = math.ceil(kv / 16)
            assert ((rows >= 0).sum(axis=1) == need).all()
            seen.extend(rows[rows >= 0].tolist())
        assert len(seen) == len(set(seen)) == st["assigned_pages"]
    s.close()


def test_c_names_are_bound():
    h = pkv.pkv_sched_create(32, 1, 2048, False, 0)
    rid = pkv.pkv_sched_submit(h, 5, 5)
    assert pkv.pkv_sched_admit(h) == [rid]
    pkv.pkv_sched_grow(h, rid, 5)
    assert pkv.pkv_sched_block_row(h, rid, 0, 2).tolist() == [0, -1]
    pkv.pkv_sched_note_batch(h, 3)
    assert pkv.pkv_sched_stats(h)["largest_batch"] == 3
    pkv.pkv_sched_finish(h, rid)
    pkv.pkv_sched_destroy(h)


def test_prefill_chunk_packing():
    from paged_kv_decode_rope_gb300.trace import pack_prefill_chunks
    calls = pack_prefill_chunks([0, 1, 2], [5, 100, 3], 48)
    assert calls == [[(0, 0, 5), (1, 0, 43)], [(1, 43, 48)], [(1, 91, 9), (2, 0, 3)]]
    assert pack_prefill_chunks([0, 1], [48, 48], 48) == [[(0, 0, 48)], [(1, 0, 48)]]
    assert pack_prefill_chunks([0, 1], [0, 7], 8) == [[(1, 0, 7)]]
    assert pack_prefill_chunks([], [], 8) == []
    with pytest.raises(ValueError):
        pack_prefill_chunks([0], [4], 0)
    rng = np.random.default_rng(7)
    for _ in range(200):
        n = int(rng.integers(1, 12))
        lens = rng.integers(0, 300, size=n).tolist()
        budget = int(rng.integers(1, 400))
        calls = pack_prefill_chunks(list(range(n)), lens, budget)
        for call in calls:
            assert 1 <= sum(c[2] for c in call) <= budget
            assert len({c[0] for c in call}) == len(call)  # one chunk per request per call
        assert all(sum(c[2] for c in call) == budget for call in calls[:-1])
        for r in range(n):  # every prompt covered once, in order
            pieces = [c for call in calls for c in call if c[0] == r]
            assert [p[1] for p in pieces] == list(np.cumsum([0] + [p[2] for p in pieces])[:-1])
            assert sum(p[2] for p in pieces) == lens[r]
