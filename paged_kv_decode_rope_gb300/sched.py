"""Binding of include/pkv_sched.h: the host page allocator and page-budget
admission for the shared KV page pool (continuous or static batching).

Argument marshalling only; the policy lives in csrc/page_sched.cpp. The
functions named like the C entry points take and return the same values;
PageScheduler wraps a handle.
"""
from __future__ import annotations

import ctypes

import numpy as np

from ._binding import PkvError, lib

_STAT_FIELDS = ("pool_pages", "free_pages", "assigned_pages", "peak_assigned_pages",
                "reserved_credits", "active", "waiting", "peak_active", "largest_batch",
                "admission_waits", "admitted", "completed", "rejected")


class SchedStats(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int) for name in _STAT_FIELDS]


def _check(fn: str, rc: int) -> int:
    if rc < 0:
        raise PkvError(fn, rc)
    return rc


def pkv_sched_create(num_pages: int, num_layers: int, context_len: int = 2048,
                     static_batching: bool = False, seed: int = 0) -> int:
    h = ctypes.c_void_p()
    _check("pkv_sched_create", lib().pkv_sched_create(ctypes.byref(h), num_pages, num_layers,
                                                      context_len, int(static_batching), seed))
    return h.value


def pkv_sched_destroy(handle: int) -> None:
    _check("pkv_sched_destroy", lib().pkv_sched_destroy(handle))


def pkv_sched_submit(handle: int, prompt_len: int, max_new: int) -> int:
    rid = ctypes.c_int(-1)
    _check("pkv_sched_submit", lib().pkv_sched_submit(handle, prompt_len, max_new, ctypes.byref(rid)))
    return rid.value


def pkv_sched_budget(handle: int, prompt_len: int, max_new: int) -> int:
    return _check("pkv_sched_budget", lib().pkv_sched_budget(handle, prompt_len, max_new))


def pkv_sched_admit(handle: int, max_ids: int = 4096) -> list[int]:
    ids = (ctypes.c_int * max(max_ids, 1))()
    n = _check("pkv_sched_admit", lib().pkv_sched_admit(handle, ids, max_ids))
    return list(ids[:n])


def pkv_sched_grow(handle: int, request_id: int, kv_len: int) -> None:
    _check("pkv_sched_grow", lib().pkv_sched_grow(handle, request_id, kv_len))


def pkv_sched_block_row(handle: int, request_id: int, layer: int, max_blocks: int) -> np.ndarray:
    row = np.empty(max_blocks, dtype=np.int32)
    _check("pkv_sched_block_row", lib().pkv_sched_block_row(
        handle, request_id, layer, row.ctypes.data_as(ctypes.c_void_p), max_blocks))
    return row


def pkv_sched_finish(handle: int, request_id: int) -> None:
    _check("pkv_sched_finish", lib().pkv_sched_finish(handle, request_id))


def pkv_sched_note_batch(handle: int, batch: int) -> None:
    _check("pkv_sched_note_batch", lib().pkv_sched_note_batch(handle, batch))


def pkv_sched_stats(handle: int) -> dict:
    st = SchedStats()
    _check("pkv_sched_stats", lib().pkv_sched_stats(handle, ctypes.byref(st)))
    return {name: getattr(st, name) for name in _STAT_FIELDS}


class PageScheduler:
    """A pkv_sched handle: submit requests, admit them under their page budgets,
    grow their pages lazily, read their block-table rows, finish them."""

    def __init__(self, num_pages: int, num_layers: int, context_len: int = 2048,
                 static_batching: bool = False, seed: int = 0):
        self.num_layers = num_layers
        self.handle = pkv_sched_create(num_pages, num_layers, context_len, static_batching, seed)

    def submit(self, prompt_len: int, max_new: int) -> int:
        return pkv_sched_submit(self.handle, prompt_len, max_new)

    def budget(self, prompt_len: int, max_new: int) -> int:
        return pkv_sched_budget(self.handle, prompt_len, max_new)

    def admit(self) -> list[int]:
        return pkv_sched_admit(self.handle)

    def grow(self, request_id: int, kv_len: int) -> None:
        pkv_sched_grow(self.handle, request_id, kv_len)

    def block_row(self, request_id: int, layer: int, max_blocks: int) -> np.ndarray:
        return pkv_sched_block_row(self.handle, request_id, layer, max_blocks)

    def block_rows(self, request_id: int, max_blocks: int) -> np.ndarray:
        """[num_layers][max_blocks] page ids of one request."""
        return np.stack([self.block_row(request_id, layer, max_blocks) for layer in range(self.num_layers)])

    def finish(self, request_id: int) -> None:
        pkv_sched_finish(self.handle, request_id)

    def note_batch(self, batch: int) -> None:
        pkv_sched_note_batch(self.handle, batch)

    def stats(self) -> dict:
        return pkv_sched_stats(self.handle)

    def close(self) -> None:
        if self.handle:
            pkv_sched_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
