"""Paged KV-cache decode step with RoPE for GB300 (sm_103a).

The CUDA library behind include/pkv.h does the work: RoPE of the new token and
its append into a shared BF16 page pool (``paged_kv_append_rope``), paged
grouped-query decode attention with split-KV and a log-sum-exp merge
(``paged_gqa_decode``), both fused into one step (``paged_decode_step``), and
the standalone merge (``paged_kv_split_combine``), and the host page allocator
with page-budget admission (``pkv_sched_*``, include/pkv_sched.h). This package
is the thin Python binding with the same names; it only marshals arguments.
"""
from ._binding import (  # noqa: F401
    ERR_PAGE_ID,
    ERR_POSITION,
    ERR_SEQ_LEN,
    ERR_SPLITS,
    ERR_TIMEOUT,
    DEFAULT_MERGE_WAIT_LOOKS,
    HEAD_DIM,
    LIBRARY,
    MAX_GROUP,
    PAGE_SIZE,
    KVPool,
    PkvError,
    alloc_decode_workspace,
    alloc_prefill_workspace,
    alloc_rope_table,
    build_rope_table,
    decode_max_splits,
    kv_pool_create,
    kv_pool_destroy,
    kv_pool_num_pages,
    kv_pool_page_bytes,
    kv_pool_set_merge_wait_limit,
    lib,
    paged_decode_plan,
    paged_decode_step,
    paged_gqa_decode,
    paged_gqa_decode_no_alloc,
    paged_gqa_decode_partials,
    paged_gqa_decode_workspace_bytes,
    paged_kv_append_rope,
    paged_kv_split_combine,
    paged_prefill,
    paged_prefill_workspace_bytes,
    paged_rope_cos_sin,
    paged_rope_table_build,
    rope_table_rows,
    pkv_get_error,
    pkv_last_cuda_error,
)
from .sched import (  # noqa: F401
    PageScheduler,
    pkv_sched_admit,
    pkv_sched_block_row,
    pkv_sched_budget,
    pkv_sched_create,
    pkv_sched_destroy,
    pkv_sched_finish,
    pkv_sched_grow,
    pkv_sched_note_batch,
    pkv_sched_stats,
    pkv_sched_submit,
)
from .step import DecodeStep  # noqa: F401
