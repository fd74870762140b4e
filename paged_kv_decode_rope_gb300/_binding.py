"""ctypes binding of the pkv C ABI (include/pkv.h).

Argument marshalling only: shapes and pointers are read off torch tensors and
passed to the CUDA library, which does all of the work on the device. There is
no fallback: if libpkv.so is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(_HERE, "libpkv.so")

HEAD_DIM = 64
PAGE_SIZE = 16
MAX_GROUP = 8
ROPE_TABLE_BYTES_PER_ROW = 1024  # PKV_ROPE_TABLE_BYTES(1)
ERR_SEQ_LEN, ERR_PAGE_ID, ERR_TIMEOUT, ERR_SPLITS, ERR_POSITION = 0x1, 0x2, 0x4, 0x8, 0x10

_lib = None
_lock = threading.Lock()

_vp, _i, _sz, _f, _d = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float, ctypes.c_double

_SIGNATURES = {
    "kv_pool_create": (_i, [ctypes.POINTER(_vp), _vp, _sz, _i, _i, _i]),
    "kv_pool_destroy": (_i, [_vp]),
    "kv_pool_num_pages": (_i, [_vp]),
    "kv_pool_page_bytes": (_sz, [_i, _i, _i]),
    "kv_pool_set_merge_wait_limit": (_i, [_vp, ctypes.c_uint32, ctypes.POINTER(ctypes.c_uint32)]),
    "paged_kv_append_rope": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _i, _d, _vp]),
    "paged_gqa_decode_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "paged_gqa_decode": (_i, [_vp, _vp, _vp, _vp, _i, _vp, _i, _i, _f, _i, _vp, _sz, _vp]),
    "paged_gqa_decode_partials": (_i, [_vp, _vp, _vp, _i, _vp, _i, _i, _f, _i, _vp, _vp, _vp, _i, _vp]),
    "paged_gqa_decode_no_alloc": (_i, [_vp, _vp, _vp, _vp, _i, _vp, _i, _i, _f, _i, _vp]),
    "paged_rope_cos_sin": (_i, [_vp, _i, _d, _vp, _vp]),
    "paged_rope_table_build": (_i, [_d, _i, _vp, _vp]),
    "paged_decode_plan": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _vp, _sz, _vp]),
    "paged_decode_step": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _f,
                               _i, _vp, _sz, _vp]),
    "paged_kv_split_combine": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _vp]),
    "paged_prefill_workspace_bytes": (_sz, [_i, _i, _i]),
    "paged_prefill": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _i, _i, _vp, _i, _f,
                           _vp, _sz, _vp]),
    "pkv_get_error": (_i, [_vp, ctypes.POINTER(_i), _i]),
    "pkv_last_cuda_error": (_i, []),
    # include/pkv_sched.h (host only)
    "pkv_sched_create": (_i, [ctypes.POINTER(_vp), _i, _i, _i, _i, ctypes.c_uint64]),
    "pkv_sched_destroy": (_i, [_vp]),
    "pkv_sched_submit": (_i, [_vp, _i, _i, ctypes.POINTER(_i)]),
    "pkv_sched_budget": (_i, [_vp, _i, _i]),
    "pkv_sched_admit": (_i, [_vp, _vp, _i]),
    "pkv_sched_grow": (_i, [_vp, _i, _i]),
    "pkv_sched_block_row": (_i, [_vp, _i, _i, _vp, _i]),
    "pkv_sched_finish": (_i, [_vp, _i]),
    "pkv_sched_note_batch": (_i, [_vp, _i]),
    "pkv_sched_stats": (_i, [_vp, _vp]),
}


class PkvError(RuntimeError):
    def __init__(self, fn: str, rc: int):
        names = {-22: "EINVAL", -28: "ENOSPC", -5: "EIO", -12: "ENOMEM", -7: "E2BIG"}
        extra = ""
        if rc == -5 and _lib is not None:
            extra = f" (cudaError {_lib.pkv_last_cuda_error()})"
        super().__init__(f"{fn} failed: {names.get(rc, rc)}{extra}")
        self.rc = rc


def lib():
    """Load libpkv.so once. Raises if it is not built: there is no other path."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIBRARY):
                raise RuntimeError(f"{LIBRARY} is not built; run paged_kv_decode_rope_gb300.build.build()")
            L = ctypes.CDLL(LIBRARY)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _check(fn: str, rc: int) -> None:
    if rc != 0:
        raise PkvError(fn, rc)


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t: torch.Tensor, dtype: torch.dtype, name: str, ndim: int | None = None) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")
    return t.data_ptr()


def _shape(t: torch.Tensor, want: tuple, name: str) -> tuple:
    """Check t's shape against `want` (an int per dimension, None for any
    size) before any pointer reaches the library: the C ABI sees bare
    pointers, so a tensor of the wrong size would be read or written out of
    bounds on the device. Returns the shape."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    got = tuple(t.shape)
    if len(got) != len(want) or any(w is not None and g != w for g, w in zip(got, want)):
        spec = "[" + ", ".join("*" if w is None else str(w) for w in want) + "]"
        raise ValueError(f"{name} must have shape {spec}, got {list(got)}")
    return got


class KVPool:
    """A page pool over caller storage (the handle of kv_pool_create)."""

    def __init__(self, handle: int, storage: torch.Tensor, num_kv_heads: int):
        self._handle = handle
        self.storage = storage  # keeps the storage alive as long as the pool
        self.num_kv_heads = num_kv_heads

    @property
    def handle(self) -> int:
        if not self._handle:
            raise ValueError("pool destroyed")
        return self._handle

    @property
    def num_pages(self) -> int:
        return lib().kv_pool_num_pages(self.handle)

    def close(self) -> None:
        if self._handle:
            h, self._handle = self._handle, None
            _check("kv_pool_destroy", lib().kv_pool_destroy(h))

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def kv_pool_page_bytes(num_kv_heads: int, head_dim: int = HEAD_DIM, page_size: int = PAGE_SIZE) -> int:
    return lib().kv_pool_page_bytes(num_kv_heads, head_dim, page_size)


def kv_pool_create(storage: torch.Tensor, num_kv_heads: int, head_dim: int = HEAD_DIM,
                   page_size: int = PAGE_SIZE) -> KVPool:
    if storage.device.type != "cuda" or not storage.is_contiguous():
        raise ValueError("storage must be a contiguous CUDA tensor")
    h = _vp()
    nbytes = storage.numel() * storage.element_size()
    _check("kv_pool_create", lib().kv_pool_create(ctypes.byref(h), storage.data_ptr(), nbytes,
                                                  num_kv_heads, head_dim, page_size))
    return KVPool(h.value, storage, num_kv_heads)


def kv_pool_destroy(pool: KVPool) -> None:
    pool.close()


def kv_pool_num_pages(pool: KVPool) -> int:
    return pool.num_pages


DEFAULT_MERGE_WAIT_LOOKS = 1 << 20


def kv_pool_set_merge_wait_limit(pool: KVPool, looks: int) -> int:
    """Bound of a decode merger's wait for other CTAs' partials, in looks (0:
    give up at once, setting ERR_TIMEOUT). Returns the previous bound."""
    prev = ctypes.c_uint32(0)
    _check("kv_pool_set_merge_wait_limit",
           lib().kv_pool_set_merge_wait_limit(pool.handle, int(looks), ctypes.byref(prev)))
    return prev.value


def paged_kv_append_rope(pool: KVPool, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                         q_rot: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor,
                         positions: torch.Tensor, rope_theta: float, stream=None) -> None:
    """q [B,Hq,64] bf16, k/v [B,Hkv,64] bf16, q_rot [B,Hq,64] fp32 out,
    block_tables [B,max_blocks] int32, seq_lens/positions [B] int32."""
    batch, hq, _ = _shape(q, (None, None, HEAD_DIM), "q")
    for t, name in ((k, "k"), (v, "v")):
        _shape(t, (batch, pool.num_kv_heads, HEAD_DIM), name)
    _shape(q_rot, (batch, hq, HEAD_DIM), "q_rot")
    _shape(block_tables, (batch, None), "block_tables")
    _shape(seq_lens, (batch,), "seq_lens")
    _shape(positions, (batch,), "positions")
    rc = lib().paged_kv_append_rope(
        pool.handle, _dev(q, torch.bfloat16, "q", 3), _dev(k, torch.bfloat16, "k", 3),
        _dev(v, torch.bfloat16, "v", 3), _dev(q_rot, torch.float32, "q_rot", 3),
        _dev(block_tables, torch.int32, "block_tables", 2), block_tables.shape[1],
        _dev(seq_lens, torch.int32, "seq_lens", 1), _dev(positions, torch.int32, "positions", 1),
        batch, hq, float(rope_theta), _stream(stream))
    _check("paged_kv_append_rope", rc)


def paged_gqa_decode_workspace_bytes(batch: int, num_q_heads: int, num_kv_heads: int,
                                     max_blocks: int, pages_per_split: int = 0) -> int:
    return lib().paged_gqa_decode_workspace_bytes(batch, num_q_heads, num_kv_heads, max_blocks,
                                                  pages_per_split)


def alloc_decode_workspace(batch: int, num_q_heads: int, num_kv_heads: int, max_blocks: int,
                           pages_per_split: int = 0, device=None) -> torch.Tensor:
    """A zero-filled workspace buffer of the required size (the decode reads a
    zero word as "not written in this call" and leaves every word it wrote at
    zero again)."""
    n = paged_gqa_decode_workspace_bytes(batch, num_q_heads, num_kv_heads, max_blocks, pages_per_split)
    if n == 0:
        raise ValueError("invalid decode sizes")
    return torch.zeros(n, dtype=torch.uint8, device=device or torch.device("cuda"))


def _decode_shapes(q_rot, out, block_tables, seq_lens) -> tuple:
    batch, hq, _ = _shape(q_rot, (None, None, HEAD_DIM), "q_rot")
    _shape(out, (batch, hq, HEAD_DIM), "out")
    _shape(block_tables, (batch, None), "block_tables")
    _shape(seq_lens, (batch,), "seq_lens")
    return batch, hq


def paged_gqa_decode(pool: KVPool, q_rot: torch.Tensor, out: torch.Tensor,
                     block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                     workspace: torch.Tensor, pages_per_split: int = 0, stream=None) -> None:
    """q_rot/out [B,Hq,64] fp32; workspace from alloc_decode_workspace()."""
    batch, hq = _decode_shapes(q_rot, out, block_tables, seq_lens)
    rc = lib().paged_gqa_decode(
        pool.handle, _dev(q_rot, torch.float32, "q_rot", 3), _dev(out, torch.float32, "out", 3),
        _dev(block_tables, torch.int32, "block_tables", 2), block_tables.shape[1],
        _dev(seq_lens, torch.int32, "seq_lens", 1), batch, hq, float(scale), pages_per_split,
        _dev(workspace, torch.uint8, "workspace", 1), workspace.numel(), _stream(stream))
    _check("paged_gqa_decode", rc)


def paged_gqa_decode_no_alloc(pool: KVPool, q_rot: torch.Tensor, out: torch.Tensor,
                              block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                              pages_per_split: int = 0, stream=None) -> None:
    """paged_gqa_decode without a workspace: for callers that cannot allocate
    device memory, the library's fixed scratch array serves instead. Calls
    that overlap on the GPU share that array and race."""
    batch, hq = _decode_shapes(q_rot, out, block_tables, seq_lens)
    rc = lib().paged_gqa_decode_no_alloc(
        pool.handle, _dev(q_rot, torch.float32, "q_rot", 3), _dev(out, torch.float32, "out", 3),
        _dev(block_tables, torch.int32, "block_tables", 2), block_tables.shape[1],
        _dev(seq_lens, torch.int32, "seq_lens", 1), batch, hq, float(scale), pages_per_split,
        _stream(stream))
    _check("paged_gqa_decode_no_alloc", rc)


def alloc_rope_table(rows: int, device=None) -> torch.Tensor:
    """A buffer for a RoPE table of ``rows`` rows (PKV_ROPE_TABLE_BYTES)."""
    return torch.empty(rows * ROPE_TABLE_BYTES_PER_ROW, dtype=torch.uint8,
                       device=device or torch.device("cuda"))


def rope_table_rows(table: torch.Tensor) -> int:
    return table.numel() // ROPE_TABLE_BYTES_PER_ROW


def paged_rope_cos_sin(positions: torch.Tensor, rope_theta: float, table: torch.Tensor,
                       stream=None) -> None:
    """positions [R] int32 -> a RoPE table of R rows (uint8 [R*1024], from
    alloc_rope_table), row r for positions[r]: float32 [R,32,4] {cos_hi,
    cos_lo, sin_hi, sin_lo}, then float64 [R,32,2] {cos, sin}."""
    (rows,) = _shape(positions, (None,), "positions")
    if table.numel() < rows * ROPE_TABLE_BYTES_PER_ROW:
        raise ValueError("rope table too small")
    rc = lib().paged_rope_cos_sin(_dev(positions, torch.int32, "positions", 1), rows,
                                  float(rope_theta), _dev(table, torch.uint8, "table", 1),
                                  _stream(stream))
    _check("paged_rope_cos_sin", rc)


def paged_rope_table_build(rope_theta: float, num_positions: int, table: torch.Tensor,
                           stream=None) -> None:
    """The RoPE table of positions 0 .. num_positions-1 (row p = position p)."""
    if table.numel() < num_positions * ROPE_TABLE_BYTES_PER_ROW:
        raise ValueError("rope table too small")
    rc = lib().paged_rope_table_build(float(rope_theta), int(num_positions),
                                      _dev(table, torch.uint8, "table", 1), _stream(stream))
    _check("paged_rope_table_build", rc)


def build_rope_table(rope_theta: float, num_positions: int, device=None, stream=None) -> torch.Tensor:
    """Allocate and build the RoPE table of positions 0 .. num_positions-1, once
    per model (the decode step and the prefill read the row of each position)."""
    table = alloc_rope_table(num_positions, device=device)
    paged_rope_table_build(rope_theta, num_positions, table, stream)
    return table


def paged_decode_plan(pool: KVPool, seq_lens: torch.Tensor, block_tables: torch.Tensor,
                      num_q_heads: int, workspace: torch.Tensor, positions: torch.Tensor | None = None,
                      rope_table: torch.Tensor | None = None, stream=None) -> None:
    """The step's work plan into ``workspace``: for paged_decode_step give the
    positions and the RoPE table it will read; for paged_gqa_decode give neither."""
    (batch,) = _shape(seq_lens, (None,), "seq_lens")
    _shape(block_tables, (batch, None), "block_tables")
    if (positions is None) != (rope_table is None):
        raise ValueError("give positions and rope_table together, or neither")
    if positions is not None:
        _shape(positions, (batch,), "positions")
    rc = lib().paged_decode_plan(
        pool.handle, _dev(seq_lens, torch.int32, "seq_lens", 1),
        None if positions is None else _dev(positions, torch.int32, "positions", 1),
        0 if rope_table is None else rope_table_rows(rope_table), batch, num_q_heads,
        block_tables.shape[1], _dev(workspace, torch.uint8, "workspace", 1), workspace.numel(),
        _stream(stream))
    _check("paged_decode_plan", rc)


def paged_decode_step(pool: KVPool, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                      rope_table: torch.Tensor, positions: torch.Tensor, out: torch.Tensor,
                      block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                      workspace: torch.Tensor, q_rot: torch.Tensor | None = None,
                      pages_per_split: int = 0, stream=None) -> None:
    """One layer's whole step (RoPE + append + decode) in one call.
    q [B,Hq,64], k/v [B,Hkv,64] bf16; rope_table a position table
    (build_rope_table), positions [B] int32 rows of it; out [B,Hq,64] fp32;
    q_rot optional fp32 out."""
    batch, hq, _ = _shape(q, (None, None, HEAD_DIM), "q")
    for t, name in ((k, "k"), (v, "v")):
        _shape(t, (batch, pool.num_kv_heads, HEAD_DIM), name)
    _shape(out, (batch, hq, HEAD_DIM), "out")
    if q_rot is not None:
        _shape(q_rot, (batch, hq, HEAD_DIM), "q_rot")
    _shape(block_tables, (batch, None), "block_tables")
    _shape(seq_lens, (batch,), "seq_lens")
    _shape(positions, (batch,), "positions")
    rows = rope_table_rows(rope_table)
    rc = lib().paged_decode_step(
        pool.handle, _dev(q, torch.bfloat16, "q", 3), _dev(k, torch.bfloat16, "k", 3),
        _dev(v, torch.bfloat16, "v", 3), _dev(rope_table, torch.uint8, "rope_table", 1), rows,
        _dev(positions, torch.int32, "positions", 1),
        None if q_rot is None else _dev(q_rot, torch.float32, "q_rot", 3),
        _dev(out, torch.float32, "out", 3), _dev(block_tables, torch.int32, "block_tables", 2),
        block_tables.shape[1], _dev(seq_lens, torch.int32, "seq_lens", 1), batch, hq,
        float(scale), pages_per_split, _dev(workspace, torch.uint8, "workspace", 1),
        workspace.numel(), _stream(stream))
    _check("paged_decode_step", rc)


def paged_prefill_workspace_bytes(total_tokens: int, batch: int, max_blocks: int) -> int:
    return lib().paged_prefill_workspace_bytes(total_tokens, batch, max_blocks)


def alloc_prefill_workspace(total_tokens: int, batch: int, max_blocks: int,
                            device=None) -> torch.Tensor:
    n = paged_prefill_workspace_bytes(total_tokens, batch, max_blocks)
    if n == 0:
        raise ValueError("invalid prefill sizes")
    return torch.empty(n, dtype=torch.uint8, device=device or torch.device("cuda"))


def paged_prefill(pool: KVPool, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                  q_rot: torch.Tensor, out: torch.Tensor, block_tables: torch.Tensor,
                  cu_tokens: torch.Tensor, start_pos: torch.Tensor, rope_table: torch.Tensor,
                  scale: float, workspace: torch.Tensor, stream=None) -> None:
    """Chunked causal prefill. q [T,Hq,64], k/v [T,Hkv,64] bf16; q_rot/out [T,Hq,64]
    fp32 out; block_tables [B,max_blocks], cu_tokens [B+1], start_pos [B] int32;
    rope_table a position table (build_rope_table)."""
    total, hq, _ = _shape(q, (None, None, HEAD_DIM), "q")
    for t, name in ((k, "k"), (v, "v")):
        _shape(t, (total, pool.num_kv_heads, HEAD_DIM), name)
    _shape(q_rot, (total, hq, HEAD_DIM), "q_rot")
    _shape(out, (total, hq, HEAD_DIM), "out")
    batch, _ = _shape(block_tables, (None, None), "block_tables")
    _shape(cu_tokens, (batch + 1,), "cu_tokens")
    _shape(start_pos, (batch,), "start_pos")
    rc = lib().paged_prefill(
        pool.handle, _dev(q, torch.bfloat16, "q", 3), _dev(k, torch.bfloat16, "k", 3),
        _dev(v, torch.bfloat16, "v", 3), _dev(q_rot, torch.float32, "q_rot", 3),
        _dev(out, torch.float32, "out", 3), _dev(block_tables, torch.int32, "block_tables", 2),
        block_tables.shape[1], _dev(cu_tokens, torch.int32, "cu_tokens", 1),
        _dev(start_pos, torch.int32, "start_pos", 1), batch, total, hq,
        _dev(rope_table, torch.uint8, "rope_table", 1), rope_table_rows(rope_table), float(scale),
        _dev(workspace, torch.uint8, "workspace", 1), workspace.numel(), _stream(stream))
    _check("paged_prefill", rc)


def decode_max_splits(max_blocks: int, pages_per_split: int) -> int:
    return max_blocks // pages_per_split + 2


def paged_gqa_decode_partials(pool: KVPool, q_rot: torch.Tensor, block_tables: torch.Tensor,
                              seq_lens: torch.Tensor, scale: float, pages_per_split: int,
                              o_part: torch.Tensor, lse_part: torch.Tensor,
                              num_splits: torch.Tensor, stream=None) -> None:
    """o_part [B*Hq, S, 64] fp32, lse_part [B*Hq, S] fp32, num_splits [B*Hq] int32 (outputs)."""
    batch, hq, _ = _shape(q_rot, (None, None, HEAD_DIM), "q_rot")
    _shape(block_tables, (batch, None), "block_tables")
    _shape(seq_lens, (batch,), "seq_lens")
    _, max_splits, _ = _shape(o_part, (batch * hq, None, HEAD_DIM), "o_part")
    _shape(lse_part, (batch * hq, max_splits), "lse_part")
    _shape(num_splits, (batch * hq,), "num_splits")
    rc = lib().paged_gqa_decode_partials(
        pool.handle, _dev(q_rot, torch.float32, "q_rot", 3),
        _dev(block_tables, torch.int32, "block_tables", 2), block_tables.shape[1],
        _dev(seq_lens, torch.int32, "seq_lens", 1), batch, hq, float(scale), pages_per_split,
        _dev(o_part, torch.float32, "o_part", 3), _dev(lse_part, torch.float32, "lse_part", 2),
        _dev(num_splits, torch.int32, "num_splits", 1), o_part.shape[1], _stream(stream))
    _check("paged_gqa_decode_partials", rc)


def paged_kv_split_combine(o_part: torch.Tensor, lse_part: torch.Tensor, num_splits: torch.Tensor,
                           out: torch.Tensor, stream=None) -> None:
    """o_part [rows, S, D], lse_part [rows, S], num_splits [rows] -> out [rows, D]
    (any shape of rows * D elements)."""
    rows, max_splits, head_dim = _shape(o_part, (None, None, None), "o_part")
    _shape(lse_part, (rows, max_splits), "lse_part")
    _shape(num_splits, (rows,), "num_splits")
    if out.numel() != rows * head_dim:
        raise ValueError(f"out must hold rows * D = {rows * head_dim} elements, got {out.numel()}")
    rc = lib().paged_kv_split_combine(
        _dev(o_part, torch.float32, "o_part", 3), _dev(lse_part, torch.float32, "lse_part", 2),
        _dev(num_splits, torch.int32, "num_splits", 1), _dev(out, torch.float32, "out"),
        rows, max_splits, head_dim, _stream(stream))
    _check("paged_kv_split_combine", rc)


def pkv_get_error(pool: KVPool, reset: bool = False) -> int:
    bits = _i(0)
    _check("pkv_get_error", lib().pkv_get_error(pool.handle, ctypes.byref(bits), int(reset)))
    return bits.value


def pkv_last_cuda_error() -> int:
    return lib().pkv_last_cuda_error()
