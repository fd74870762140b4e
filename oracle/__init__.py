"""fp64 CPU oracle for the paged-KV decode step (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU legs (the
CPU baseline and ``--impl reference``) may import this package. It wraps the plain C oracle in ``pkv_oracle.c``
(built on first use) with numpy marshalling; it shares no code with the CUDA
library and never imports it.
"""
from __future__ import annotations

import ctypes
import threading

import numpy as np

from . import build as _build

_lib = None
_lock = threading.Lock()

_u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
_c_int, _c_long, _c_double = ctypes.c_int, ctypes.c_long, ctypes.c_double


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            L = ctypes.CDLL(path)
            L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_double.restype = _c_double
            L.oracle_bf16_from_double.argtypes = [_c_double]
            L.oracle_bf16_from_double.restype = ctypes.c_uint16
            L.oracle_bf16_from_double_array.argtypes = [_f64p, _u16p, _c_long]
            L.oracle_bf16_from_double_array.restype = None
            L.oracle_rope_inv_freq.argtypes = [_c_double, _c_int, _c_int]
            L.oracle_rope_inv_freq.restype = _c_double
            L.oracle_rope_rotate_many.argtypes = [_f64p, _f64p, _c_long, _c_int, _i32p, _c_double]
            L.oracle_rope_rotate_many.restype = _c_int
            L.oracle_cos_sin_many.argtypes = [_f64p, _f64p, _f64p, _c_long]
            L.oracle_cos_sin_many.restype = _c_long
            L.oracle_append_rope.argtypes = [_u16p, _c_long, _c_int, _c_int, _c_int, _u16p, _u16p,
                                             _u16p, _f64p, _i32p, _c_int, _i32p, _i32p, _c_int,
                                             _c_int, _c_double]
            L.oracle_append_rope.restype = _c_int
            L.oracle_gqa_decode.argtypes = [_u16p, _c_long, _c_int, _c_int, _c_int, _f64p, _i32p,
                                            _c_int, _i32p, _c_int, _c_int, _c_double, _f64p]
            L.oracle_gqa_decode.restype = _c_int
            L.oracle_gqa_decode_split.argtypes = [_u16p, _c_long, _c_int, _c_int, _c_int, _f64p,
                                                  _i32p, _c_int, _i32p, _c_int, _c_int, _c_double,
                                                  _c_int, _c_int, _f64p, _f64p, _i32p]
            L.oracle_gqa_decode_split.restype = _c_int
            L.oracle_lse_combine.argtypes = [_f64p, _f64p, _i32p, _c_int, _c_int, _c_int, _f64p]
            L.oracle_lse_combine.restype = None
            L.oracle_prefill.argtypes = [_u16p, _c_long, _c_int, _c_int, _c_int, _u16p, _u16p, _u16p,
                                         _i32p, _c_int, _i32p, _i32p, _c_int, _c_int, _c_double,
                                         _c_double, _f64p, _f64p]
            L.oracle_prefill.restype = _c_int
            _lib = L
    return _lib


def _u16(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    return np.ascontiguousarray(a, dtype=np.uint16)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=np.int32)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=np.float64)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


def bf16_to_double(bits) -> np.ndarray:
    """Exact widening (the bf16 bits are the top half of a float32); NaN
    encodings stay NaN (the cast of a signalling NaN is not an error here)."""
    bits = _u16(bits)
    with np.errstate(invalid="ignore"):
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_from_double(x) -> np.ndarray:
    x = _f64(x)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_bf16_from_double_array(x.reshape(-1), out.reshape(-1), x.size)
    return out


def rope_inv_freq(theta: float, head_dim: int) -> np.ndarray:
    return np.array([lib().oracle_rope_inv_freq(theta, j, head_dim) for j in range(head_dim // 2)])


def rope_rotate(x, positions, theta: float) -> np.ndarray:
    """Rotate vectors x [n, D] (fp64) at positions [n]."""
    x = _f64(x)
    n, d = x.shape
    y = np.empty_like(x)
    _check(lib().oracle_rope_rotate_many(x, y, n, d, _i32(positions).reshape(n), float(theta)),
           "rope_rotate (cos/sin not decidable)")
    return y


def cos_sin(angles) -> tuple[np.ndarray, np.ndarray, int]:
    """Correctly rounded fp64 cos and sin of fp64 angles; also returns how many
    values the rounding test could not decide (0 expected)."""
    a = _f64(angles)
    c = np.empty_like(a)
    s = np.empty_like(a)
    bad = lib().oracle_cos_sin_many(a.reshape(-1), c.reshape(-1), s.reshape(-1), a.size)
    return c, s, int(bad)


def rope_angles(positions, theta: float, head_dim: int = 64) -> np.ndarray:
    """The fp64 angles fl(pos * inv_freq_j), [n][head_dim/2], as the rotation forms them."""
    inv = rope_inv_freq(theta, head_dim)
    pos = np.asarray(positions, dtype=np.float64).reshape(-1, 1)
    return pos * inv[None, :]  # one rounded fp64 product per element


def append_rope(pool_u16: np.ndarray, *, num_kv_heads: int, q, k, v, block_tables, max_blocks: int,
                seq_lens, positions, batch: int, num_q_heads: int, theta: float,
                head_dim: int = 64, page_size: int = 16) -> np.ndarray:
    """Append the new tokens into ``pool_u16`` (modified in place); return q_rot fp64."""
    assert pool_u16.dtype == np.uint16 and pool_u16.flags.c_contiguous
    page_elems = 2 * num_kv_heads * page_size * head_dim
    num_pages = pool_u16.size // page_elems
    q_rot = np.empty((batch, num_q_heads, head_dim), dtype=np.float64)
    rc = lib().oracle_append_rope(pool_u16.reshape(-1), num_pages, num_kv_heads, head_dim, page_size,
                                  _u16(q).reshape(-1), _u16(k).reshape(-1), _u16(v).reshape(-1),
                                  q_rot.reshape(-1), _i32(block_tables).reshape(-1), max_blocks,
                                  _i32(seq_lens), _i32(positions), batch, num_q_heads, float(theta))
    _check(rc, "append_rope")
    return q_rot


def gqa_decode(pool_u16: np.ndarray, *, num_kv_heads: int, q_rot, block_tables, max_blocks: int,
               seq_lens, batch: int, num_q_heads: int, scale: float, head_dim: int = 64,
               page_size: int = 16) -> np.ndarray:
    page_elems = 2 * num_kv_heads * page_size * head_dim
    num_pages = pool_u16.size // page_elems
    out = np.empty((batch, num_q_heads, head_dim), dtype=np.float64)
    rc = lib().oracle_gqa_decode(_u16(pool_u16).reshape(-1), num_pages, num_kv_heads, head_dim,
                                 page_size, _f64(q_rot).reshape(-1), _i32(block_tables).reshape(-1),
                                 max_blocks, _i32(seq_lens), batch, num_q_heads, float(scale),
                                 out.reshape(-1))
    _check(rc, "gqa_decode")
    return out



def prefill(pool_u16: np.ndarray, *, num_kv_heads: int, q, k, v, block_tables, max_blocks: int,
            cu_tokens, start_pos, num_q_heads: int, theta: float, scale: float,
            head_dim: int = 64, page_size: int = 16):
    """Chunked causal prefill (appends into ``pool_u16`` in place). q [T,Hq,D],
    k/v [T,Hkv,D] bf16 bits; cu_tokens [B+1], start_pos [B]. Returns
    (q_rot [T,Hq,D], out [T,Hq,D]) in fp64."""
    assert pool_u16.dtype == np.uint16 and pool_u16.flags.c_contiguous
    page_elems = 2 * num_kv_heads * page_size * head_dim
    num_pages = pool_u16.size // page_elems
    cu = _i32(cu_tokens)
    total = int(cu[-1])
    batch = len(cu) - 1
    q_rot = np.zeros((total, num_q_heads, head_dim), dtype=np.float64)
    out = np.zeros((total, num_q_heads, head_dim), dtype=np.float64)
    rc = lib().oracle_prefill(pool_u16.reshape(-1), num_pages, num_kv_heads, head_dim, page_size,
                              _u16(q).reshape(-1), _u16(k).reshape(-1), _u16(v).reshape(-1),
                              _i32(block_tables).reshape(-1), max_blocks, cu, _i32(start_pos),
                              batch, num_q_heads, float(theta), float(scale), q_rot.reshape(-1),
                              out.reshape(-1))
    _check(rc, "prefill")
    return q_rot, out

def gqa_decode_split(pool_u16: np.ndarray, *, num_kv_heads: int, q_rot, block_tables,
                     max_blocks: int, seq_lens, batch: int, num_q_heads: int, scale: float,
                     tokens_per_split: int, head_dim: int = 64, page_size: int = 16):
    """Return (o_part [rows, S, D], lse_part [rows, S], num_splits [rows])."""
    page_elems = 2 * num_kv_heads * page_size * head_dim
    num_pages = pool_u16.size // page_elems
    max_splits = max(1, -(-max_blocks * page_size // tokens_per_split))
    rows = batch * num_q_heads
    o_part = np.zeros((rows, max_splits, head_dim), dtype=np.float64)
    lse_part = np.full((rows, max_splits), -np.inf, dtype=np.float64)
    num_splits = np.zeros(rows, dtype=np.int32)
    rc = lib().oracle_gqa_decode_split(_u16(pool_u16).reshape(-1), num_pages, num_kv_heads,
                                       head_dim, page_size, _f64(q_rot).reshape(-1),
                                       _i32(block_tables).reshape(-1), max_blocks, _i32(seq_lens),
                                       batch, num_q_heads, float(scale), tokens_per_split,
                                       max_splits, o_part.reshape(-1), lse_part.reshape(-1),
                                       num_splits)
    _check(rc, "gqa_decode_split")
    return o_part, lse_part, num_splits


def lse_combine(o_part, lse_part, num_splits) -> np.ndarray:
    o_part = _f64(o_part)
    rows, max_splits, head_dim = o_part.shape
    out = np.empty((rows, head_dim), dtype=np.float64)
    lib().oracle_lse_combine(o_part.reshape(-1), _f64(lse_part).reshape(-1), _i32(num_splits),
                             rows, max_splits, head_dim, out.reshape(-1))
    return out
