"""The C-ABI library loads and exports every symbol include/*.h declares.

No compute call runs here (no GPU needed): only host-side entry points and the
argument checks that reject a call before any CUDA work.
"""
import ctypes
import os
import re

import pytest

from tests.golden.figures import page_figures

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("pkv.h", "pkv_sched.h")]
EINVAL, ENOSPC = -22, -28


def _declared_functions():
    text = "\n".join(open(h, encoding="utf-8").read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\**\s*([a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_decode_rope_gb300 import build
    build.build()
    return ctypes.CDLL(build.LIBRARY)


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("kv_pool_create", "paged_kv_append_rope", "paged_gqa_decode",
                     "paged_kv_split_combine"):
        assert required in names
    assert "pkv_sched_admit" in names and "pkv_sched_grow" in names
    assert len(names) >= 20


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"libpkv.so does not export {name}"


def test_binding_has_every_declared_name():
    import paged_kv_decode_rope_gb300 as pkv
    for name in _declared_functions():
        assert hasattr(pkv, name), f"binding lacks {name}"


def test_page_bytes_and_page_figures(lib):
    lib.kv_pool_page_bytes.restype = ctypes.c_size_t
    figs = page_figures()
    page = lib.kv_pool_page_bytes(8, 64, figs["tokens_per_page"])
    assert page == 8 * 2 * 16 * 64 * 2 == 32768
    # The default 128 MiB pool holds 4096 Llama-3.2-1B pages = 65536 token slots,
    # i.e. 4096 tokens of context in each of the 16 layers.
    pages = figs["default_pool_mib"] * 2**20 // page
    assert pages == 4096
    assert pages * figs["tokens_per_page"] // figs["llama_layers"] == 4096
    # 32 query heads of dim 64 make the 2048-wide hidden state.
    assert 32 * 64 == figs["llama_hidden"]
    assert lib.kv_pool_page_bytes(2, 64, 16) == 8192
    assert lib.kv_pool_page_bytes(8, 128, 16) == 0
    assert lib.kv_pool_page_bytes(8, 64, 32) == 0
    assert lib.kv_pool_page_bytes(0, 64, 16) == 0


def test_argument_checks_before_any_cuda_call(lib):
    vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.kv_pool_create.argtypes = [ctypes.POINTER(vp), vp, sz, i, i, i]
    h = vp()
    assert lib.kv_pool_create(None, 256, 1 << 20, 8, 64, 16) == EINVAL
    assert lib.kv_pool_create(ctypes.byref(h), None, 1 << 20, 8, 64, 16) == EINVAL
    assert lib.kv_pool_create(ctypes.byref(h), 0x1008, 1 << 20, 8, 64, 16) == EINVAL  # misaligned
    assert lib.kv_pool_create(ctypes.byref(h), 0x1000, 1 << 20, 8, 128, 16) == EINVAL
    assert lib.kv_pool_create(ctypes.byref(h), 0x1000, 1 << 20, 8, 64, 8) == EINVAL
    assert lib.kv_pool_create(ctypes.byref(h), 0x1000, 100, 8, 64, 16) == ENOSPC
    lib.paged_kv_append_rope.argtypes = [vp] * 6 + [i, vp, vp, i, i, ctypes.c_double, vp]
    assert lib.paged_kv_append_rope(None, 1, 1, 1, 1, 1, 4, 1, 1, 2, 32, 1e4, None) == EINVAL
    lib.paged_gqa_decode.argtypes = [vp, vp, vp, vp, i, vp, i, i, ctypes.c_float, i, vp, sz, vp]
    assert lib.paged_gqa_decode(None, 1, 1, 1, 4, 1, 2, 32, 0.125, 0, 1, 1 << 20, None) == EINVAL
    lib.paged_gqa_decode_partials.argtypes = [vp, vp, vp, i, vp, i, i, ctypes.c_float, i, vp, vp,
                                              vp, i, vp]
    assert lib.paged_gqa_decode_partials(None, 1, 1, 4, 1, 2, 32, 0.125, 1, 1, 1, 1, 8, None) == EINVAL
    lib.paged_kv_split_combine.argtypes = [vp, vp, vp, vp, i, i, i, vp]
    assert lib.paged_kv_split_combine(1, 1, 1, 1, -1, 4, 64, None) == EINVAL
    assert lib.paged_kv_split_combine(1, 1, 1, 1, 4, 0, 64, None) == EINVAL
    assert lib.paged_kv_split_combine(None, 1, 1, 1, 4, 2, 64, None) == EINVAL
    assert lib.paged_kv_split_combine(1, 1, 1, 1, 0, 2, 64, None) == 0  # nothing to do
    lib.pkv_get_error.argtypes = [vp, ctypes.POINTER(i), i]
    assert lib.pkv_get_error(None, None, 0) == EINVAL
    assert lib.kv_pool_destroy(None) == 0
    assert lib.kv_pool_num_pages(None) == EINVAL


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    import paged_kv_decode_rope_gb300._binding as B
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "LIBRARY", str(tmp_path / "libpkv.so"))
    with pytest.raises(RuntimeError, match="not built"):
        B.lib()


def test_binding_rejects_mismatched_shapes_before_the_library():
    """The C ABI takes bare pointers, so the binding checks that the tensors
    agree in shape (batch, head counts, head_dim 64) before any pointer is
    passed: a mismatch would otherwise be read out of bounds on the device."""
    import torch

    import paged_kv_decode_rope_gb300._binding as B
    pool = B.KVPool(0, None, 8)  # shapes only: the checks run before the handle is used
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    q, k, v = torch.zeros(4, 32, 64, dtype=bf), torch.zeros(4, 8, 64, dtype=bf), torch.zeros(4, 8, 64, dtype=bf)
    qr, out = torch.zeros(4, 32, 64, dtype=f32), torch.zeros(4, 32, 64, dtype=f32)
    bt, sl, pos = torch.zeros(4, 16, dtype=i32), torch.ones(4, dtype=i32), torch.zeros(4, dtype=i32)
    ws, table = torch.zeros(1024, dtype=torch.uint8), torch.zeros(4 * 1024, dtype=torch.uint8)
    bad = {
        "k": torch.zeros(4, 4, 64, dtype=bf),        # not the pool's kv heads
        "v": torch.zeros(3, 8, 64, dtype=bf),        # batch
        "q": torch.zeros(4, 32, 32, dtype=bf),       # head_dim
        "q_rot": torch.zeros(4, 16, 64, dtype=f32),  # heads
        "block_tables": torch.zeros(5, 16, dtype=i32),
        "seq_lens": torch.ones(3, dtype=i32),
        "positions": torch.zeros(5, dtype=i32),
    }

    def append(**kw):
        a = dict(q=q, k=k, v=v, q_rot=qr, block_tables=bt, seq_lens=sl, positions=pos)
        a.update(kw)
        B.paged_kv_append_rope(pool, a["q"], a["k"], a["v"], a["q_rot"], a["block_tables"],
                               a["seq_lens"], a["positions"], 500000.0)

    for name, t in bad.items():
        with pytest.raises(ValueError, match=f"{name} must have shape"):
            append(**{name: t})

    def step(**kw):
        a = dict(q=q, k=k, v=v, out=out, block_tables=bt, seq_lens=sl, positions=pos)
        a.update(kw)
        B.paged_decode_step(pool, a["q"], a["k"], a["v"], table, a["positions"], a["out"],
                            a["block_tables"], a["seq_lens"], 0.125, ws)

    for name in ("k", "v", "q", "block_tables", "seq_lens", "positions"):
        with pytest.raises(ValueError, match=f"{name} must have shape"):
            step(**{name: bad[name]})
    with pytest.raises(ValueError, match="out must have shape"):
        step(out=torch.zeros(4, 32, 63, dtype=f32))
    with pytest.raises(ValueError, match="out must have shape"):
        B.paged_gqa_decode(pool, qr, torch.zeros(4, 31, 64, dtype=f32), bt, sl, 0.125, ws)
    with pytest.raises(ValueError, match="seq_lens must have shape"):
        B.paged_gqa_decode_no_alloc(pool, qr, out, bt, torch.ones(2, dtype=i32), 0.125)
    with pytest.raises(ValueError, match="positions must have shape"):
        B.paged_rope_cos_sin(torch.zeros(4, 1, dtype=i32), 1e4, table)
    # prefill: T tokens over B sequences
    pq, pk = torch.zeros(10, 32, 64, dtype=bf), torch.zeros(10, 8, 64, dtype=bf)
    pqr, pout = torch.zeros(10, 32, 64, dtype=f32), torch.zeros(10, 32, 64, dtype=f32)
    pbt, cu, st = torch.zeros(2, 16, dtype=i32), torch.tensor([0, 4, 10], dtype=i32), torch.zeros(2, dtype=i32)
    with pytest.raises(ValueError, match="cu_tokens must have shape"):
        B.paged_prefill(pool, pq, pk, pk, pqr, pout, pbt, cu[:2], st, table, 0.125, ws)
    with pytest.raises(ValueError, match="k must have shape"):
        B.paged_prefill(pool, pq, pk[:9], pk, pqr, pout, pbt, cu, st, table, 0.125, ws)
    with pytest.raises(ValueError, match="start_pos must have shape"):
        B.paged_prefill(pool, pq, pk, pk, pqr, pout, pbt, cu, torch.zeros(2, 1, dtype=i32), table,
                        0.125, ws)
    with pytest.raises(ValueError, match="rope table too small"):
        B.paged_rope_table_build(1e4, 10, torch.zeros(9 * 1024, dtype=torch.uint8))
    # split results and their merge
    rows = 4 * 32
    with pytest.raises(ValueError, match="o_part must have shape"):
        B.paged_gqa_decode_partials(pool, qr, bt, sl, 0.125, 1, torch.zeros(rows - 1, 3, 64),
                                    torch.zeros(rows - 1, 3), torch.zeros(rows - 1, dtype=i32))
    with pytest.raises(ValueError, match="lse_part must have shape"):
        B.paged_kv_split_combine(torch.zeros(5, 3, 64), torch.zeros(5, 2), torch.zeros(5, dtype=i32),
                                 torch.zeros(5, 64))
    with pytest.raises(ValueError, match="out must hold"):
        B.paged_kv_split_combine(torch.zeros(5, 3, 64), torch.zeros(5, 3), torch.zeros(5, dtype=i32),
                                 torch.zeros(5, 63))


def test_binding_constants_match_the_header():
    """The Python binding's copies of the header's constants (sizes it
    allocates and checks, error bits it decodes) equal the macros."""
    import paged_kv_decode_rope_gb300._binding as B
    text = open(HEADERS[0], encoding="utf-8").read()

    def macro(name):
        m = re.search(rf"#define {name}\s+(\S+)", text)
        assert m, name
        return int(m.group(1), 0)

    assert B.HEAD_DIM == macro("PKV_HEAD_DIM")
    assert B.PAGE_SIZE == macro("PKV_PAGE_SIZE")
    assert B.MAX_GROUP == macro("PKV_MAX_GROUP")
    assert (B.ERR_SEQ_LEN, B.ERR_PAGE_ID, B.ERR_TIMEOUT, B.ERR_SPLITS, B.ERR_POSITION) == tuple(
        macro(f"PKV_ERR_{n}") for n in ("SEQ_LEN", "PAGE_ID", "TIMEOUT", "SPLITS", "POSITION"))
    m = re.search(r"#define PKV_ROPE_TABLE_BYTES\(rows\) \(\(size_t\)\(rows\) \* (\d+)u\)", text)
    assert m and int(m.group(1)) == B.ROPE_TABLE_BYTES_PER_ROW
    assert B.DEFAULT_MERGE_WAIT_LOOKS == 1 << 20
