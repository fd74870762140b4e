"""Seeded synthetic workloads for the batched paged-KV decode step.

This module is shared by the tests, the benchmark and the oracle checks. It
holds none of the method's arithmetic: no rotary embedding, no rounding rule,
no attention. It only fixes shapes, draws seeded random numbers and hands out
physical pages.

Shapes follow the two model families the source pages name:

* Llama-3.2-1B: 32 query heads, 8 KV heads, head_dim 64, 16 layers, RoPE base
  500000. ("Hours of YouTube and 85 handtyped pages of notes on LLM
  Inference – Start here", the fixed Llama 3.2 1B weight-layout item.)
* Qwen2.5-0.5B: 14 query heads, 2 KV heads, head_dim 64, 24 layers, RoPE base
  1e6. ("llmc — 从零写一个大模型推理引擎（配套代码）", the model the engine runs.)

Every page holds 16 tokens of K and V ("Hours of YouTube …", the shared BF16
KV page pool item). A page's bytes are laid out [kv_head][K|V][slot][dim],
bf16, so one KV head's keys and values for a page form one contiguous
4 KiB block.

Conventions used throughout:

* ``cached_lens[b]`` (L_b) tokens are in the cache before the step;
  ``seq_lens[b] = L_b + 1`` is the attention length after the new token is
  appended at cache index L_b; ``positions[b] = L_b`` is its RoPE position.
* Block tables are per layer: ``block_tables[l, b, i]`` is the physical page
  holding tokens [16 i, 16 i + 16) of sequence b in layer l; unused entries
  are -1.
* The new token's page is already assigned (the host hands out pages lazily
  before the step, as the pages describe).
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

HEAD_DIM = 64
PAGE_SIZE = 16
#: bf16 quiet-NaN pattern written into slots that hold no token when a test
#: asks for a sentinel pool; any read of such a slot shows up as NaN.
SENTINEL_BF16 = 0x7FC1


@dataclasses.dataclass
class Workload:
    name: str
    batch: int
    num_layers: int
    num_q_heads: int
    num_kv_heads: int
    rope_theta: float
    scale: float
    cached_lens: np.ndarray  # [B] int32
    seq_lens: np.ndarray  # [B] int32 (= cached_lens + 1)
    positions: np.ndarray  # [B] int32
    max_blocks: int
    num_pages: int
    block_tables: np.ndarray  # [NL, B, max_blocks] int32
    pool: torch.Tensor  # [num_pages * page_elems] bf16
    q: torch.Tensor  # [NL, B, Hq, D] bf16
    k: torch.Tensor  # [NL, B, Hkv, D] bf16
    v: torch.Tensor  # [NL, B, Hkv, D] bf16
    seed: int = 0
    description: str = ""

    @property
    def head_dim(self) -> int:
        return HEAD_DIM

    @property
    def page_size(self) -> int:
        return PAGE_SIZE

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def page_elems(self) -> int:
        return 2 * self.num_kv_heads * PAGE_SIZE * HEAD_DIM

    @property
    def page_bytes(self) -> int:
        return 2 * self.page_elems

    def kv_bytes_per_layer(self) -> int:
        """Algorithmic K+V bytes one decode launch reads: valid tokens only."""
        return int(self.seq_lens.astype(np.int64).sum()) * self.num_kv_heads * HEAD_DIM * 2 * 2

    def kv_bytes_per_step(self) -> int:
        return self.kv_bytes_per_layer() * self.num_layers


def _bf16_normal(gen: torch.Generator, shape, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def _assign_pages(rng: np.random.Generator, seq_lens: np.ndarray, num_layers: int,
                  num_pages: int, max_blocks: int, contiguous: bool = False) -> np.ndarray:
    """Hand out physical pages from a shuffled free list, layer by layer.

    With ``contiguous`` the free list is in order, so every (layer, sequence)
    gets consecutive pages: a contiguous cache per sequence and layer, the
    baseline against which paging's scattered placement is measured."""
    npages = (seq_lens.astype(np.int64) + PAGE_SIZE - 1) // PAGE_SIZE
    need = int(npages.sum()) * num_layers
    if need > num_pages:
        raise ValueError(f"pool of {num_pages} pages cannot hold {need} pages")
    free = (np.arange(num_pages) if contiguous else rng.permutation(num_pages)).astype(np.int32)
    bt = np.full((num_layers, len(seq_lens), max_blocks), -1, dtype=np.int32)
    cur = 0
    for layer in range(num_layers):
        for b, n in enumerate(npages):
            bt[layer, b, :n] = free[cur:cur + n]
            cur += n
    return bt


def _sentinel_unused(pool: torch.Tensor, wl_shape, block_tables: np.ndarray,
                     cached_lens: np.ndarray) -> None:
    """Overwrite every slot that holds no cached token with the NaN sentinel."""
    num_pages, hkv = wl_shape
    view = pool.view(num_pages, hkv, 2, PAGE_SIZE, HEAD_DIM)
    used = np.zeros((num_pages, PAGE_SIZE), dtype=bool)
    nl, bsz, _ = block_tables.shape
    for layer in range(nl):
        for b in range(bsz):
            t = np.arange(int(cached_lens[b]))
            if t.size:
                used[block_tables[layer, b, t // PAGE_SIZE], t % PAGE_SIZE] = True
    unused = torch.from_numpy(~used).to(pool.device)
    # written as 16-bit integers: a bf16 assignment may canonicalise the NaN
    bits = pool.view(torch.int16).view(num_pages, hkv, 2, PAGE_SIZE, HEAD_DIM)
    mask = unused[:, None, None, :, None].expand_as(view)
    bits[mask] = SENTINEL_BF16


def build(name: str, *, batch: int, num_layers: int, num_q_heads: int, num_kv_heads: int,
          cached_lens, rope_theta: float, num_pages: int | None = None,
          pool_slack: float = 1.1, seed: int = 0, device="cpu", sentinel: bool = False,
          big_key_frac: float = 0.0, max_blocks: int | None = None,
          block_tables: np.ndarray | None = None, description: str = "",
          materialize: bool = True, contiguous: bool = False) -> Workload:
    """Assemble a workload from explicit cached lengths (host arrays).

    With ``materialize=False`` only the host-side structure (lengths, page
    assignment) is built and the tensors are left as None.
    """
    rng = np.random.default_rng(seed)
    cached = np.asarray(cached_lens, dtype=np.int32).reshape(batch)
    seq_lens = (cached + 1).astype(np.int32)
    if max_blocks is None:
        max_blocks = int(math.ceil(int(seq_lens.max(initial=1)) / PAGE_SIZE))
    need = int(((seq_lens.astype(np.int64) + PAGE_SIZE - 1) // PAGE_SIZE).sum()) * num_layers
    if num_pages is None:
        num_pages = max(1, int(math.ceil(need * pool_slack)))
    if block_tables is None:
        block_tables = _assign_pages(rng, seq_lens, num_layers, num_pages, max_blocks, contiguous)
    pool = q = k = v = None
    if not materialize:
        return Workload(
            name=name, batch=batch, num_layers=num_layers, num_q_heads=num_q_heads,
            num_kv_heads=num_kv_heads, rope_theta=float(rope_theta), scale=1.0 / math.sqrt(HEAD_DIM),
            cached_lens=cached, seq_lens=seq_lens, positions=cached.copy(), max_blocks=int(max_blocks),
            num_pages=int(num_pages), block_tables=block_tables, pool=pool, q=q, k=k, v=v, seed=seed,
            description=description)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    page_elems = 2 * num_kv_heads * PAGE_SIZE * HEAD_DIM
    pool = _bf16_normal(gen, (num_pages * page_elems,), device)
    q = _bf16_normal(gen, (num_layers, batch, num_q_heads, HEAD_DIM), device)
    k = _bf16_normal(gen, (num_layers, batch, num_kv_heads, HEAD_DIM), device)
    v = _bf16_normal(gen, (num_layers, batch, num_kv_heads, HEAD_DIM), device)
    if big_key_frac > 0.0:
        # A "key row" is one (page, kv head, slot) 64-vector of the cache, and one
        # (layer, sequence, kv head) vector of the new keys. Scaling by 8 is exact in bf16.
        view = pool.view(num_pages, num_kv_heads, 2, PAGE_SIZE, HEAD_DIM)
        sel = torch.rand((num_pages, num_kv_heads, PAGE_SIZE), generator=gen, device=device) < big_key_frac
        view[:, :, 0] = torch.where(sel[..., None], view[:, :, 0] * 8, view[:, :, 0])
        selk = torch.rand((num_layers, batch, num_kv_heads), generator=gen, device=device) < big_key_frac
        k = torch.where(selk[..., None], k * 8, k)
    if sentinel:
        _sentinel_unused(pool, (num_pages, num_kv_heads), block_tables, cached)
    return Workload(
        name=name, batch=batch, num_layers=num_layers, num_q_heads=num_q_heads,
        num_kv_heads=num_kv_heads, rope_theta=float(rope_theta), scale=1.0 / math.sqrt(HEAD_DIM),
        cached_lens=cached, seq_lens=seq_lens, positions=cached.copy(), max_blocks=int(max_blocks),
        num_pages=int(num_pages), block_tables=block_tables, pool=pool, q=q, k=k, v=v, seed=seed,
        description=description)


LLAMA = dict(num_q_heads=32, num_kv_heads=8, rope_theta=500000.0)
QWEN = dict(num_q_heads=14, num_kv_heads=2, rope_theta=1e6)

#: The named workloads. Keys say what each one is.
WORKLOADS = (
    "llama1b_b1_l1_len37",
    "llama1b_b8_l16_u512",
    "llama1b_b64_l16_u2048",
    "qwen05b_b32_l24_u1024_4096",
    "llama1b_b256_l16_skew",
    "llama1b_b64_l16_u2048_contig",
)


def make(name: str, seed: int = 0, device="cpu", sentinel: bool = False,
         materialize: bool = True, layers: int | None = None) -> Workload:
    """Build one of the named workloads with the given seed.

    ``layers`` keeps the workload's shapes and lengths but uses that many
    layers and a pool just large enough for them (1.1x): a smaller case of the
    same kernel launches, for profiling.
    """
    if layers is not None:
        full = make(name, seed=seed, materialize=False)
        return build(f"{name}_first{layers}l", batch=full.batch, num_layers=layers,
                     num_q_heads=full.num_q_heads, num_kv_heads=full.num_kv_heads,
                     cached_lens=full.cached_lens, rope_theta=full.rope_theta, pool_slack=1.1,
                     max_blocks=full.max_blocks, seed=seed, device=device, sentinel=sentinel,
                     materialize=materialize, big_key_frac=0.1 if "u2048" in name and "b64" in name else 0.0,
                     description=full.description + f"; first {layers} layers, pool fitted")
    rng = np.random.default_rng([seed, 0x5EED])
    common = dict(seed=seed, device=device, sentinel=sentinel, materialize=materialize)
    if name == "llama1b_b1_l1_len37":
        # One sequence, one layer, 37 cached tokens + 1 appended; a 64-page pool
        # whose block table is a seeded permutation of all 64 pages.
        bt = rng.permutation(64).astype(np.int32).reshape(1, 1, 64)
        return build(name, batch=1, num_layers=1, cached_lens=[37], num_pages=64,
                     max_blocks=64, block_tables=bt, description="Llama-3.2-1B shape, 1 sequence, 1 layer, 37 cached + 1", **common, **LLAMA)
    if name == "llama1b_b8_l16_u512":
        cached = rng.integers(1, 512, size=8, endpoint=True)
        # 128 MiB pool = 4096 pages of 32 KiB.
        return build(name, batch=8, num_layers=16, cached_lens=cached, num_pages=4096,
                     max_blocks=33,
                     description="Llama-3.2-1B shape, batch 8, 16 layers, L~U[1,512], 128 MiB pool", **common, **LLAMA)
    if name == "llama1b_b64_l16_u2048_contig":
        # The batch-64 workload (same lengths, same data draw) with every
        # (layer, sequence) on consecutive pages: the contiguous-cache baseline.
        cached = rng.integers(1, 2048, size=64, endpoint=True)
        return build(name, batch=64, num_layers=16, cached_lens=cached, num_pages=81920,
                     max_blocks=129, big_key_frac=0.1, contiguous=True,
                     description="batch-64 workload with each (layer, sequence) on consecutive pages "
                                 "(contiguous-cache baseline)",
                     **common, **LLAMA)
    if name == "llama1b_b64_l16_u2048":
        cached = rng.integers(1, 2048, size=64, endpoint=True)
        # 2.5 GiB pool = 81920 pages of 32 KiB; 10% of key rows scaled by 8.
        return build(name, batch=64, num_layers=16, cached_lens=cached, num_pages=81920,
                     max_blocks=129, big_key_frac=0.1,
                     description="Llama-3.2-1B shape, batch 64, 16 layers, L~U[1,2048], 2.5 GiB pool, 10% keys x8",
                     **common, **LLAMA)
    if name == "qwen05b_b32_l24_u1024_4096":
        cached = rng.integers(1024, 4096, size=32, endpoint=True)
        return build(name, batch=32, num_layers=24, cached_lens=cached, pool_slack=1.1,
                     max_blocks=257,
                     description="Qwen2.5-0.5B shape (14/2 heads), batch 32, 24 layers, L~U[1024,4096]", **common, **QWEN)
    if name == "llama1b_b256_l16_skew":
        n_long = int(round(0.1 * 256))
        short = rng.integers(16, 256, size=256 - n_long, endpoint=True)
        long_ = rng.integers(1024, 2048, size=n_long, endpoint=True)
        cached = rng.permutation(np.concatenate([short, long_]))
        return build(name, batch=256, num_layers=16, cached_lens=cached, pool_slack=1.1,
                     max_blocks=129,
                     description="Llama-3.2-1B shape, batch 256, 16 layers, 230 x U[16,256] + 26 x U[1024,2048]",
                     **common, **LLAMA)
    raise KeyError(name)


# ---------------------------------------------------------------------------
# Multi-step decode traces (continuous batching over the page pool)


@dataclasses.dataclass
class TraceRequest:
    """One request of a synthetic trace: prompt_len cached tokens after its
    prefill, at most max_new generated tokens, and the number it actually
    generates before stopping (<= max_new; early stop when smaller)."""
    prompt_len: int
    max_new: int
    stop_after: int


def trace_requests(n: int, seed: int, prompt_range=(1, 512), new_range=(1, 256),
                   early_stop_frac: float = 0.3) -> list[TraceRequest]:
    """n seeded requests: prompts and output budgets uniform in the ranges; a
    fraction stops early at a uniform point of its budget."""
    rng = np.random.default_rng([seed, 0x7ACE])
    out = []
    for _ in range(n):
        p = int(rng.integers(prompt_range[0], prompt_range[1], endpoint=True))
        m = int(rng.integers(new_range[0], new_range[1], endpoint=True))
        stop = int(rng.integers(1, m, endpoint=True)) if rng.random() < early_stop_frac else m
        out.append(TraceRequest(p, m, stop))
    return out


def trace_prompt_qkv(seed: int, request: int, num_layers: int, num_q_heads: int,
                     num_kv_heads: int, prompt_len: int):
    """A request's prompt as its prefill sees it: q [num_layers][prompt_len][Hq][64]
    and k, v [num_layers][prompt_len][Hkv][64], bf16 N(0,1), on the CPU;
    independent of which other requests share the prefill call."""
    gen = torch.Generator()
    gen.manual_seed(hash((seed, request, 0x9E)) & 0x7FFFFFFF)
    q = _bf16_normal(gen, (num_layers, prompt_len, num_q_heads, HEAD_DIM), "cpu")
    k = _bf16_normal(gen, (num_layers, prompt_len, num_kv_heads, HEAD_DIM), "cpu")
    v = _bf16_normal(gen, (num_layers, prompt_len, num_kv_heads, HEAD_DIM), "cpu")
    return q, k, v


def trace_step_qkv(seed: int, request: int, step: int, num_layers: int, num_q_heads: int,
                   num_kv_heads: int):
    """The new token's q, k, v of one request at one of its decode steps:
    bf16 N(0,1) [num_layers][H][64] each, on the CPU; independent of which
    other requests share the batch."""
    gen = torch.Generator()
    gen.manual_seed(hash((seed, request, step, 0x51)) & 0x7FFFFFFF)
    q = _bf16_normal(gen, (num_layers, num_q_heads, HEAD_DIM), "cpu")
    k = _bf16_normal(gen, (num_layers, num_kv_heads, HEAD_DIM), "cpu")
    v = _bf16_normal(gen, (num_layers, num_kv_heads, HEAD_DIM), "cpu")
    return q, k, v
