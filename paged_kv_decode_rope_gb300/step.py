"""One batched decode step over all layers, through the C ABI.

Per layer l, on one stream: RoPE of the new token's q and k at its position
and the append of its K/V into the layer's pages, then every query head's
attention over its sequence's pages. By default one ``paged_decode_step``
call does both; with ``fused=False`` the two separate entry points
``paged_kv_append_rope`` and ``paged_gqa_decode`` run instead. This is
the decode half of the per-layer loop the "Hours of YouTube and 85 handtyped
pages of notes on LLM Inference – Start here" engine runs for each packed
decode batch (its batched decode item); the projections around it are not
part of this library.
"""
from __future__ import annotations

import torch

from . import _binding as B


class DecodeStep:
    def __init__(self, pool_storage: torch.Tensor, *, num_kv_heads: int, num_q_heads: int,
                 num_layers: int, block_tables: torch.Tensor, seq_lens: torch.Tensor,
                 positions: torch.Tensor, rope_theta: float, scale: float,
                 pages_per_split: int = 0):
        dev = pool_storage.device
        self.num_layers = num_layers
        self.batch = int(seq_lens.shape[0])
        self.num_q_heads = num_q_heads
        self.num_kv_heads = num_kv_heads
        self.rope_theta = float(rope_theta)
        self.scale = float(scale)
        self.pages_per_split = pages_per_split
        self.pool = B.kv_pool_create(pool_storage, num_kv_heads)
        self.block_tables = block_tables
        self.seq_lens = seq_lens
        self.positions = positions
        self.max_blocks = int(block_tables.shape[-1])
        self.q_rot = torch.empty(num_layers, self.batch, num_q_heads, B.HEAD_DIM,
                                 dtype=torch.float32, device=dev)
        self.out = torch.empty_like(self.q_rot)
        self.workspace = B.alloc_decode_workspace(self.batch, num_q_heads, num_kv_heads,
                                                  self.max_blocks, pages_per_split, device=dev)
        self.rope_cos_sin = B.alloc_rope_table(self.batch, device=dev)

    def launches_per_step(self, fused: bool = True) -> int:
        """Kernels one step launches: per layer and batch chunk of 2048 a decode
        and a merge, plus per layer the append kernel when not fused, or once
        per step the cos/sin table when fused."""
        if not self.batch:
            return 0
        chunks = -(-self.batch // 2048)
        return self.num_layers * (2 * chunks + (0 if fused else 1)) + (1 if fused else 0)

    def append(self, layer: int, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, stream=None) -> None:
        B.paged_kv_append_rope(self.pool, q[layer], k[layer], v[layer], self.q_rot[layer],
                               self.block_tables[layer], self.seq_lens, self.positions,
                               self.rope_theta, stream)

    def decode(self, layer: int, stream=None) -> None:
        B.paged_gqa_decode(self.pool, self.q_rot[layer], self.out[layer], self.block_tables[layer],
                           self.seq_lens, self.scale, self.workspace, self.pages_per_split, stream)

    def rope_table(self, stream=None) -> None:
        """The step's cos/sin table (same positions in every layer)."""
        B.paged_rope_cos_sin(self.positions, self.rope_theta, self.rope_cos_sin, stream)

    def fused_layer(self, layer: int, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                    stream=None) -> None:
        B.paged_decode_step(self.pool, q[layer], k[layer], v[layer], self.rope_cos_sin, self.out[layer],
                            self.block_tables[layer], self.seq_lens, self.scale, self.workspace,
                            q_rot=self.q_rot[layer], pages_per_split=self.pages_per_split,
                            stream=stream)

    def run(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, stream=None,
            fused: bool = True) -> torch.Tensor:
        """q [NL,B,Hq,64], k/v [NL,B,Hkv,64] bf16 on the device -> out [NL,B,Hq,64] fp32."""
        if fused:
            self.rope_table(stream)
        for layer in range(self.num_layers):
            if fused:
                self.fused_layer(layer, q, k, v, stream)
            else:
                self.append(layer, q, k, v, stream)
                self.decode(layer, stream)
        return self.out

    def error_bits(self, reset: bool = False) -> int:
        return B.pkv_get_error(self.pool, reset)

    def close(self) -> None:
        self.pool.close()
