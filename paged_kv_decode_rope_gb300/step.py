"""One batched decode step over all layers, through the C ABI.

Once per step, the decode's work plan (``paged_decode_plan``: the partition
of the work over the warps depends only on the sequence lengths, the same in
every layer). Then per layer l, on one stream: RoPE of the new token's q and
k at its position and the append of its K/V into the layer's pages, then
every query head's attention over its sequence's pages. By default one
``paged_decode_step`` call does both; with ``fused=False`` the two separate
entry points ``paged_kv_append_rope`` and ``paged_gqa_decode`` run instead. This is
the decode half of the per-layer loop the "Hours of YouTube and 85 handtyped
pages of notes on LLM Inference – Start here" engine runs for each packed
decode batch (its batched decode item); the projections around it are not
part of this library.
"""
from __future__ import annotations

import torch

from . import _binding as B


def host_copy_groups(num_layers: int) -> list[tuple[int, int]]:
    """Layer ranges [lo, hi) whose inputs DecodeStep.run_from_host copies
    together: layer 0, layers 1-3, the rest (empty ranges dropped)."""
    nl = num_layers
    return [g for g in ((0, 1), (1, min(4, nl)), (min(4, nl), nl)) if g[0] < g[1]]


class DecodeStep:
    def __init__(self, pool_storage: torch.Tensor, *, num_kv_heads: int, num_q_heads: int,
                 num_layers: int, block_tables: torch.Tensor, seq_lens: torch.Tensor,
                 positions: torch.Tensor, rope_theta: float, scale: float,
                 pages_per_split: int = 0, fused_q_rot: bool = True,
                 rope_positions: int | None = None):
        dev = pool_storage.device
        self.num_layers = num_layers
        self.batch = int(seq_lens.shape[0])
        self.num_q_heads = num_q_heads
        self.num_kv_heads = num_kv_heads
        self.rope_theta = float(rope_theta)
        self.scale = float(scale)
        self.pages_per_split = pages_per_split
        # the fused step writes the rotated queries only when asked (the
        # attention itself does not need them in memory)
        self.fused_q_rot = fused_q_rot
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
        # cos/sin of every position a token of these block tables can have,
        # built once (the fused step reads the row of each new token's position)
        self.rope_positions = rope_positions or self.max_blocks * B.PAGE_SIZE
        self.rope = B.build_rope_table(self.rope_theta, self.rope_positions, device=dev)

    def launches_per_step(self, fused: bool = True) -> int:
        """Kernels one step launches: the plan (one-launch batches of at most
        2048 sequences, automatic partition), then per layer one decode per
        batch chunk of 2048, plus the append kernel when not fused (the
        cos/sin table was built once, at construction)."""
        if not self.batch:
            return 0
        chunks = -(-self.batch // 2048)
        plan = 1 if self.plans() else 0
        return plan + self.num_layers * (chunks + (0 if fused else 1))

    def plans(self) -> bool:
        return self.batch <= 2048 and self.pages_per_split == 0

    def plan(self, fused: bool = True, stream=None) -> None:
        """The step's work plan (the lengths and positions of this step)."""
        if not self.plans():
            return
        B.paged_decode_plan(self.pool, self.seq_lens, self.block_tables[0], self.num_q_heads,
                            self.workspace, positions=self.positions if fused else None,
                            rope_table=self.rope if fused else None, stream=stream)

    def append(self, layer: int, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, stream=None) -> None:
        B.paged_kv_append_rope(self.pool, q[layer], k[layer], v[layer], self.q_rot[layer],
                               self.block_tables[layer], self.seq_lens, self.positions,
                               self.rope_theta, stream)

    def decode(self, layer: int, stream=None) -> None:
        B.paged_gqa_decode(self.pool, self.q_rot[layer], self.out[layer], self.block_tables[layer],
                           self.seq_lens, self.scale, self.workspace, self.pages_per_split, stream)

    def fused_layer(self, layer: int, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                    stream=None) -> None:
        B.paged_decode_step(self.pool, q[layer], k[layer], v[layer], self.rope, self.positions,
                            self.out[layer], self.block_tables[layer], self.seq_lens, self.scale,
                            self.workspace,
                            q_rot=self.q_rot[layer] if self.fused_q_rot else None,
                            pages_per_split=self.pages_per_split,
                            stream=stream)

    def run(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, stream=None,
            fused: bool = True) -> torch.Tensor:
        """q [NL,B,Hq,64], k/v [NL,B,Hkv,64] bf16 on the device -> out [NL,B,Hq,64] fp32."""
        self.plan(fused, stream)
        for layer in range(self.num_layers):
            if fused:
                self.fused_layer(layer, q, k, v, stream)
            else:
                self.append(layer, q, k, v, stream)
                self.decode(layer, stream)
        return self.out

    def run_from_host(self, host_in: dict, dev_in: dict, host_out: torch.Tensor,
                      copy_streams=None) -> None:
        """One step with its inputs in pinned host memory, layer-pipelined.

        host_in / dev_in map "q", "k", "v" ([NL,...] bf16), "block_tables"
        ([NL,...] int32), "seq_lens" and "positions" to pinned host tensors and
        their device copies (dev_in's tables, lengths and positions must be the
        tensors this step was built with). The step (fused path) runs on the
        current stream. copy_streams[0] copies the layers' block tables and
        q/k/v in three groups: layer 0 (with the lengths and positions), the
        next three layers (they land while layer 0 runs), then the rest (while
        layers 0-3 run). The step waits for each group just before its first
        layer; the step's plan runs once the first group, with the lengths
        and positions, has landed. Each such wait costs the chain of decode launches its
        programmatic overlap at that layer, several microseconds, so the
        groups are few; more, smaller ones (1, 1, 2, 4, ... layers) were 5-13
        us per step slower on batch 64 and the Qwen shape. copy_streams[1]
        copies each layer's output back to host_out as soon as that layer is
        done. The current stream finally waits for both copy streams.
        """
        cur = torch.cuda.current_stream()
        cs_in, cs_out = copy_streams or (torch.cuda.Stream(), torch.cuda.Stream())
        nl = self.num_layers
        cs_in.wait_stream(cur)
        cs_out.wait_stream(cur)
        groups = host_copy_groups(nl)
        ready = []
        with torch.cuda.stream(cs_in):
            for lo, hi in groups:
                dev_in["block_tables"][lo:hi].copy_(host_in["block_tables"][lo:hi], non_blocking=True)
                if lo == 0:
                    for key in ("seq_lens", "positions"):
                        dev_in[key].copy_(host_in[key], non_blocking=True)
                for key in ("q", "k", "v"):
                    dev_in[key][lo:hi].copy_(host_in[key][lo:hi], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(cs_in)
                ready.append((lo, ev))
        ev_done = [torch.cuda.Event() for _ in range(nl)]
        for layer in range(nl):
            for lo, ev in ready:
                if lo == layer:
                    cur.wait_event(ev)
            if layer == 0:
                self.plan()
            self.fused_layer(layer, dev_in["q"], dev_in["k"], dev_in["v"])
            ev_done[layer].record(cur)
        with torch.cuda.stream(cs_out):
            for layer in range(nl):
                cs_out.wait_event(ev_done[layer])
                host_out[layer].copy_(self.out[layer], non_blocking=True)
        cur.wait_stream(cs_out)
        cur.wait_stream(cs_in)

    def error_bits(self, reset: bool = False) -> int:
        return B.pkv_get_error(self.pool, reset)

    def close(self) -> None:
        self.pool.close()
