"""Helpers for the GPU-vs-oracle parity tests.

The GPU side runs through the C ABI (the package binding); the expected side is
the fp64 oracle on host copies of the same seeded inputs. Nothing here computes
any part of the method itself: it moves bytes and picks samples.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads

# Output tolerance for fp32 attention against the fp64 oracle.
ATOL, RTOL = 2e-4, 2e-3


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class DeviceWorkload:
    """A workload's tensors on the GPU, plus the step object running it."""

    def __init__(self, wl: workloads.Workload, pages_per_split: int = 0, device="cuda",
                 fused_q_rot: bool = True, rope_positions: int | None = None):
        from paged_kv_decode_rope_gb300 import DecodeStep
        self.wl = wl
        self.pool = wl.pool.to(device, copy=True).contiguous()  # wl.pool stays the "before" state
        self.q, self.k, self.v = (t.to(device).contiguous() for t in (wl.q, wl.k, wl.v))
        self.block_tables = torch.from_numpy(wl.block_tables).to(device)
        self.seq_lens = torch.from_numpy(wl.seq_lens).to(device)
        self.positions = torch.from_numpy(wl.positions).to(device)
        self.step = DecodeStep(self.pool, num_kv_heads=wl.num_kv_heads, num_q_heads=wl.num_q_heads,
                               num_layers=wl.num_layers, block_tables=self.block_tables,
                               seq_lens=self.seq_lens, positions=self.positions,
                               rope_theta=wl.rope_theta, scale=wl.scale,
                               pages_per_split=pages_per_split, fused_q_rot=fused_q_rot,
                               rope_positions=rope_positions)

    def run(self, fused: bool = True):
        out = self.step.run(self.q, self.k, self.v, fused=fused)
        torch.cuda.synchronize()
        return out


def oracle_layer(pool_u16: np.ndarray, wl: workloads.Workload, layer: int, q, k, v,
                 seqs=None):
    """Oracle append (into pool_u16, in place) then decode for one layer.

    q/k/v are host bf16 bit arrays [B,H,64] of that layer. With ``seqs`` only
    those sequences are processed (their rows of q/k/v, tables and lengths).
    Returns (q_rot fp64, out fp64) for the processed sequences.
    """
    bt = wl.block_tables[layer]
    sl, pos = wl.seq_lens, wl.positions
    if seqs is not None:
        seqs = np.asarray(seqs)
        bt, sl, pos, q, k, v = bt[seqs], sl[seqs], pos[seqs], q[seqs], k[seqs], v[seqs]
    n = len(sl)
    q_rot = oracle.append_rope(pool_u16, num_kv_heads=wl.num_kv_heads, q=q, k=k, v=v,
                               block_tables=bt, max_blocks=wl.max_blocks, seq_lens=sl,
                               positions=pos, batch=n, num_q_heads=wl.num_q_heads,
                               theta=wl.rope_theta)
    out = oracle.gqa_decode(pool_u16, num_kv_heads=wl.num_kv_heads, q_rot=q_rot, block_tables=bt,
                            max_blocks=wl.max_blocks, seq_lens=sl, batch=n,
                            num_q_heads=wl.num_q_heads, scale=wl.scale)
    return q_rot, out


def gather_pages(pool_dev: torch.Tensor, wl: workloads.Workload, layer: int, seqs):
    """Copy only the pages that (layer, seqs) use to a compact host pool.

    Returns (pool_u16 compact, block tables remapped to it)."""
    bt = wl.block_tables[layer][np.asarray(seqs)]
    used = np.unique(bt[bt >= 0])
    remap = np.full(wl.num_pages, -1, dtype=np.int64)
    remap[used] = np.arange(len(used))
    pages = pool_dev.view(wl.num_pages, -1)[torch.from_numpy(used).to(pool_dev.device)]
    compact = u16(pages).reshape(-1).copy()
    bt2 = np.where(bt >= 0, remap[np.maximum(bt, 0)], -1).astype(np.int32)
    return compact, bt2


def assert_close(got: np.ndarray, want: np.ndarray, what: str):
    got = np.asarray(got, dtype=np.float64)
    bad = np.abs(got - want) > ATOL + RTOL * np.abs(want)
    if bad.any() or not np.all(np.isfinite(got)):
        idx = np.argwhere(bad | ~np.isfinite(got))[:5]
        err = np.max(np.abs(got - want))
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside atol {ATOL} + rtol {RTOL}; "
                             f"max |err| {err:.3g}; first at {idx.tolist()}")
    return float(np.max(np.abs(got - want))) if got.size else 0.0
