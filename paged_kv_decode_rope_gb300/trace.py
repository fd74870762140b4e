"""Multi-step decode traces: continuous batching over the shared page pool.

A PageScheduler admits requests under their page budgets and hands out pages
lazily. The requests admitted in one pass are prefilled together through the
C ABI (paged_prefill: their prompts' keys rotated and stored in their pages,
causal attention over the prompt), in calls of at most prefill_tokens chunk
tokens, a long prompt split into chunks over several calls. Then every step
runs the fused decode step (RoPE, append, paged GQA decode) for the active
batch, whose sequences grow by one token per step and cross page boundaries
as they go. This is the batched engine loop of "Hours of YouTube and 85
handtyped pages of notes on LLM Inference – Start here" (continuous batching
and dense causal prefill items) around this library's kernels; the model's
projections are not part of the library, so every prompt and step token
brings its q/k/v from the caller: either two callables (a request's prompt
rows, a request's step rows) or, for timing, a seeded draw on the device.

Per request: after its prefill it holds prompt_len tokens and has produced its
first token; each decode step processes the newest token (appending it at its
absolute position, which is the current length) and produces the next; it
stops after stop_after generated tokens, so at most prompt + max_new - 1
tokens are ever processed: the budget the scheduler reserved.
"""
from __future__ import annotations

import time

import numpy as np
import torch

from . import _binding as B
from .sched import PageScheduler


def pack_prefill_chunks(requests, prompt_lens, budget: int):
    """Chunks (request, start, length) of the prompts, packed in order into calls
    of at most budget tokens. A prompt that does not fit the rest of a call
    continues in the next one, so a call never holds two chunks of one request
    (a chunk's attention reads the pages its earlier chunks stored)."""
    if budget < 1:
        raise ValueError("budget must be positive")
    calls, cur, room = [], [], budget
    for r, n_tok in zip(requests, prompt_lens):
        start, left = 0, int(n_tok)
        while left > 0:
            n = min(left, room)
            cur.append((r, start, n))
            start, left, room = start + n, left - n, room - n
            if room == 0:
                calls.append(cur)
                cur, room = [], budget
    if cur:
        calls.append(cur)
    return calls


class DecodeTrace:
    def __init__(self, requests, *, num_pages: int, num_layers: int, num_q_heads: int,
                 num_kv_heads: int, rope_theta: float, seed: int = 0, context_len: int = 2048,
                 static_batching: bool = False, max_batch: int = 256, device="cuda",
                 device_inputs: bool = False, prefill_tokens: int = 8192,
                 prompt_qkv=None, step_qkv=None):
        """prompt_qkv(request, prompt_len) -> (q [L][T][Hq][64], k, v [L][T][Hkv][64])
        and step_qkv(request, step) -> (q [L][Hq][64], k, v [L][Hkv][64]), bf16
        host tensors, give each request's inputs independently of the batch it
        shares (for parity checks). With device_inputs=True they are not used:
        every call draws its rows on the device from a generator seeded with
        `seed` (for timing)."""
        if not device_inputs and (prompt_qkv is None or step_qkv is None):
            raise ValueError("give prompt_qkv and step_qkv, or device_inputs=True")
        self._prompt_src, self._step_src = prompt_qkv, step_qkv
        self.requests = list(requests)
        self.num_layers, self.hq, self.hkv = num_layers, num_q_heads, num_kv_heads
        self.rope_theta, self.seed = float(rope_theta), seed
        self.scale = 1.0 / float(np.sqrt(B.HEAD_DIM))
        self.max_blocks = (context_len + B.PAGE_SIZE - 1) // B.PAGE_SIZE
        self.max_batch = max_batch
        self.device = torch.device(device)
        self.sched = PageScheduler(num_pages, num_layers, context_len, static_batching, seed=seed + 1)
        page_elems = 2 * num_kv_heads * B.PAGE_SIZE * B.HEAD_DIM
        self.pool = torch.zeros(num_pages * page_elems, dtype=torch.bfloat16, device=self.device)
        self.kvpool = B.kv_pool_create(self.pool, num_kv_heads)
        # cos/sin of every position up to the context length, built once
        self.rope = B.build_rope_table(self.rope_theta, self.max_blocks * B.PAGE_SIZE,
                                       device=self.device)
        self.ws = B.alloc_decode_workspace(max_batch, num_q_heads, num_kv_heads, self.max_blocks,
                                           device=self.device)
        self.ids = {}        # request index -> scheduler id
        self.state = {}      # request index -> [kv_len, generated, steps_done]
        self.rows = {}       # request index -> [num_layers][max_blocks] int32 page rows
        self.waiting = list(range(len(self.requests)))
        self.done = []
        self.steps = 0
        self.tokens = 0      # decode tokens processed
        self.kv_bytes = 0    # KV bytes the decode steps read (valid tokens)
        self.device_ms = 0.0
        self.prefill_tokens = int(prefill_tokens)
        if self.prefill_tokens < 1:
            raise ValueError("prefill_tokens must be positive")
        self.prefill_calls = 0
        self.prompt_tokens = 0
        self.prefill_ms = 0.0
        # device_inputs: draw each step's q/k/v on the GPU in one call (for
        # timing); otherwise per (request, step) on the host (reproducible
        # whatever the batch, for parity checks)
        self.device_inputs = device_inputs
        self._gen = torch.Generator(device=self.device)
        self._gen.manual_seed(seed)
        self._prompts = {}   # request index -> its prompt q/k/v (host inputs)

    # -- host side -----------------------------------------------------------
    def _prompt_qkv(self, r: int):
        if r not in self._prompts:
            self._prompts[r] = self._prompt_src(r, self.requests[r].prompt_len)
        return self._prompts[r]

    def run_prefill(self, chunks, on_prefill=None) -> None:
        """One paged_prefill per layer over the chunks [(request, start, length)]."""
        dev = self.device
        nb = len(chunks)
        lens = np.array([c[2] for c in chunks], dtype=np.int32)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        start = np.array([c[1] for c in chunks], dtype=np.int32)
        total = int(cu[-1])
        bt = np.stack([self.rows[c[0]] for c in chunks], axis=1)  # [L][B][max_blocks]
        if self.device_inputs:
            def draw(h):
                return torch.randn((self.num_layers, total, h, B.HEAD_DIM), generator=self._gen,
                                   device=dev).to(torch.bfloat16)
            q, k, v = draw(self.hq), draw(self.hkv), draw(self.hkv)
        else:
            parts = [self._prompt_qkv(r) for r, _, _ in chunks]
            q, k, v = (torch.cat([p[i][:, s:s + n] for p, (_, s, n) in zip(parts, chunks)], dim=1)
                       .to(dev) for i in range(3))
        d_cu = torch.from_numpy(cu).to(dev)
        d_start = torch.from_numpy(start).to(dev)
        d_bt = torch.from_numpy(np.ascontiguousarray(bt)).to(dev)
        q_rot = torch.empty(self.num_layers, total, self.hq, B.HEAD_DIM, dtype=torch.float32,
                            device=dev)
        out = torch.empty_like(q_rot)
        ws = B.alloc_prefill_workspace(total, nb, self.max_blocks, device=dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for layer in range(self.num_layers):
            B.paged_prefill(self.kvpool, q[layer], k[layer], v[layer], q_rot[layer], out[layer],
                            d_bt[layer], d_cu, d_start, self.rope, self.scale, ws)
        e1.record()
        torch.cuda.synchronize()
        self.prefill_ms += e0.elapsed_time(e1)
        self.prefill_calls += 1
        self.prompt_tokens += total
        if on_prefill is not None:
            on_prefill(chunks, (cu, start, bt, q, k, v), q_rot, out)

    def _refresh_rows(self, r: int) -> None:
        self.rows[r] = self.sched.block_rows(self.ids[r], self.max_blocks)

    def admit(self, on_admit=None, on_prefill=None) -> list[int]:
        """Submit what is waiting (once) and admit under the budgets; prefill the
        admitted. on_admit(r, rows) sees each admitted request's page rows,
        on_prefill(chunks, inputs, q_rot, out) every prefill call."""
        for r in self.waiting:
            if r not in self.ids:
                req = self.requests[r]
                self.ids[r] = self.sched.submit(req.prompt_len, req.max_new)
        by_id = {v: k for k, v in self.ids.items()}
        admitted = [by_id[i] for i in self.sched.admit()]
        for r in admitted:
            self.waiting.remove(r)
            self.sched.grow(self.ids[r], self.requests[r].prompt_len)
            self._refresh_rows(r)
            if on_admit is not None:
                on_admit(r, self.rows[r])
        lens = [self.requests[r].prompt_len for r in admitted]
        for chunks in pack_prefill_chunks(admitted, lens, self.prefill_tokens):
            self.run_prefill(chunks, on_prefill)
        for r in admitted:
            req = self.requests[r]
            self._prompts.pop(r, None)
            self.state[r] = [req.prompt_len, 1, 0]
            if req.stop_after <= 1:  # its only token came from the prefill
                self._finish(r)
        return admitted

    def _finish(self, r: int) -> None:
        self.sched.finish(self.ids[r])
        del self.state[r]
        self.rows.pop(r, None)
        self.done.append(r)

    def batch(self) -> list[int]:
        return sorted(self.state)

    # -- one decode step -----------------------------------------------------
    def step_inputs(self, batch: list[int]):
        """Host tensors of one step: positions, seq_lens, block tables
        [L][B][max_blocks], and q/k/v [L][B][H][64] (bf16)."""
        nb = len(batch)
        pos = np.empty(nb, dtype=np.int32)
        for j, r in enumerate(batch):
            kv_len = self.state[r][0]
            if kv_len % B.PAGE_SIZE == 0:  # the new token opens a page
                self.sched.grow(self.ids[r], kv_len + 1)
                self._refresh_rows(r)
            pos[j] = kv_len
        bt = np.stack([self.rows[r] for r in batch], axis=1)  # [L][B][max_blocks]
        if self.device_inputs:
            def draw(h):
                return torch.randn((self.num_layers, nb, h, B.HEAD_DIM), generator=self._gen,
                                   device=self.device).to(torch.bfloat16)
            q, k, v = draw(self.hq), draw(self.hkv), draw(self.hkv)
            return pos, pos + 1, bt, q, k, v
        qkv = [self._step_src(r, self.state[r][2]) for r in batch]
        q = torch.stack([x[0] for x in qkv], dim=1)
        k = torch.stack([x[1] for x in qkv], dim=1)
        v = torch.stack([x[2] for x in qkv], dim=1)
        return pos, pos + 1, bt, q, k, v

    def run_step(self, pos, seq_lens, bt, q, k, v):
        """The fused decode step of every layer for this batch; returns out [L][B][Hq][64] fp32."""
        dev = self.device
        nb = len(pos)
        d_pos = torch.from_numpy(pos).to(dev)
        d_sl = torch.from_numpy(seq_lens).to(dev)
        d_bt = torch.from_numpy(np.ascontiguousarray(bt)).to(dev)
        dq, dk, dv = q.to(dev), k.to(dev), v.to(dev)
        out = torch.empty(self.num_layers, nb, self.hq, B.HEAD_DIM, dtype=torch.float32, device=dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for layer in range(self.num_layers):
            B.paged_decode_step(self.kvpool, dq[layer], dk[layer], dv[layer], self.rope, d_pos,
                                out[layer], d_bt[layer], d_sl, self.scale, self.ws)
        e1.record()
        torch.cuda.synchronize()
        self.device_ms += e0.elapsed_time(e1)
        return out

    def advance(self, batch: list[int], seq_lens) -> None:
        for j, r in enumerate(batch):
            st = self.state[r]
            st[0] += 1
            st[1] += 1
            st[2] += 1
            self.kv_bytes += int(seq_lens[j]) * self.hkv * B.HEAD_DIM * 2 * 2 * self.num_layers
            if st[1] >= self.requests[r].stop_after:
                self._finish(r)
        self.tokens += len(batch)
        self.steps += 1

    def run(self, on_step=None, on_admit=None, on_prefill=None,
            max_steps: int = 1_000_000) -> dict:
        """Drive the trace to completion. on_step(batch, inputs, out) sees every
        decode step, on_admit(r, rows) every admission, on_prefill(chunks,
        inputs, q_rot, out) every prefill call."""
        t0 = time.perf_counter()
        while (self.waiting or self.state) and self.steps < max_steps:
            self.admit(on_admit, on_prefill)
            batch = self.batch()
            if not batch:
                if self.waiting and not self.state:
                    continue  # everything finished at its prefill; admit more
                break
            if len(batch) > self.max_batch:
                raise RuntimeError("decode batch larger than max_batch")
            self.sched.note_batch(len(batch))
            inputs = self.step_inputs(batch)
            out = self.run_step(*inputs)
            if on_step is not None:
                on_step(batch, inputs, out)
            self.advance(batch, inputs[1])
        wall = time.perf_counter() - t0
        if B.pkv_get_error(self.kvpool):
            raise RuntimeError("device error flags set during the trace")
        return {"steps": self.steps, "decode_tokens": self.tokens, "kv_bytes": self.kv_bytes,
                "device_ms": self.device_ms, "wall_s": wall, "completed": len(self.done),
                "prefill_calls": self.prefill_calls, "prompt_tokens": self.prompt_tokens,
                "prefill_ms": self.prefill_ms,
                "sched": self.sched.stats()}

    def close(self) -> None:
        self.kvpool.close()
        self.sched.close()
