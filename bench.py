#!/usr/bin/env python3
"""Benchmark of the batched paged-KV decode step on GB300.

A step is one pass of the whole hot path over one batch: for every layer,
RoPE + append of the new token (paged_kv_append_rope) and paged GQA decode
with split-KV and its fused log-sum-exp merge (paged_gqa_decode).

Prints ONE JSON line (rank 0). The metric is decode-attention KV read GB/s
(algorithmic bytes: K and V of every valid token, per layer, per step) over the
device-timed step; the line also carries us per step, the decode kernel's
roofline, an end-to-end figure with host buffers, the fp64 oracle's CPU
baseline, and the SM clocks seen during the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

With N > 1 (torchrun) every rank runs an independent replica of the workload
(different seed) on its own GPU: the path has no exchange step, so there is no
data-path collective; the barrier and the max over ranks use torch.distributed.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

DEFAULT_WORKLOAD = "llama1b_b64_l16_u2048"
METRIC = "decode-attention KV read GB/s (% of GB300 HBM peak); us per batched decode step"
L2_BYTES = 129 * 10**6

# DRAM traffic (read + write bytes) per decode launch from one ncu capture, with
# the hash of the decode source it was taken on; reported only while the source
# is unchanged.
TRAFFIC = {
    # (workload, seed) -> (sha256 prefix of gqa_decode.cu, read + write bytes per layer call),
    # ncu dram__bytes_read.sum + dram__bytes_write.sum of the first layer launches of a 2-layer
    # copy of the workload (same lengths, pool fitted), mean over the eager warm-up launches
    ("llama1b_b64_l16_u2048", 0): ("82a357034b7135d5", 158961451),
    ("llama1b_b64_l16_u2048", 1): ("82a357034b7135d5", 142436266),
    ("llama1b_b64_l16_u2048", 2): ("82a357034b7135d5", 143683242),
    ("llama1b_b64_l16_u2048", 3): ("82a357034b7135d5", 130654805),
    ("llama1b_b64_l16_u2048", 4): ("82a357034b7135d5", 138696533),
    ("llama1b_b256_l16_skew", 0): ("82a357034b7135d5", 156204928),
    ("llama1b_b256_l16_skew", 1): ("82a357034b7135d5", 157123200),
    ("llama1b_b256_l16_skew", 2): ("82a357034b7135d5", 154208000),
    ("llama1b_b256_l16_skew", 3): ("82a357034b7135d5", 147307605),
    ("llama1b_b256_l16_skew", 4): ("82a357034b7135d5", 147698901),
    ("qwen05b_b32_l24_u1024_4096", 0): ("82a357034b7135d5", 47021568),
    ("qwen05b_b32_l24_u1024_4096", 1): ("82a357034b7135d5", 44072491),
    ("qwen05b_b32_l24_u1024_4096", 2): ("82a357034b7135d5", 42225579),
    ("qwen05b_b32_l24_u1024_4096", 3): ("82a357034b7135d5", 41516715),
    ("qwen05b_b32_l24_u1024_4096", 4): ("82a357034b7135d5", 43569621),
}
# DRAM traffic (read + write bytes) per prefill_tc_kernel launch, one layer of
# a fresh-prompt pass, from one ncu capture (mean of three launches), with the
# hash of the prefill source it was taken on; reported only while unchanged.
PREFILL_TRAFFIC = {
    # (sequences, prompt tokens) -> (sha256 prefix of prefill.cu, read + write bytes per launch)
    (4, 2048): ("48b626bfea4feb4a", 111688704),
}
# The other workloads the 70% target names, timed as sub-records of the default line.
SUB_WORKLOADS = ["llama1b_b256_l16_skew", "qwen05b_b32_l24_u1024_4096"]


def _source_hash(name: str) -> str:
    p = os.path.join(ROOT, "paged_kv_decode_rope_gb300", "csrc", name)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def _decode_source_hash() -> str:
    return _source_hash("gqa_decode.cu")


def _peaks() -> tuple[float, str]:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _tensor_peak(sustained: bool = True) -> tuple[float, str]:
    """Dense bf16 TFLOP/s: the measured cuBLAS rate (sustained for a kernel
    timed inside a long loop, burst for one timed alone), else the fallback."""
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)[key]), "measured"
    except Exception:
        return (1700.0 if sustained else 1900.0), "fallback"


def prefill_roofline(pairs: float, ms: float, peak: float, source: str, traffic: int | None = None) -> dict:
    """The prefill pass's roofline: causal attention is a dense contraction,
    bound by the bf16 tensor cores. Algorithmic flops are 2 products x 2 x 64
    per (query head, visible key) pair; the kernel's hi/lo operand split and
    the masked halves of diagonal steps are work on top of that, not counted.
    traffic: the attention kernel's DRAM bytes per launch, where measured."""
    achieved = pairs * 4 * 64 / (ms / 1e3) / 1e12
    return {"bound": "tensor", "kernel": "prefill_tc_kernel (tcgen05), with the pass's append",
            "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4), "traffic": traffic,
            "peak_source": f"{source} (MEASURED_PEAKS.json bf16_tflops_sustained, cuBLAS bf16)"
                           if source == "measured" else "fallback (1.7 PFLOP/s sustained)",
            "flops_per_pass": pairs * 4 * 64}


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.proc = None
        self.path = None
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            ident = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            ident = str(device)
        self.ident = ident

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.ident, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        try:
            with open(self.path) as f:
                lines = f.readlines()
            os.unlink(self.path)
            return summarise_clocks(lines)
        except Exception:
            return None


def summarise_clocks(lines) -> dict | None:
    """Median SM clock, the largest max clock and every throttle reason seen
    Active, from nvidia-smi CSV lines in ClockSampler.FIELDS order (no header,
    no units). None when no line parses."""
    rows = []
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) >= 9:
            rows.append(parts)
    if not rows:
        return None

    def num(x):
        try:
            return float(x)
        except ValueError:
            return None

    sm = [v for v in (num(r[1]) for r in rows) if v is not None]
    mx = [v for v in (num(r[2]) for r in rows) if v is not None]
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
            "reasons": reasons, "samples": len(rows)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _barrier_max(value: float, ws: int) -> float:
    if ws == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _barrier_sum(value: float, ws: int) -> float:
    if ws == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def _barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def _config(wl: workloads.Workload) -> dict:
    step_bytes = wl.kv_bytes_per_step()
    return {"workload": wl.name, "batch": wl.batch, "layers": wl.num_layers, "q_heads": wl.num_q_heads,
            "kv_heads": wl.num_kv_heads, "head_dim": 64, "page_size": 16,
            "seq_len_min": int(wl.seq_lens.min()), "seq_len_max": int(wl.seq_lens.max()),
            "seq_len_mean": round(float(wl.seq_lens.mean()), 1), "pool_pages": wl.num_pages,
            "kv_bytes_per_step": step_bytes,
            "l2": ("inputs larger than L2: %.2f GB of KV per step vs 129 MB L2, every layer reads distinct pages"
                   % (step_bytes / 1e9)) if step_bytes > 4 * L2_BYTES else
                  "L2 flushed before every timed step (write of 2x L2)",
            "description": wl.description}


def oracle_sample_step(wl: workloads.Workload, pool_src: torch.Tensor, layer: int, seqs: np.ndarray):
    """One sampled step of the fp64 oracle: append + decode of `seqs` in `layer`.

    Returns (KV bytes read, seconds). Only the pages these sequences use are
    copied to the host (outside the timed part)."""
    import oracle
    bt = wl.block_tables[layer][seqs]
    used = np.unique(bt[bt >= 0])
    remap = np.full(wl.num_pages, -1, dtype=np.int64)
    remap[used] = np.arange(len(used))
    pages = pool_src.view(wl.num_pages, -1)[torch.from_numpy(used).to(pool_src.device)]
    mini = pages.contiguous().view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1).copy()
    bt2 = np.where(bt >= 0, remap[np.maximum(bt, 0)], -1).astype(np.int32)
    u = lambda t: t[layer][torch.from_numpy(seqs).to(t.device)].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)  # noqa: E731
    q, k, v = u(wl.q), u(wl.k), u(wl.v)
    sl, pos = wl.seq_lens[seqs], wl.positions[seqs]
    t0 = time.perf_counter()
    q_rot = oracle.append_rope(mini, num_kv_heads=wl.num_kv_heads, q=q, k=k, v=v, block_tables=bt2,
                               max_blocks=wl.max_blocks, seq_lens=sl, positions=pos, batch=len(seqs),
                               num_q_heads=wl.num_q_heads, theta=wl.rope_theta)
    oracle.gqa_decode(mini, num_kv_heads=wl.num_kv_heads, q_rot=q_rot, block_tables=bt2,
                      max_blocks=wl.max_blocks, seq_lens=sl, batch=len(seqs),
                      num_q_heads=wl.num_q_heads, scale=wl.scale)
    dt = time.perf_counter() - t0
    nbytes = int(sl.astype(np.int64).sum()) * wl.num_kv_heads * 64 * 2 * 2
    return nbytes, dt


def cpu_baseline(wl, pool_src, budget_s: float = 10.0, max_passes: int = 8) -> dict:
    """The oracle as it stands, single-threaded, on a bounded sample of the workload:
    whole steps (every sequence of every layer), repeated until budget_s has passed."""
    total_b, total_t, layers = 0, 0.0, 0
    seqs = np.arange(wl.batch)
    for _ in range(max_passes):
        for layer in range(wl.num_layers):
            b, t = oracle_sample_step(wl, pool_src, layer, seqs)
            total_b += b
            total_t += t
            layers += 1
            if total_t >= 2 * budget_s:
                break
        if total_t >= budget_s:
            break
    return {"value": round(total_b / total_t / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"fp64 C oracle, 1 thread: append+decode of all {wl.batch} sequences, "
                      f"{layers} layer passes ({layers / wl.num_layers:.2f} steps, {total_b / 1e9:.2f} GB of KV, "
                      f"{total_t:.1f} s)"}


def run_reference(args, ws, rank):
    if rank != 0:
        return 0
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    wl = workloads.make(args.workload, seed=args.seed, device=dev, layers=args.layers)
    rng = np.random.default_rng(7)
    nseq = max(1, min(wl.batch, 4))
    samples = [(i % wl.num_layers, np.sort(rng.choice(wl.batch, size=nseq, replace=False)))
               for i in range(args.warmup + args.steps)]
    for layer, seqs in samples[:args.warmup]:
        oracle_sample_step(wl, wl.pool, layer, seqs)
    tb, tt = 0, 0.0
    for layer, seqs in samples[args.warmup:]:
        b, t = oracle_sample_step(wl, wl.pool, layer, seqs)
        tb += b
        tt += t
    value = tb / tt / 1e9
    step_ms = tt / args.steps * 1e3
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)", "config": _config(wl),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"each step: fp64 C oracle append+decode of {nseq} of {wl.batch} "
                                       f"sequences of one layer (layers in turn)"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def _timed_step(pkv, wl, dev, args, ws) -> tuple[dict, object]:
    """Device time of one whole step of ``wl``: warm-up, one CUDA graph of the
    step (every layer's fused call), W untimed replays, then K replays timed
    with CUDA events between a barrier and a synchronize; the max over ranks.
    Workloads whose step reads less than 4x L2 get an L2 flush (a write of
    2x L2) before every timed replay. Returns the figures and the step."""
    bt = torch.from_numpy(wl.block_tables).to(dev)
    sl = torch.from_numpy(wl.seq_lens).to(dev)
    pos = torch.from_numpy(wl.positions).to(dev)
    step = pkv.DecodeStep(wl.pool, num_kv_heads=wl.num_kv_heads, num_q_heads=wl.num_q_heads,
                          num_layers=wl.num_layers, block_tables=bt, seq_lens=sl, positions=pos,
                          rope_theta=wl.rope_theta, scale=wl.scale, pages_per_split=args.pages_per_split,
                          fused_q_rot=False)
    stream = torch.cuda.current_stream()
    step_bytes = wl.kv_bytes_per_step()
    flush = None
    if step_bytes <= 4 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    for _ in range(3):  # eager warm-up (first calls cache kernel attributes)
        step.run(wl.q, wl.k, wl.v)
    torch.cuda.synchronize()
    assert step.error_bits() == 0, "device error flags set during warm-up"
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step.run(wl.q, wl.k, wl.v)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    _barrier(ws)
    torch.cuda.synchronize()
    if flush is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
    else:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for s in range(args.steps):
            flush.fill_(float(s))
            evs[s][0].record(stream)
            graph.replay()
            evs[s][1].record(stream)
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
    _barrier(ws)
    ms_max = _barrier_max(ms, ws)
    total_bytes = _barrier_sum(float(step_bytes), ws)
    assert step.error_bits() == 0, "device error flags set during the timed steps"
    del graph
    return {"ms": ms_max, "value": total_bytes / (ms_max / 1e3) / 1e9, "kv_bytes_per_step": step_bytes,
            "layer_bytes": wl.kv_bytes_per_layer(), "layers": wl.num_layers,
            "launches": step.launches_per_step() * args.steps, "flush": flush is not None,
            "seq_len_mean": round(float(wl.seq_lens.mean()), 1)}, step


def _seed_sweep(pkv, name, seeds, dev, args, ws, rank) -> list[dict]:
    """_timed_step of workload ``name`` at each seed (rank r adds 1000 r)."""
    runs = []
    for sd in seeds:
        wl = workloads.make(name, seed=sd + 1000 * rank, device=dev, layers=args.layers)
        r, step = _timed_step(pkv, wl, dev, args, ws)
        r["seed"] = sd
        runs.append(r)
        step.close()
        del wl, step
        torch.cuda.empty_cache()
    return runs


def _median_run(runs: list[dict]) -> dict:
    return sorted(runs, key=lambda r: r["value"])[len(runs) // 2]


def _roofline(r: dict, name: str, seed: int, peak: float, peak_kind: str, steps: int) -> dict:
    """The decode kernel's roofline from a _timed_step result: algorithmic K/V
    bytes of one layer call over the mean layer-call time in graph replays."""
    dec_avg_s = r["ms"] / r["layers"] / 1e3
    achieved = r["layer_bytes"] / dec_avg_s / 1e9
    h = _decode_source_hash()
    traffic = None
    if (name, seed) in TRAFFIC and TRAFFIC[(name, seed)][0] == h:
        traffic = TRAFFIC[(name, seed)][1]
    return {"bound": "hbm",
            "kernel": "paged_decode_step call per layer: gqa_decode_kernel (step mode, split pieces merged in the kernel)",
            "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)",
            "bytes_per_launch": r["layer_bytes"], "launch_us_mean": round(dec_avg_s * 1e6, 2),
            "timing": f"CUDA events around {steps} replays of a graph of the step's {r['layers']} "
                      "paged_decode_step calls (inter-kernel gaps included)",
            "decode_source": h}


def run_ours(args, ws, rank, local):
    import paged_kv_decode_rope_gb300 as pkv
    from paged_kv_decode_rope_gb300.build import build
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device")
    build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peak, peak_kind = _peaks()
    seeds = [args.seed + i for i in range(max(1, args.seeds))]
    sub_names = [n for n in SUB_WORKLOADS if n != args.workload] \
        if args.workload == DEFAULT_WORKLOAD and not args.layers and not args.no_sub else []

    # Device-timed steps: the workload at every seed, then the other named
    # workloads of the target, with the SM clocks sampled throughout.
    clocks = ClockSampler(local)
    clocks.start()
    t_wall = time.perf_counter()
    runs = _seed_sweep(pkv, args.workload, seeds, dev, args, ws, rank)
    sub_runs = {name: _seed_sweep(pkv, name, seeds, dev, args, ws, rank) for name in sub_names}
    wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    head = _median_run(runs)
    value, ms_step_max = head["value"], head["ms"]

    # The median seed's workload again, for the end-to-end figure and the CPU baseline.
    wl = workloads.make(args.workload, seed=head["seed"] + 1000 * rank, device=dev, layers=args.layers)
    pool = wl.pool
    bt = torch.from_numpy(wl.block_tables).to(dev)
    sl = torch.from_numpy(wl.seq_lens).to(dev)
    pos = torch.from_numpy(wl.positions).to(dev)
    step = pkv.DecodeStep(pool, num_kv_heads=wl.num_kv_heads, num_q_heads=wl.num_q_heads,
                          num_layers=wl.num_layers, block_tables=bt, seq_lens=sl, positions=pos,
                          rope_theta=wl.rope_theta, scale=wl.scale, pages_per_split=args.pages_per_split,
                          fused_q_rot=False)
    stream = torch.cuda.current_stream()
    total_bytes = _barrier_sum(float(wl.kv_bytes_per_step()), ws)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if head["flush"] else None

    # end to end: host buffers in pinned memory; per step copy q/k/v, tables,
    # lengths and positions in, run the step through the C ABI, copy outputs out.
    hq = wl.q.cpu().pin_memory()
    hk = wl.k.cpu().pin_memory()
    hv = wl.v.cpu().pin_memory()
    hbt = torch.from_numpy(wl.block_tables).pin_memory()
    hsl = torch.from_numpy(wl.seq_lens).pin_memory()
    hpos = torch.from_numpy(wl.positions).pin_memory()
    hout = torch.empty(step.out.shape, dtype=torch.float32).pin_memory()
    dq, dk, dv = torch.empty_like(wl.q), torch.empty_like(wl.k), torch.empty_like(wl.v)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hbt, hsl, hpos))
    d2h = hout.numel() * 4
    e2e_steps = max(3, min(args.steps, 20))

    host_in = {"q": hq, "k": hk, "v": hv, "block_tables": hbt, "seq_lens": hsl, "positions": hpos}
    dev_in = {"q": dq, "k": dk, "v": dv, "block_tables": bt, "seq_lens": sl, "positions": pos}
    copy_streams = (torch.cuda.Stream(dev), torch.cuda.Stream(dev))

    def e2e_step():
        step.run_from_host(host_in, dev_in, hout, copy_streams)

    # The whole end-to-end step (host copies in, every layer's call, result
    # copy out) is captured once as a CUDA graph, as a serving loop would.
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_e2e):
        e2e_step()
    for _ in range(2):
        g_e2e.replay()
    torch.cuda.synchronize()
    _barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        if flush is not None:
            flush.fill_(1.0)
        g_e2e.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = _barrier_max(e0.elapsed_time(e1) / e2e_steps, ws)
    e2e_value = total_bytes / (e2e_ms / 1e3) / 1e9

    def record(r, name):
        return {"value": round(r["value"], 2), "unit": "GB/s", "us_per_step": round(r["ms"] * 1e3, 2),
                "pct_of_hbm_peak": round(100 * r["value"] / ws / peak, 2),
                "pct_of_8tbs": round(100 * r["value"] / ws / 8000, 2), "seed": r["seed"],
                "kv_bytes_per_step": r["kv_bytes_per_step"], "seq_len_mean": r["seq_len_mean"],
                "roofline_frac": _roofline(r, name, r["seed"], peak, peak_kind, args.steps)["frac"]}

    def sweep(rs, name):
        return {"median_of_seeds": [r["seed"] for r in rs],
                "per_seed": [{"seed": r["seed"], "value": round(r["value"], 2),
                              "us_per_step": round(r["ms"] * 1e3, 2),
                              "seq_len_mean": r["seq_len_mean"]} for r in rs]}

    sub = {}
    for name, rs in sub_runs.items():
        m = _median_run(rs)
        sub[name] = {**record(m, name), **sweep(rs, name),
                     "roofline": _roofline(m, name, m["seed"], peak, peak_kind, args.steps),
                     "clocks": "the line's clocks (sampled across every device-timed step)"}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step_max, 4), "us_per_step": round(ms_step_max * 1e3, 2),
        "pct_of_hbm_peak": round(100 * value / ws / peak, 2), "pct_of_8tbs": round(100 * value / ws / 8000, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "storage": ("bf16 KV pages; new key rounded as fp64 rotation would round it; q.K and P.V on "
                    "tensor cores with bf16 hi+lo operand pairs for q and P (about 16 mantissa bits) "
                    "and fp32 accumulation; fp32 softmax"),
        "data": "synthetic (seeded; bf16 N(0,1) q/k/v and cache)",
        "config": {**_config(wl), "seed": head["seed"],
                   "headline": f"median over seeds {seeds[0]}..{seeds[-1]} of the per-seed GB/s; "
                               "us_per_step, roofline and config are the median seed's"},
        "seeds": sweep(runs, args.workload),
        "roofline": _roofline(head, args.workload, head["seed"], peak, peak_kind, args.steps),
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                "timing": "CUDA events around replays of a CUDA graph of DecodeStep.run_from_host: "
                          "pinned host -> device copies of block tables, lengths, positions and each "
                          "layer's q/k/v, the step through the C ABI, device -> pinned host copy of "
                          "each layer's output; copies on two copy streams, layer-pipelined"},
        "gpu_launches": head["launches"],
        "timing": "CUDA events around K replays of a CUDA graph of one whole step, per seed",
        "clocks": clk, "wall_s_timed": round(wall, 3),
    }
    if sub:
        line["workloads"] = sub
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, pool)
    if rank == 0:
        print(json.dumps(line), flush=True)
    step.close()
    return 0


def run_trace(args, ws, rank, local) -> int:
    """A continuous-batching trace (page scheduler, paged prefill of the admitted
    prompts, fused decode steps), Llama-3.2-1B shape, 16 layers, 2.5 GiB pool.
    Prints one JSON line of its own."""
    import paged_kv_decode_rope_gb300 as pkv  # noqa: F401  (loads the library)
    from paged_kv_decode_rope_gb300.build import build
    from paged_kv_decode_rope_gb300.trace import DecodeTrace
    build()
    torch.cuda.set_device(local)
    reqs = workloads.trace_requests(args.trace, seed=args.seed + 1000 * rank, prompt_range=(64, 1024),
                                    new_range=(32, 256), early_stop_frac=0.3)
    tr = DecodeTrace(reqs, num_pages=81920, num_layers=16, num_q_heads=32, num_kv_heads=8,
                     rope_theta=500000.0, seed=args.seed + 1000 * rank, max_batch=256,
                     device=torch.device("cuda", local), device_inputs=True, prefill_tokens=8192)
    st = tr.run()
    tr.close()
    ms = _barrier_max(st["device_ms"], ws)
    tokens = _barrier_sum(float(st["decode_tokens"]), ws)
    kv = _barrier_sum(float(st["kv_bytes"]), ws)
    if rank == 0:
        line = {"metric": "decode trace: decode tokens/s (device time of the decode steps)",
                "value": round(tokens / (ms / 1e3), 1), "unit": "tokens/s", "n_gpus": ws,
                "higher_is_better": True, "kv_gb_per_s": round(kv / (ms / 1e3) / 1e9, 1),
                "steps": st["steps"], "decode_tokens": st["decode_tokens"],
                "device_ms": round(st["device_ms"], 2), "wall_s": round(st["wall_s"], 2),
                "wall_tokens_per_s": round(st["decode_tokens"] / st["wall_s"], 1),
                "completed": st["completed"], "sched": st["sched"],
                "prefill": {"calls": st["prefill_calls"], "prompt_tokens": st["prompt_tokens"],
                            "device_ms": round(st["prefill_ms"], 2),
                            "tokens_per_s": round(st["prompt_tokens"] / (st["prefill_ms"] / 1e3), 1)},
                "config": {"requests": args.trace, "prompt": "U[64,1024]", "max_new": "U[32,256]",
                           "early_stop": 0.3, "layers": 16, "q_heads": 32, "kv_heads": 8,
                           "pool_pages": 81920, "batching": "continuous",
                           "prefill_call_tokens": 8192},
                "data": "synthetic (seeded)",
                "timing": "CUDA events around each step's RoPE table and per-layer fused decode "
                          "calls, summed (prefill: around each call's RoPE table and per-layer "
                          "paged_prefill calls); wall time includes host scheduling, input "
                          "draws and copies"}
        print(json.dumps(line), flush=True)
    return 0


def _prefill_traffic(nb: int, t: int) -> int | None:
    ent = PREFILL_TRAFFIC.get((nb, t))
    return ent[1] if ent and ent[0] == _source_hash("prefill.cu") else None


def run_prefill(args, ws, rank, local) -> int:
    """Chunked causal prefill of fresh prompts (Llama-3.2-1B shape, 16 layers):
    B sequences of T tokens each, one paged_prefill call per layer, captured as a
    CUDA graph. Prints one JSON line of its own."""
    import paged_kv_decode_rope_gb300 as pkv
    from paged_kv_decode_rope_gb300.build import build
    build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    nb, t = (int(x) for x in args.prefill.split(","))
    nl, hq, hkv, theta = 16, 32, 8, 500000.0
    gen = torch.Generator(device=dev)
    gen.manual_seed(args.seed + 1000 * rank)
    mb = -(-t // 16)
    num_pages = nl * nb * mb
    pool = torch.randn(num_pages * 2 * hkv * 16 * 64, generator=gen, device=dev).to(torch.bfloat16)
    kp = pkv.kv_pool_create(pool, hkv)
    perm = torch.randperm(num_pages, generator=gen, device=dev).to(torch.int32)
    bt = perm.view(nl, nb, mb)
    total = nb * t
    q = torch.randn(nl, total, hq, 64, generator=gen, device=dev).to(torch.bfloat16)
    k = torch.randn(nl, total, hkv, 64, generator=gen, device=dev).to(torch.bfloat16)
    v = torch.randn(nl, total, hkv, 64, generator=gen, device=dev).to(torch.bfloat16)
    cu = torch.arange(0, total + 1, t, dtype=torch.int32, device=dev)
    st = torch.zeros(nb, dtype=torch.int32, device=dev)
    q_rot = torch.empty(nl, total, hq, 64, device=dev)
    out = torch.empty(nl, total, hq, 64, device=dev)
    wsp = pkv.alloc_prefill_workspace(total, nb, mb, device=dev)
    rope = pkv.build_rope_table(theta, mb * 16, device=dev)  # once per model, like its weights

    def step():  # every layer's prefill of the prompts
        for layer in range(nl):
            pkv.paged_prefill(kp, q[layer], k[layer], v[layer], q_rot[layer], out[layer], bt[layer],
                              cu, st, rope, 0.125, wsp)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(ws)
    e0.record()
    for _ in range(args.steps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = _barrier_max(e0.elapsed_time(e1) / args.steps, ws)
    assert pkv.pkv_get_error(kp) == 0
    kp.close()
    tokens = _barrier_sum(float(total), ws)
    # causal attention flops: 2 products of 2*64 flops per (query head, key) pair
    pairs = nb * t * (t + 1) / 2 * hq * nl
    if rank == 0:
        line = {"metric": "prefill: prompt tokens/s (16 layers, all layers per pass)",
                "value": round(tokens / (ms / 1e3), 1), "unit": "tokens/s", "n_gpus": ws,
                "higher_is_better": True, "ms_per_pass": round(ms, 4), "steps": args.steps,
                "warmup": args.warmup,
                "attention_tflops": round(pairs * 4 * 64 / (ms / 1e3) / 1e12, 2),
                "roofline": prefill_roofline(pairs, ms, *_tensor_peak(sustained=True),
                                             traffic=_prefill_traffic(nb, t)),
                "config": {"sequences": nb, "prompt_tokens": t, "layers": nl, "q_heads": hq,
                           "kv_heads": hkv, "start": 0},
                "data": "synthetic (seeded)",
                "timing": "CUDA events around replays of a CUDA graph of 16 paged_prefill calls"}
        print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(workloads.WORKLOADS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--seeds", type=int, default=5,
                    help="time the workload at this many seeds (seed, seed+1, ...); the line's value is the median")
    ap.add_argument("--no-sub", action="store_true",
                    help="skip the sub-records of the other target workloads")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--pages-per-split", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=None,
                    help="use only this many layers with a fitted pool (smaller case for profiling)")
    ap.add_argument("--trace", type=int, default=0, metavar="N",
                    help="instead: run a continuous-batching decode trace of N requests")
    ap.add_argument("--prefill", default="", metavar="B,T",
                    help="instead: time the chunked causal prefill of B fresh T-token prompts")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            return run_reference(args, ws, rank)
        if args.trace:
            return run_trace(args, ws, rank, local)
        if args.prefill:
            return run_prefill(args, ws, rank, local)
        return run_ours(args, ws, rank, local)
    finally:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
