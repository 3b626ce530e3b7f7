#!/usr/bin/env python
"""Benchmark of the paged KV-cache hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
slot mapping -> KV-cache write of the step's new tokens -> paged attention
(decode: the split-KV kernel, which merges the pieces of cut sequences
itself; mixed batches: decode rows plus prefill chunks).  The default workload is the batch-256 GQA decode configuration
(32 q-heads / 8 kv-heads, head_dim 128, bf16, block size 16, context lengths
from a power law x^-1.2 on [16, 4096], 64 sequences sharing a 1024-token
prefix).

Metric: paged-decode KV GB/s = algorithmic bytes of the step (unique KV
bytes, q and out, the new K/V rows read and written, table entries) divided
by the step's device time; attention tokens/s is reported beside it.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs its own replica (no collective on the data
path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from pagedattention_kv_cache_reshape_gb300 import workloads as W  # noqa: E402

METRIC = "paged-decode KV GB/s (% of GB300 HBM peak) and attention tokens/s per step"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="gqa256_bf16", choices=list(W.FULL_CONFIGS) + list(W.EXTRA_CONFIGS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-graph", action="store_true", help="launch each step's kernels directly")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the oracle CPU sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration measurements of all five workloads")
    ap.add_argument("--next-rows", action="store_true",
                    help="measure the NEXT rows instead (block fork / swap / pack, encode-only "
                         "attention, host block allocator): one JSON line each")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_tflops():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return FALLBACK_BF16_TFLOPS


def workload_bytes(w: W.Workload):
    """Algorithmic bytes of one step, split by part."""
    eb = w.k_cache.element_size()
    ctx = w.context_lens.cpu().numpy().astype(np.int64)
    row = w.num_kv_heads * w.head_dim * eb                      # one token, all kv-heads, K or V
    logical_tokens = int(ctx.sum())
    shared = max(w.shared_prefix_seqs - 1, 0) * w.shared_prefix_blocks * w.block_size
    unique_tokens = logical_tokens - shared
    q_bytes = w.total_q * w.num_heads * w.head_dim * eb
    nb = int(sum(w.blocks_per_seq))
    meta = nb * 4 + w.num_seqs * 4 * 3 + w.total_q * 8 * 2     # table entries, lengths, slots w+r
    new_kv = w.total_q * row * 2 * 2                              # K,V rows read and written
    return dict(kv_unique=unique_tokens * row * 2, kv_logical=logical_tokens * row * 2,
                q=q_bytes, out=q_bytes, new_kv=new_kv, meta=meta,
                unique_tokens=unique_tokens, logical_tokens=logical_tokens)


def prefill_flops(w: W.Workload):
    ql = w.q_lens
    ctx = w.context_lens.cpu().numpy()
    f = 0
    for q, c in zip(ql, ctx):
        if q > 1:
            pos = np.arange(c - q, c) + 1                 # keys visible to each query row
            f += int(4 * w.num_heads * w.head_dim * pos.sum())
    return f


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed loop runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        sel = []
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            sel = []
        self.cmd = ["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                    "-lms", "100"]

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        if not getattr(self, "lines", None):
            return None
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() in ("active", "1", "yes"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ oracle (CPU) sample

def cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it (x86: model name; Arm: the
    implementer and part codes), with the machine type."""
    import platform
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip(), v.strip())
    except OSError:
        pass
    if "model name" in fields:
        return f"{fields['model name']} ({platform.machine()})"
    if "CPU part" in fields:
        return f"{platform.machine()} CPU implementer {fields.get('CPU implementer', '?')} part {fields['CPU part']}"
    return platform.machine() or "unknown"


def oracle_sample(w_cpu: W.Workload, budget_s: float, nthreads: int, repeat: bool = False):
    """Times the oracle, as it stands, on a prefix of the workload's sequences
    sized to about `budget_s`.  With `repeat`, a sample that is the whole
    workload and runs well under the budget is run again until about half the
    budget is spent, so that one short run's noise does not set the figure.
    Returns (bytes_per_s, seconds, description, sequences, sample)."""
    import oracle as O

    def sub(n):
        cu = w_cpu.cu_seqlens_q[:n + 1]
        rows = int(cu[-1])
        return W.Workload(
            name=w_cpu.name, dtype=w_cpu.dtype, num_heads=w_cpu.num_heads, num_kv_heads=w_cpu.num_kv_heads,
            head_dim=w_cpu.head_dim, block_size=w_cpu.block_size, num_blocks=w_cpu.num_blocks,
            max_blocks=w_cpu.max_blocks, block_tables=w_cpu.block_tables[:n].contiguous(),
            context_lens=w_cpu.context_lens[:n].contiguous(), seq_start=w_cpu.seq_start[:n].contiguous(),
            cu_seqlens_q=cu.contiguous(), q=w_cpu.q[:rows].contiguous(), key=w_cpu.key[:rows].contiguous(),
            value=w_cpu.value[:rows].contiguous(), k_cache=w_cpu.k_cache, v_cache=w_cpu.v_cache,
            scale=w_cpu.scale, shared_prefix_seqs=min(w_cpu.shared_prefix_seqs, n),
            shared_prefix_blocks=w_cpu.shared_prefix_blocks, blocks_per_seq=w_cpu.blocks_per_seq[:n])

    def run(ws):
        t0 = time.perf_counter()
        slots = O.slot_mapping(ws.block_tables, ws.seq_start, ws.cu_seqlens_q, ws.block_size, ws.num_blocks)
        O.reshape_and_cache(ws.key, ws.value, ws.k_cache, ws.v_cache, slots, ws.block_size)
        O.paged_attention(ws.q, ws.k_cache, ws.v_cache, ws.block_tables, ws.context_lens, ws.scale,
                          cu_seqlens_q=None if ws.decode_only else ws.cu_seqlens_q, nthreads=nthreads)
        return time.perf_counter() - t0

    n = 1
    t = run(sub(n))
    while n < w_cpu.num_seqs and t < budget_s / 4:
        n = min(w_cpu.num_seqs, max(n + 1, int(n * min(8.0, budget_s / max(t, 1e-3) / 2))))
        t = run(sub(n))
    ws = sub(n)
    reps = 1
    if repeat and t < budget_s / 4:
        reps = max(2, int(budget_s / 2 / max(t, 1e-3)))
        t = sum(run(ws) for _ in range(reps))
    b = workload_bytes(ws)
    total = (b["kv_unique"] + b["q"] + b["out"] + b["new_kv"] + b["meta"]) * reps
    desc = (f"first {n} of {w_cpu.num_seqs} sequences of {w_cpu.name} (seed-identical inputs)"
            + (f", run {reps} times" if reps > 1 else "")
            + f", slot mapping + cache write + attention, fp64 oracle, {nthreads} threads")
    return total / t, t, desc, n, ws


# ------------------------------------------------------------------ NEXT rows

def run_next_rows(args):
    """One JSON line per NEXT row, each against its roofline:
      f1 fork      pa_copy_blocks inside one device pool (HBM: read + write);
      f1 swap out  device pool -> pinned host pool, f1 swap in: back (the host
                   link; beside it the copy engine's rate for the same bytes);
      f4 pack      pool -> contiguous device buffer, f4 unpack: back (HBM);
      f3 encode    pa_varlen_encode, 8 chunks of 512 rows over 0-2048 cached
                   tokens, non-causal (tensor pipe);
      f2 allocator pa_allocate_slots for a 256-sequence decode step (host).
    Pools are shaped like the decode workloads' (16 tokens x 8 kv-heads x 128
    dims bf16: 32 KB a block a pool); block ids are seeded random permutations.
    Device timings: CUDA events on the launching stream, L2 flushed before
    each call, median of 20."""
    from pagedattention_kv_cache_reshape_gb300 import build, pa
    build.build()
    pa.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    peak, peak_kind = measured_peaks()
    tc_peak = measured_tflops()
    rng = np.random.default_rng(args.seed)
    gen = torch.Generator(device=dev)
    gen.manual_seed(args.seed)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    evict = torch.zeros(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    evict_sum = torch.empty((), dtype=torch.float32, device=dev)

    def timed(fn, reps=20, warm=3):
        ts = []
        for i in range(reps + warm):
            flush.zero_()
            torch.sum(evict, dim=0, out=evict_sum)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            if i >= warm:
                ts.append(a.elapsed_time(b) / 1e3)
        return float(np.median(ts))

    def emit(row, value, unit, roofline, config):
        print(json.dumps({"row": row, "value": round(value, 2), "unit": unit, "roofline": roofline,
                          "config": config, "data": "synthetic (seeded)"}), flush=True)

    def hbm_roof(nbytes, secs):
        ach = nbytes / secs / 1e9
        return {"bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                "frac": round(ach / peak, 4), "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                "bytes_per_call": int(nbytes), "ms": round(secs * 1e3, 4)}

    status = torch.zeros(1, dtype=torch.int32, device=dev)
    nblk, npairs = 8192, 2048
    shape = (nblk, 16, 8, 128)
    k = torch.randn(shape, generator=gen, device=dev).to(torch.bfloat16)
    v = torch.randn(shape, generator=gen, device=dev).to(torch.bfloat16)
    block_bytes = 16 * 8 * 128 * 2
    perm = rng.permutation(nblk).astype(np.int32)
    src, dst = perm[:npairs], perm[npairs:2 * npairs]           # distinct, and no destination is a source
    cfg = {"pool_blocks": nblk, "pairs": npairs, "block": "16 x 8 x 128 bf16 (32 KB a pool)"}

    # f1 fork inside one pool
    fork = torch.from_numpy(np.stack([src, dst], 1)).to(dev)
    t = timed(lambda: pa.copy_blocks(k, v, k, v, fork, dev_status=status))
    nbytes = npairs * 2 * block_bytes * 2
    emit("f1 fork (block copy inside the device pool)", nbytes / t / 1e9, "GB/s", hbm_roof(nbytes, t), cfg)

    # f4 pack to / unpack from a contiguous buffer
    buf_k = torch.empty((npairs,) + shape[1:], dtype=torch.bfloat16, device=dev)
    buf_v = torch.empty_like(buf_k)
    seq = np.arange(npairs, dtype=np.int32)
    pack = torch.from_numpy(np.stack([src, seq], 1)).to(dev)
    unpack = torch.from_numpy(np.stack([seq, dst], 1)).to(dev)
    t = timed(lambda: pa.copy_blocks(k, v, buf_k, buf_v, pack, dev_status=status))
    emit("f4 pack (pool blocks to a contiguous transfer buffer)", nbytes / t / 1e9, "GB/s", hbm_roof(nbytes, t), cfg)
    t = timed(lambda: pa.copy_blocks(buf_k, buf_v, k, v, unpack, dev_status=status))
    emit("f4 unpack (transfer buffer to pool blocks)", nbytes / t / 1e9, "GB/s", hbm_roof(nbytes, t), cfg)

    # f1 swap out / in through a pinned host pool, beside the copy engine on the same bytes
    host_k = torch.empty((npairs,) + shape[1:], dtype=torch.bfloat16).pin_memory()
    host_v = torch.empty_like(host_k).pin_memory()
    one_way = npairs * 2 * block_bytes
    t_out = timed(lambda: pa.copy_blocks(k, v, host_k, host_v, pack, dev_status=status))
    t_in = timed(lambda: pa.copy_blocks(host_k, host_v, k, v, unpack, dev_status=status))
    t_ce_out = timed(lambda: (host_k.copy_(buf_k, non_blocking=True), host_v.copy_(buf_v, non_blocking=True)))
    t_ce_in = timed(lambda: (buf_k.copy_(host_k, non_blocking=True), buf_v.copy_(host_v, non_blocking=True)))
    for row, tt, tce in (("f1 swap out (device pool to pinned host pool)", t_out, t_ce_out),
                         ("f1 swap in (pinned host pool to device pool)", t_in, t_ce_in)):
        ach, ce = one_way / tt / 1e9, one_way / tce / 1e9
        emit(row, ach, "GB/s", {"bound": "host link", "achieved": round(ach, 1), "peak": round(ce, 1),
                                "unit": "GB/s", "frac": round(ach / ce, 4),
                                "peak_source": "the copy engine moving the same bytes contiguously (measured here)",
                                "bytes_per_call": one_way, "ms": round(tt * 1e3, 4)}, cfg)
    torch.cuda.synchronize()
    if pa.get_device_status(status) != 0:
        raise RuntimeError("device status set by a block copy")

    # f3 encode-only attention on mixed-step-shaped chunks
    w = W.mixed(args.seed, pa.num_blocks_needed, num_decode=0, device=dev)
    q_lens = (w.cu_seqlens_q[1:] - w.cu_seqlens_q[:-1]).cpu().numpy()
    ctx = w.context_lens.cpu().numpy()
    flops = float(sum(4 * w.num_heads * w.head_dim * int(ql) * int(c) for ql, c in zip(q_lens, ctx)))
    out = torch.empty_like(w.q)
    ws = torch.empty(pa.varlen_prefill_workspace_size(w.num_seqs, w.total_q, w.num_heads, w.num_kv_heads,
                                                      w.head_dim, w.block_size, w.max_blocks),
                     dtype=torch.uint8, device=dev)
    t = timed(lambda: pa.varlen_prefill(w.q, w.cu_seqlens_q, w.k_cache, w.v_cache, w.block_tables,
                                        w.context_lens, w.scale, int(q_lens.max()), out=out, workspace=ws,
                                        causal=False))
    ach = flops / t / 1e12
    emit("f3 encode-only varlen attention", ach, "TFLOP/s",
         {"bound": "tensor", "achieved": round(ach, 1), "peak": tc_peak, "unit": "TFLOP/s",
          "frac": round(ach / tc_peak, 4), "peak_source": "measured (MEASURED_PEAKS.json bf16_tflops)",
          "flops_per_call": flops, "ms": round(t * 1e3, 4)},
         {"chunks": int(len(q_lens)), "rows": int(w.total_q), "context_tokens": int(ctx.sum()),
          "heads": f"{w.num_heads} q / {w.num_kv_heads} kv", "head_dim": w.head_dim})

    # f2 host allocator: one decode step of 256 sequences (one new token each)
    g = W.make("gqa256_bf16", args.seed, pa.num_blocks_needed, device="cpu")
    steps = 200
    lens = [int(c) for c in g.context_lens.tolist()]
    need = sum(pa.num_blocks_needed(c + steps, 16) for c in lens)
    m = pa.BlockManager(need + 256, 16, pa.num_blocks_needed(max(lens) + steps, 16))
    for s_, c in enumerate(lens):
        if m.allocate_slots(s_, c - 1) != pa.OK:
            raise RuntimeError("allocator: prompt allocation failed")
    bad = 0
    ids = np.arange(g.num_seqs, dtype=np.int64)
    ones = np.ones(g.num_seqs, dtype=np.int32)
    half = steps // 2
    t0 = time.perf_counter()
    for _ in range(half):                       # one pa_allocate_slots_batch call a step
        bad += m.allocate_slots_batch(ids, ones) != pa.OK
    dt_batch = (time.perf_counter() - t0) / half
    t0 = time.perf_counter()
    for _ in range(steps - half):               # one pa_allocate_slots call a sequence
        for s_ in range(g.num_seqs):
            bad += m.allocate_slots(s_, 1) != pa.OK
    dt_each = (time.perf_counter() - t0) / (steps - half)
    m.close()
    if bad:
        raise RuntimeError("allocator: a decode-step allocation failed")
    emit("f2 host allocator (allocate_slots, one token for each of 256 sequences)", dt_batch * 1e6,
         "us per step",
         {"bound": "host", "us_per_sequence": round(dt_batch * 1e6 / g.num_seqs, 4),
          "one_call_per_sequence_us_per_step": round(dt_each * 1e6, 2),
          "note": "value: one pa_allocate_slots_batch call a step through the Python binding; beside it, "
                  "one pa_allocate_slots call a sequence"},
         {"sequences": g.num_seqs, "steps": steps})


# ------------------------------------------------------------------ our path

def run_e2e(args, w, w_out, step, stream, dev, flush_l2, use_graph):
    """The step end to end through the C ABI, inputs from pinned host memory and
    the output back to pinned host memory, every step.

    Two measurements:
      serial    -- copy-in, step, copy-out of one step after another (one stream,
                   replayed as a CUDA graph), L2 flushed before each step;
      pipelined -- how a serving loop runs it: double-buffered device inputs and
                   outputs, the copy-in of step i+1 and the copy-out of step i-1
                   on their own streams, overlapping step i.  No flush between
                   steps: each step streams the whole KV working set (several
                   times the 129 MB L2), so one step leaves the next little to
                   reuse.  Timed from the first copy-in to the last copy-out.
    The pipelined figure is the one reported as `e2e.value`.
    """
    names = ("q", "key", "value", "block_tables", "context_lens", "seq_start", "cu_seqlens_q")
    offs, total, h2d = {}, 0, 0
    for k in names:
        t = getattr(w, k)
        nbytes = t.numel() * t.element_size()
        offs[k] = (total, nbytes)
        h2d += nbytes
        total = (total + nbytes + 255) // 256 * 256
    # the step's inputs packed in one pinned host buffer: one H2D copy per step
    host_stage = torch.empty(total, dtype=torch.uint8).pin_memory()
    for k in names:
        t = getattr(w, k)
        o, nbytes = offs[k]
        host_stage[o:o + nbytes].copy_(t.detach().cpu().contiguous().view(-1).view(torch.uint8))
    nbuf = 2
    dev_stage = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(nbuf)]
    devb = []
    for b in range(nbuf):
        d = {}
        for k in names:
            t = getattr(w, k)
            o, nbytes = offs[k]
            d[k] = dev_stage[b][o:o + nbytes].view(t.dtype).view(t.shape)
        devb.append(d)
    out_dev = [torch.empty_like(w.q) for _ in range(nbuf)]
    out_host = [torch.empty(w.q.shape, dtype=w.q.dtype, pin_memory=True) for _ in range(nbuf)]
    d2h = out_host[0].numel() * out_host[0].element_size()
    K2 = min(args.steps, 100)

    def call(b, s):
        d = devb[b]
        step(q=d["q"], key=d["key"], value=d["value"], bt=d["block_tables"], ctx=d["context_lens"],
             ss=d["seq_start"], cu=d["cu_seqlens_q"], o=out_dev[b], pa_stream=s)

    # ---- serial: one stream, a CUDA graph of copy-in, step, copy-out
    def serial_step(s):
        dev_stage[0].copy_(host_stage, non_blocking=True)
        call(0, s)
        out_host[0].copy_(out_dev[0], non_blocking=True)

    serial_graph = None
    if use_graph:
        ge = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            serial_step(side)
            side.synchronize()
            with torch.cuda.graph(ge, stream=side, capture_error_mode="thread_local"):
                serial_step(side)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        serial_graph = ge
    e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K2)]
    for i in range(K2 + 3):
        flush_l2()
        if i >= 3:
            e_ev[i - 3][0].record(stream)
        if serial_graph is not None:
            serial_graph.replay()
        else:
            with torch.cuda.stream(stream):
                serial_step(stream)
        if i >= 3:
            e_ev[i - 3][1].record(stream)
    torch.cuda.synchronize()
    serial_ms = float(np.mean([a.elapsed_time(b) for a, b in e_ev]))

    # ---- pipelined: copy-in / step / copy-out on three streams, two buffers
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    for s_ in (s_in, s_cmp, s_out):
        s_.wait_stream(stream)
    ev_in = [torch.cuda.Event() for _ in range(nbuf)]
    ev_cmp = [torch.cuda.Event() for _ in range(nbuf)]
    ev_out = [torch.cuda.Event() for _ in range(nbuf)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def pipelined(n, timed):
        for i in range(n):
            b = i % nbuf
            if timed and i == 0:
                t0.record(s_in)
            with torch.cuda.stream(s_in):
                if i >= nbuf:
                    s_in.wait_event(ev_cmp[b])      # step i-2 has read buffer b
                dev_stage[b].copy_(host_stage, non_blocking=True)
                ev_in[b].record(s_in)
            s_cmp.wait_event(ev_in[b])
            if i >= nbuf:
                s_cmp.wait_event(ev_out[b])         # step i-2's output has left buffer b
            call(b, s_cmp)
            ev_cmp[b].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_cmp[b])
                out_host[b].copy_(out_dev[b], non_blocking=True)
                ev_out[b].record(s_out)
        if timed:
            t1.record(s_out)
        torch.cuda.synchronize()

    pipelined(4, False)
    pipelined(K2, True)
    pipe_ms = t0.elapsed_time(t1) / K2
    # every step computes the same batch, and the kernels are deterministic: the
    # outputs that came back must equal the device-timed step's bit for bit
    ref = w_out.detach().cpu()
    for b in range(nbuf):
        if not torch.equal(out_host[b], ref):
            raise RuntimeError("pipelined end-to-end output differs from the device-timed step")
    return dict(ms=pipe_ms, h2d=h2d, d2h=d2h, serial_ms=serial_ms,
                launch="pipelined: copy-in of step i+1 and copy-out of step i-1 overlap step i "
                       "(three streams, double-buffered device inputs and outputs, direct calls); "
                       "no L2 flush between steps (each step streams the whole KV working set)",
                serial_launch="CUDA graph of copy-in, step, copy-out, one step after another, "
                              "L2 flushed before each step" if serial_graph is not None else
                              "direct calls: copy-in, step, copy-out, L2 flushed before each step")


def make_flush(dev):
    """Writes 2x L2 of unrelated data, then reads another 2x L2, so that the
    lines left in L2 are clean (no write-back of the flush lands in the next
    timed step)."""
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)   # 258 MB, 2x L2
    evict = torch.zeros(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    evict_sum = torch.empty((), dtype=torch.float32, device=dev)

    def flush_l2():
        flush.zero_()
        torch.sum(evict, dim=0, out=evict_sum)
    return flush_l2


def capture_graph(fn, dev, stream):
    """fn(stream) run once, then captured as a CUDA graph on a side stream."""
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        fn(side)
        side.synchronize()
        with torch.cuda.graph(g, stream=side, capture_error_mode="thread_local"):
            fn(side)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    return g


class StepRunner:
    """One workload resident on the device, its step through the library's
    one-call step entry points, and the timing of that step and of its main
    attention kernel (CUDA events on the launching stream, L2 flushed before
    each timed step)."""

    def __init__(self, pa, w: W.Workload, dev, warmup: int, use_graph: bool):
        self.pa, self.w, self.dev = pa, w, dev
        self.decode_only = w.decode_only
        self.max_q = int(w.q_lens.max())
        self.slots = torch.empty(w.total_q, dtype=torch.int64, device=dev)
        self.out = torch.empty_like(w.q)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        ws_bytes = (pa.decode_workspace_size(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim,
                                             w.block_size, w.max_blocks) if self.decode_only else
                    pa.varlen_prefill_workspace_size(w.num_seqs, w.total_q, w.num_heads, w.num_kv_heads,
                                                     w.head_dim, w.block_size, w.max_blocks))
        self.workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        self.stream = torch.cuda.current_stream(dev)
        # decode: plan (with the cache write), decode; mixed: plan (with the
        # cache write and the prefill plan), decode, prefill
        self.launches_per_step = 2 if self.decode_only else 3
        for _ in range(max(warmup, 3)):
            self.step()
        torch.cuda.synchronize()
        self.check_status("warm-up")
        self.graph = capture_graph(lambda s: self.step(pa_stream=s), dev, self.stream) if use_graph else None
        # the attention call alone, as a graph, for timing it on the device (a
        # mixed call chains its kernels, so events around eager launches would
        # also count host set-up between them)
        self.attn_graph = None
        if use_graph and not self.decode_only:
            self.attn_graph = capture_graph(self.attention, dev, self.stream)

    def step(self, q=None, key=None, value=None, bt=None, ctx=None, ss=None, cu=None, o=None,
             pa_stream=None):
        w, pa = self.w, self.pa
        q = w.q if q is None else q
        key = w.key if key is None else key
        value = w.value if value is None else value
        bt = w.block_tables if bt is None else bt
        ctx = w.context_lens if ctx is None else ctx
        ss = w.seq_start if ss is None else ss
        cu = w.cu_seqlens_q if cu is None else cu
        o = self.out if o is None else o
        pa_stream = self.stream if pa_stream is None else pa_stream
        if self.decode_only:
            # slot mapping + cache write + decode through the one-call step entry
            pa.decode_step(q, key, value, w.k_cache, w.v_cache, bt, ctx, ss, cu, w.scale, out=o,
                           slot_mapping=self.slots, workspace=self.workspace, dev_status=self.status,
                           stream=pa_stream)
            return
        # slot mapping + cache write + varlen attention through the one-call step entry
        pa.varlen_step(q, key, value, w.k_cache, w.v_cache, cu, bt, ctx, ss, w.scale, self.max_q, out=o,
                       slot_mapping=self.slots, workspace=self.workspace, dev_status=self.status,
                       stream=pa_stream)

    def attention(self, pa_stream):
        w = self.w
        self.pa.varlen_prefill(w.q, w.cu_seqlens_q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                               w.scale, self.max_q, out=self.out, workspace=self.workspace,
                               dev_status=self.status, stream=pa_stream)

    def check_status(self, when):
        st = self.pa.get_device_status(self.status)
        if st != 0:
            raise RuntimeError(f"device status {self.pa.status_string(st)} {when} ({self.w.name})")

    def time_steps(self, K: int, flush_l2):
        """Device time of K steps, one by one (ms each)."""
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for i in range(K):
            flush_l2()
            ev[i][0].record(self.stream)
            if self.graph is not None:
                self.graph.replay()
            else:
                self.step()
            ev[i][1].record(self.stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in ev]

    def time_kernel(self, n: int, flush_l2):
        """Device time of the main attention kernel (ms each): the events the
        library records around that launch on the launching stream (direct
        launches); a mixed batch's attention call is timed as a graph of it."""
        kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in kev:
            a.record(); b.record()
        torch.cuda.synchronize()
        for i in range(n):
            flush_l2()
            if self.attn_graph is not None:
                kev[i][0].record(self.stream)
                self.attn_graph.replay()
                kev[i][1].record(self.stream)
            else:
                self.pa.set_timing_events(*kev[i])
                self.step()
        self.pa.set_timing_events(None, None)
        torch.cuda.synchronize()
        self.check_status("in the timed region")
        return [a.elapsed_time(b) for a, b in kev]


def stats_us(ms):
    return {"median": round(1e3 * float(np.median(ms)), 3), "mean": round(1e3 * float(np.mean(ms)), 3)}


def measure_configs(args, pa, dev, flush_l2, n):
    """Each of the five workload configurations through the same step and
    timing as the headline: median and mean of n event-timed steps (L2 flushed
    before each), its main attention kernel likewise, and its roofline
    fraction.  For the mixed step also the prefill chunks alone, and the
    prefill kernel alone at 8 chunks of 512 tokens over 2048 cached ones."""
    peak, _ = measured_peaks()
    tc_peak = measured_tflops()
    out = {}
    # the five configurations, then the headline one at cache block sizes 8 and 32
    makers = [(name, (lambda n=name: W.make(n, args.seed, pa.num_blocks_needed, device=dev)))
              for name in W.FULL_CONFIGS]
    makers += [(f"gqa256_bf16_block{B}", (lambda B=B: W.gqa(args.seed, pa.num_blocks_needed, block_size=B,
                                                              device=dev))) for B in (8, 32)]
    for name, make in makers:
        w = make()
        r = StepRunner(pa, w, dev, 3, not args.no_graph)
        step_ms = r.time_steps(n, flush_l2)
        kern_ms = r.time_kernel(n, flush_l2)
        r.check_status("in a config's timed region")
        b = workload_bytes(w)
        step_bytes = b["kv_unique"] + b["q"] + b["out"] + b["new_kv"] + b["meta"]
        kern_bytes = b["kv_unique"] + b["q"] + b["out"]
        km = float(np.median(kern_ms))
        e = {"steps": n, "step_us": stats_us(step_ms), "kernel_us": stats_us(kern_ms),
             "step_gbs": round(step_bytes / (float(np.median(step_ms)) / 1e3) / 1e9, 1)}
        if w.decode_only:
            e["kernel"] = "split_decode_kernel" if w.dtype == torch.bfloat16 else "generic_attention_kernel"
            e["kernel_gbs"] = round(kern_bytes / (km / 1e3) / 1e9, 1)
            e["frac"] = round(kern_bytes / (km / 1e3) / 1e9 / peak, 4)
        else:
            flops = prefill_flops(w)
            e["kernel"] = "attention call: split_decode_kernel + prefill_kernel, concurrent"
            e["decode_rows_gbs"] = round(kern_bytes / (km / 1e3) / 1e9, 1)
            e["decode_rows_frac"] = round(kern_bytes / (km / 1e3) / 1e9 / peak, 4)
            e["prefill_tflops"] = round(flops / (km / 1e3) / 1e12, 1)
            e["prefill_frac_of_call"] = round(flops / (km / 1e3) / 1e12 / tc_peak, 4)
        del r
        if not w.decode_only:
            # the step's prefill chunks alone (same prefixes, no decode rows): the
            # call is a plan launch and the prefill kernel
            wp = W.mixed(args.seed, pa.num_blocks_needed, num_decode=0, device=dev)
            rp = StepRunner(pa, wp, dev, 3, not args.no_graph)
            pm = rp.time_kernel(n, flush_l2)
            pf = prefill_flops(wp)
            pmed = float(np.median(pm))
            e["prefill_alone"] = {"call_us": stats_us(pm), "flops": pf,
                                  "tflops": round(pf / (pmed / 1e3) / 1e12, 1),
                                  "frac": round(pf / (pmed / 1e3) / 1e12 / tc_peak, 4)}
            del rp, wp
        out[name] = e
        del w
        torch.cuda.empty_cache()
    # the prefill kernel on its own at the mixed step's chunk shape with the
    # longest cached prefix (8 chunks of 512 new tokens over 2048 cached
    # tokens): the call is a plan launch and the prefill kernel
    wp = W.prefill_chunks(args.seed, pa.num_blocks_needed, device=dev)
    rp = StepRunner(pa, wp, dev, 3, not args.no_graph)
    pm = rp.time_kernel(n, flush_l2)
    rp.check_status("in a config's timed region")
    pf = prefill_flops(wp)
    pmed = float(np.median(pm))
    out["prefill8x512_bf16"] = {"steps": n, "kernel": "plan + prefill_kernel", "call_us": stats_us(pm),
                                "flops": pf, "tflops": round(pf / (pmed / 1e3) / 1e12, 1),
                                "frac": round(pf / (pmed / 1e3) / 1e12 / tc_peak, 4)}
    del rp, wp
    torch.cuda.empty_cache()
    return out


def run_ours(args, world, rank, local):
    from pagedattention_kv_cache_reshape_gb300 import build, pa
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    pa.load()
    w = W.make(args.config, args.seed + rank, pa.num_blocks_needed, device=dev)
    flush_l2 = make_flush(dev)
    r = StepRunner(pa, w, dev, args.warmup, not args.no_graph)
    K = args.steps

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall0 = time.perf_counter()
        step_ms = r.time_steps(K, flush_l2)
        t_wall = time.perf_counter() - t_wall0
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    total_ms = float(sum(step_ms))
    kern_ms = r.time_kernel(min(K, 100), flush_l2)

    # end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, r.out, r.step, r.stream, dev, flush_l2, r.graph is not None)

    configs = None
    if world == 1 and not args.no_configs:
        configs = measure_configs(args, pa, dev, flush_l2, max(K, 50))

    return dict(w=w, total_ms=total_ms, step_ms=step_ms, kern_ms=kern_ms, clocks=clk.summary(),
                graph=r.graph is not None, launches=r.launches_per_step * K, e2e=e2e, wall=t_wall,
                configs=configs)


def main():
    args = parse_args()
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    if args.impl == "reference":
        return main_reference(args, world, rank)
    if args.next_rows:
        return run_next_rows(args)

    r = run_ours(args, world, rank, local)
    w = r["w"]
    b = workload_bytes(w)
    step_bytes = b["kv_unique"] + b["q"] + b["out"] + b["new_kv"] + b["meta"]
    total_s = r["total_ms"] / 1e3
    # whole job: units of all ranks over the slowest rank's time
    total_s, job_bytes = job_totals(total_s, float(step_bytes) * args.steps, world,
                                    torch.device("cuda", local))
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    K = args.steps
    gbs = job_bytes / total_s / 1e9
    ms_per_step = r["total_ms"] / K
    peak, peak_kind = measured_peaks()
    kern_ms = float(np.mean(r["kern_ms"]))
    kern_bytes = b["kv_unique"] + b["q"] + b["out"]
    achieved = kern_bytes / (kern_ms / 1e3) / 1e9
    traffic = read_profile_traffic(args.config)
    line = {
        "metric": METRIC,
        "value": round(gbs, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "ms_per_step_median": round(float(np.median(r["step_ms"])), 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.dtype == torch.bfloat16 else "f32",
        "data": "synthetic (seeded N(0,1) values, power-law lengths, shuffled block pool)",
        "config": {
            "workload": w.name, "num_seqs": w.num_seqs, "num_heads": w.num_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
            "num_blocks": w.num_blocks, "context_tokens": b["logical_tokens"],
            "unique_context_tokens": b["unique_tokens"], "query_tokens": w.total_q,
            "l2": "flushed before every timed step: 258 MB written, then 258 MB read (clean lines)",
            "launch": "CUDA graph of the step's kernels" if r["graph"] else "direct launches",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "tokens_per_s": round(world * w.total_q * K / total_s, 1),
        "context_tokens_per_s": round(world * b["logical_tokens"] * K / total_s, 1),
        "kv_gbs_logical": round(b["kv_logical"] * K * world / total_s / 1e9, 2),
        "pct_of_hbm_peak": round(100 * gbs / world / peak, 2),
        "pct_of_nominal_8tbs": round(100 * gbs / world / 8000.0, 2),
        "roofline": {
            "kernel": "split_decode_kernel",
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
            if peak_kind == "measured" else "fallback 6.8 TB/s",
            "traffic": traffic, "bytes_per_launch": kern_bytes, "avg_launch_ms": round(kern_ms, 5),
            "median_launch_ms": round(float(np.median(r["kern_ms"])), 5),
            "frac_of_nominal_8tbs": round(achieved / 8000.0, 4),
        },
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
    }
    if r["e2e"] is not None:
        e = r["e2e"]
        line["e2e"] = {"value": round(step_bytes / (e["ms"] / 1e3) / 1e9 * world, 2), "unit": "GB/s",
                       "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"],
                       "ms_per_step": round(e["ms"], 5), "launch": e["launch"],
                       "serial": {"value": round(step_bytes / (e["serial_ms"] / 1e3) / 1e9 * world, 2),
                                  "ms_per_step": round(e["serial_ms"], 5), "launch": e["serial_launch"]}}
    if not w.decode_only:
        # one varlen call: the decode rows (HBM) and the prefill chunks (tensor
        # pipe) run concurrently, so the call is timed as a whole and each part's
        # roofline time is set against it; the call's bound is the larger one
        flops = prefill_flops(w)
        tc_peak = measured_tflops()
        t_hbm = kern_bytes / (peak * 1e9)
        t_tc = flops / (tc_peak * 1e12)
        call_s = kern_ms / 1e3
        line["prefill_flops_per_step"] = flops
        line["roofline"].update({
            "kernel": "split_decode_kernel + prefill_kernel (one call, run concurrently)",
            "bound": "hbm" if t_hbm >= t_tc else "tensor",
            "call_bound_frac": round(max(t_hbm, t_tc) / call_s, 4),
            "tensor": {"achieved": round(flops / call_s / 1e12, 1), "peak": tc_peak, "unit": "TFLOP/s",
                       "frac": round(flops / call_s / 1e12 / tc_peak, 4),
                       "peak_source": "measured (MEASURED_PEAKS.json bf16_tflops)"},
        })
    if r["configs"] is not None:
        # all five workloads, each timed like the headline (median of >= 50
        # steps, L2 flushed before each); units: microseconds, GB/s, TFLOP/s
        line["configs"] = r["configs"]
    if world == 1 and not args.no_cpu_baseline:
        import oracle as O
        nthreads = os.cpu_count() or 1
        w_cpu = w.to("cpu")
        bps, secs, desc, n, _ = oracle_sample(w_cpu, args.cpu_seconds, nthreads, repeat=True)
        bps1, secs1, desc1, _, _ = oracle_sample(w_cpu, args.cpu_seconds / 4, 1)
        line["cpu_baseline"] = {"value": round(bps / 1e9, 4), "unit": "GB/s", "cores": nthreads,
                                "kind": "oracle", "sample": desc, "seconds": round(secs, 2),
                                "cpu_model": cpu_model(),
                                "single_thread": {"value": round(bps1 / 1e9, 4), "unit": "GB/s",
                                                  "sample": desc1, "seconds": round(secs1, 2)}}
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def job_totals(seconds: float, bytes_done: float, world: int, device):
    """(slowest rank's seconds, bytes of all ranks): the whole-job aggregate of a
    replicated run.  No collective touches the data path; this one all-reduce
    runs once, after the timed region."""
    if world <= 1:
        return seconds, bytes_done
    import torch.distributed as dist
    t = torch.tensor([seconds, bytes_done], dtype=torch.float64, device=device)
    tmax = t.clone()
    dist.all_reduce(tmax, op=dist.ReduceOp.MAX)
    tsum = t.clone()
    dist.all_reduce(tsum, op=dist.ReduceOp.SUM)
    return float(tmax[0]), float(tsum[1])


def read_profile_traffic(config):
    """DRAM bytes per launch of the main kernel from the committed ncu summary,
    if one exists for this workload and kernel build; else None."""
    path = os.path.join(ROOT, "profiles", f"split_decode_kernel_{config}.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("kernel_source_sha") != kernel_source_sha():
            return None
        return d.get("dram_bytes_per_launch")
    except Exception:
        return None


def kernel_source_sha():
    import hashlib
    h = hashlib.sha256()
    p = os.path.join(ROOT, "pagedattention_kv_cache_reshape_gb300", "csrc", "attn_decode.cu")
    with open(p, "rb") as f:
        h.update(f.read())
    return h.hexdigest()[:16]


def main_reference(args, world, rank):
    """The oracle as it stands on the host cores, on the same workload."""
    if rank != 0:
        return
    import oracle as O
    O.build()
    w = W.make(args.config, args.seed, O.num_blocks_needed, device="cpu")
    nthreads = os.cpu_count() or 1
    per_step = max(0.05, 150.0 / max(args.steps + args.warmup, 1))
    # size one step's sample once, then time K steps of it
    _, _, desc, n, ws = oracle_sample(w, per_step, nthreads)
    b = workload_bytes(ws)
    step_bytes = b["kv_unique"] + b["q"] + b["out"] + b["new_kv"] + b["meta"]

    def one():
        t0 = time.perf_counter()
        slots = O.slot_mapping(ws.block_tables, ws.seq_start, ws.cu_seqlens_q, ws.block_size, ws.num_blocks)
        O.reshape_and_cache(ws.key, ws.value, ws.k_cache, ws.v_cache, slots, ws.block_size)
        O.paged_attention(ws.q, ws.k_cache, ws.v_cache, ws.block_tables, ws.context_lens, ws.scale,
                          cu_seqlens_q=None if ws.decode_only else ws.cu_seqlens_q, nthreads=nthreads)
        return time.perf_counter() - t0

    for _ in range(args.warmup):
        one()
    times = [one() for _ in range(args.steps)]
    total = sum(times)
    gbs = step_bytes * args.steps / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) values, power-law lengths, shuffled block pool)",
        "config": {"workload": w.name, "sample_sequences": n, "num_seqs": w.num_seqs},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": nthreads, "kind": "oracle",
                         "sample": desc, "cpu_model": cpu_model()},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
