#!/usr/bin/env python
"""Benchmark: one decode step of the NVFP4-compressed MLA cache per model layer.

A step = quantize-on-append of every session's new token (nvfp4_mla_append)
followed by sparse absorbed-MLA decode over the compressed cache
(sparse_mla_decode), for one layer. Consecutive steps walk through `--layers`
independent layer caches (own pool, own queries, own top-k sets), so the
rows a step reads were last touched several layers ago: the selected rows
of the rotation (>= 4 x 47.6 MB) exceed the 129 MB L2.

Prints one JSON line (rank 0). `--impl reference` times the CPU oracle on
the host cores instead (a deliberately slow baseline, not a target).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-MLA decode: compressed-KV GB/s and µs/launch vs GB300 HBM roofline"
ROW_BYTES = {0: 352, 1: 576}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="agent",
                    choices=["tiny", "decode_batch", "agent", "multi_token", "append_dense"])
    ap.add_argument("--row-format", type=int, default=0, choices=[0, 1])
    ap.add_argument("--layers", type=int, default=0, help="layer caches rotated (0 = auto)")
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--event-every", type=int, default=8,
                    help="time the append and decode launches of every n-th timed step with "
                         "CUDA events (each event pair adds a gap to the stream)")
    ap.add_argument("--blhnc", action="store_true",
                    help="one pool whose blocks hold every layer's page back to back "
                         "(block stride = layers x page bytes) instead of one pool per layer")
    ap.add_argument("--staged", action="store_true",
                    help="fused decode vs the staged comparison path (selected rows to an FP8 "
                         "buffer, then the FP8 decode) on --config; one JSON line")
    ap.add_argument("--cpu-table", action="store_true",
                    help="CPU baseline over every config: the oracle timed single-threaded and "
                         "on all host threads on a bounded sample, scaled to the full config; "
                         "one JSON line per config and thread count (no GPU)")
    ap.add_argument("--sweep", action="store_true",
                    help="head sweep (16/32/64/128 heads on decode_batch) and the 15 query "
                         "tokens x 16 heads x top-2048 point; one JSON line per point")
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def describe(wl, row_format):
    return {
        "workload": f"{wl.name}: {wl.num_seqs} sequences, {wl.num_q} query tokens, "
                    f"{wl.num_heads} heads, top-k {wl.topk}, "
                    f"{'NVFP4 352-B' if row_format == 0 else 'FP8 576-B'} rows, 64-token pages",
        "num_q": wl.num_q, "num_heads": wl.num_heads, "topk": wl.topk,
        "valid_rows_per_step": wl.valid_slots(), "cached_tokens": wl.total_tokens,
        "row_format": "nvfp4_352" if row_format == 0 else "fp8_576",
    }


def algorithmic(wl, row_format):
    """Per decode launch: bytes a perfect kernel moves, tensor FLOPs, compressed-KV bytes."""
    rows = wl.valid_slots()
    kv = rows * ROW_BYTES[row_format]
    q = wl.num_q * wl.num_heads * 576 * 2
    out = wl.num_q * wl.num_heads * (512 * 2 + 4)
    idx = wl.num_q * wl.topk * 4
    flops = 2.0 * wl.num_heads * (576 + 512) * rows
    return {"kv_bytes": kv, "bytes": kv + q + out + idx, "flops": flops}


def max_over_ranks(ms: float, world: int, device=None) -> float:
    """The slowest rank's time (every rank gets it); `device` holds the
    reduction tensor (a CUDA device under nccl, None = CPU under gloo)."""
    if world <= 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(kv_bytes_per_step: int, steps: int, world: int, ms: float) -> float:
    """Compressed-KV GB/s of the whole job: every rank's steps over the slowest rank's time."""
    return kv_bytes_per_step * steps * world / (ms * 1e-3) / 1e9


# --------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        inside = [l for (t, l) in self.lines if self.t0 <= t <= self.t1 + 0.05]
        if not inside:
            inside = [l for (_, l) in self.lines]
        sm, mx, reasons = [], [], set()
        for l in inside:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------- our implementation
def run_ours(args, rank, world, local_rank):
    import torch

    import nvfp4_compressed_mla_gb300 as nm
    from nvfp4_compressed_mla_gb300 import _native
    from workloads import all_tokens, make_workload, redraw_indices

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    lib = _native.load()
    wl = make_workload(args.config, seed=(1000 + ["tiny", "decode_batch", "agent", "multi_token",
                                                  "append_dense"].index(args.config) + 1
                                          + 7919 * rank))
    fmt = args.row_format
    rb = ROW_BYTES[fmt]
    page_bytes = 64 * rb
    pool_bytes = wl.num_blocks * page_bytes
    alg = algorithmic(wl, fmt)
    layers = args.layers or max(2, min(16, math.ceil(4 * 129e6 / max(alg["kv_bytes"], 1)) + 1))
    free, _ = torch.cuda.mem_get_info(dev)
    layers = max(1, min(layers, int(0.6 * free // max(pool_bytes, 1))))
    # one pool per layer, or (BLHNC) one pool whose block b holds layer l's page at
    # byte l * page_bytes: layer l is the pool from that offset with the wider stride
    stride = layers * page_bytes if args.blhnc else page_bytes
    shared_pool = (torch.empty(wl.num_blocks * stride, dtype=torch.uint8, device=dev)
                   if args.blhnc else None)

    g = torch.Generator(device=dev)
    bt = torch.from_numpy(wl.block_table).to(dev)
    seq_lens = torch.from_numpy(wl.seq_lens).to(dev)
    q_seq = torch.from_numpy(wl.q_seq).to(dev)
    all_seq, all_pos = all_tokens(wl)
    all_seq_d = torch.from_numpy(all_seq).to(dev)
    all_pos_d = torch.from_numpy(all_pos).to(dev)

    def rand_bf16(n, d, outliers):
        x = torch.randn((n, d), generator=g, device=dev, dtype=torch.float32)
        if outliers:
            m = torch.rand((n, d), generator=g, device=dev) < wl.outlier_frac
            x = torch.where(m, x * wl.outlier_mult, x)
        return x.to(torch.bfloat16)

    # step inputs: new tokens appended by the step (one per query token, at its own position)
    if wl.prefix_len:
        app_seq = torch.from_numpy(np.repeat(np.arange(wl.num_seqs, dtype=np.int32),
                                             wl.seq_lens - wl.prefix_len)).to(dev)
        app_pos = torch.from_numpy(np.concatenate(
            [np.arange(wl.prefix_len, n, dtype=np.int32) for n in wl.seq_lens])).to(dev)
    else:
        app_seq = torch.from_numpy(wl.q_seq).to(dev)
        app_pos = torch.from_numpy(wl.q_pos).to(dev)
    n_app = int(app_seq.numel())

    L = []
    for li in range(layers):
        g.manual_seed(12345 + 1000 * rank + li)
        pool = (shared_pool[li * page_bytes:] if args.blhnc
                else torch.empty(pool_bytes, dtype=torch.uint8, device=dev))
        chunk = 1 << 20
        for s in range(0, all_seq.size, chunk):
            e = min(s + chunk, all_seq.size)
            nm.nvfp4_mla_append(rand_bf16(e - s, 512, True), rand_bf16(e - s, 64, False),
                                all_seq_d[s:e], all_pos_d[s:e], bt, 64, pool, wl.num_blocks,
                                stride, fmt)
        idx = wl.topk_idx if li == 0 else redraw_indices(wl, li)
        L.append(dict(
            pool=pool,
            ql=rand_bf16(wl.num_q * wl.num_heads, 512, False).view(wl.num_q, wl.num_heads, 512),
            qr=rand_bf16(wl.num_q * wl.num_heads, 64, False).view(wl.num_q, wl.num_heads, 64),
            idx=torch.from_numpy(np.ascontiguousarray(idx)).to(dev),
            new_lat=rand_bf16(n_app, 512, True), new_rope=rand_bf16(n_app, 64, False)))
    torch.cuda.synchronize()

    out = torch.empty((wl.num_q, wl.num_heads, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((wl.num_q, wl.num_heads), dtype=torch.float32, device=dev)
    splits = args.num_splits or lib.sparse_mla_decode_num_splits(wl.num_q, wl.num_heads, wl.topk)
    ws_bytes = nm.sparse_mla_decode_workspace_size(wl.num_q, wl.num_heads, wl.topk, splits)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    # pre-bound C-ABI argument tuples: the timed loop is two foreign calls per step
    app_args, dec_args = [], []
    for d in L:
        app_args.append((d["new_lat"].data_ptr(), d["new_rope"].data_ptr(), app_seq.data_ptr(),
                         app_pos.data_ptr(), n_app, bt.data_ptr(), wl.num_seqs,
                         wl.max_blocks_per_seq, 64, d["pool"].data_ptr(), wl.num_blocks, stride,
                         fmt, 1.0, 1.0, None, sh))
        dec_args.append((d["ql"].data_ptr(), d["qr"].data_ptr(), q_seq.data_ptr(),
                         d["idx"].data_ptr(), wl.num_q, wl.num_heads, wl.topk, bt.data_ptr(),
                         wl.num_seqs, wl.max_blocks_per_seq, seq_lens.data_ptr(), 64,
                         d["pool"].data_ptr(), wl.num_blocks, stride, fmt, wl.sm_scale, 1.0,
                         1.0, out.data_ptr(), 0, lse.data_ptr(), ws.data_ptr(), ws.numel(),
                         splits, None, sh))
    append_fn, decode_fn = lib.nvfp4_mla_append, lib.sparse_mla_decode

    def step(i):
        a = append_fn(*app_args[i % layers])
        b = decode_fn(*dec_args[i % layers])
        if a or b:
            raise RuntimeError(f"status append={a} decode={b}")

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    K = args.steps
    every = max(1, args.event_every)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(0, K, every)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    gpu_id = torch.cuda.get_device_properties(dev).uuid
    sampler = ClockSampler(f"GPU-{gpu_id}" if not str(gpu_id).startswith("GPU-") else str(gpu_id))
    if rank == 0:
        sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.mark("t0")
    t_start.record(stream)
    for i in range(K):
        if i % every:
            step(i)
            continue
        e = ev[i // every]
        e[0].record(stream)
        append_fn(*app_args[i % layers])
        e[1].record(stream)
        decode_fn(*dec_args[i % layers])
        e[2].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    sampler.mark("t1")
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if rank == 0 else None
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    # per-launch times: the mean over the timed steps that carry events, times K
    append_ms = sum(e[0].elapsed_time(e[1]) for e in ev) * K / len(ev)
    decode_ms = sum(e[1].elapsed_time(e[2]) for e in ev) * K / len(ev)

    res = dict(total_ms=total_ms, append_ms=append_ms, decode_ms=decode_ms, layers=layers,
               splits=splits, clocks=clocks, wl=wl, alg=alg, fmt=fmt,
               launches_per_step=2 + (1 if splits > 1 else 0))

    if not args.no_e2e:
        res["e2e"] = run_e2e(args, wl, L, nm, dev, bt, seq_lens, q_seq, app_seq, app_pos, stride,
                             fmt, splits, ws, world)
    return res


def run_e2e(args, wl, L, nm, dev, bt, seq_lens, q_seq, app_seq, app_pos, stride, fmt, splits,
            ws, world):
    """Same step through the C ABI with host buffers: inputs from pinned host memory each step.

    Every step copies its inputs (queries, top-k, new tokens; packed in one
    buffer) host -> device and its result (out and LSE; one buffer) device ->
    host. The copies run on their own streams, double-buffered, so step i + 1's
    inputs arrive and step i - 1's result leaves while step i computes; events
    order each buffer's reuse. The two library calls of a step take argument
    tuples bound once, as in the device-timed loop, so the host issues steps
    faster than the GPU runs them (`host_ms_per_step` is the issue time).
    """
    import torch

    from nvfp4_compressed_mla_gb300 import _native
    lib = _native.load()
    layers = len(L)
    keys = ("ql", "qr", "idx", "new_lat", "new_rope")
    offs, in_bytes = [], 0
    for k in keys:  # 256-byte aligned slices of one buffer
        offs.append(in_bytes)
        t = L[0][k]
        in_bytes += (t.numel() * t.element_size() + 255) // 256 * 256
    host = []
    for d in L:
        hb = torch.zeros(in_bytes, dtype=torch.uint8).pin_memory()
        for k, o in zip(keys, offs):
            src = d[k].contiguous().view(torch.uint8).reshape(-1).cpu()
            hb[o:o + src.numel()].copy_(src)
        host.append(hb)
    dbuf = [torch.empty(in_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    out_bytes = wl.num_q * wl.num_heads * 512 * 2
    lse_off = (out_bytes + 255) // 256 * 256
    res_bytes = lse_off + wl.num_q * wl.num_heads * 4
    dres = [torch.empty(res_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    hres = [torch.empty(res_bytes, dtype=torch.uint8).pin_memory() for _ in range(2)]
    comp = torch.cuda.current_stream(dev)
    sh = comp.cuda_stream
    n_app = int(app_seq.numel())
    app, dec = {}, {}
    for li in range(layers):
        for b in range(2):
            ptr = {k: dbuf[b].data_ptr() + o for k, o in zip(keys, offs)}
            pool = L[li]["pool"].data_ptr()
            app[li, b] = (ptr["new_lat"], ptr["new_rope"], app_seq.data_ptr(), app_pos.data_ptr(),
                          n_app, bt.data_ptr(), wl.num_seqs, wl.max_blocks_per_seq, 64, pool,
                          wl.num_blocks, stride, fmt, 1.0, 1.0, None, sh)
            dec[li, b] = (ptr["ql"], ptr["qr"], q_seq.data_ptr(), ptr["idx"], wl.num_q,
                          wl.num_heads, wl.topk, bt.data_ptr(), wl.num_seqs,
                          wl.max_blocks_per_seq, seq_lens.data_ptr(), 64, pool, wl.num_blocks,
                          stride, fmt, wl.sm_scale, 1.0, 1.0, dres[b].data_ptr(), 0,
                          dres[b].data_ptr() + lse_off, ws.data_ptr(), ws.numel(), splits, None,
                          sh)
    append_fn, decode_fn = lib.nvfp4_mla_append, lib.sparse_mla_decode
    cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready = [ev(), ev()]
    used = [ev(), ev()]       # step's inputs and outputs are no longer needed by the compute
    out_read = [ev(), ev()]   # step's result has reached the host
    for b in range(2):        # every event starts out recorded
        for e_ in (in_ready[b], used[b], out_read[b]):
            e_.record(comp)

    def step(i):
        b = i & 1
        li = i % layers
        cin.wait_event(used[b])               # inputs of step i into buffer b
        with torch.cuda.stream(cin):
            dbuf[b].copy_(host[li], non_blocking=True)
        in_ready[b].record(cin)
        comp.wait_event(in_ready[b])
        comp.wait_event(out_read[b])          # buffer b's previous result has been read
        a, c = append_fn(*app[li, b]), decode_fn(*dec[li, b])
        if a or c:
            raise RuntimeError(f"status append={a} decode={c}")
        used[b].record(comp)
        cout.wait_event(used[b])              # result of step i to the host
        with torch.cuda.stream(cout):
            hres[b].copy_(dres[b], non_blocking=True)
        out_read[b].record(cout)

    for i in range(5):
        step(i)
    torch.cuda.synchronize()
    K = args.e2e_steps
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    s.record(comp)
    t0 = time.perf_counter()
    for i in range(K):
        step(i)
    host_ms = (time.perf_counter() - t0) * 1e3
    comp.wait_event(out_read[0])
    comp.wait_event(out_read[1])
    e.record(comp)
    torch.cuda.synchronize()
    ms = max_over_ranks(s.elapsed_time(e), world, dev)
    kv = wl.valid_slots() * ROW_BYTES[fmt]
    return {"value": round(whole_job_gbs(kv, K, world, ms), 3), "unit": "GB/s",
            "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": res_bytes, "steps": K,
            "ms_per_step": round(ms / K, 5), "host_ms_per_step": round(host_ms / K, 5),
            "copies": "one host->device and one device->host copy per step on their own "
                      "streams, double-buffered"}


# ------------------------------------------------------------ CPU oracle
def oracle_sample(wl, fmt, budget_s, max_tokens=None, heads=None):
    """Time the oracle (append of the step's new tokens + decode) on a bounded sample.

    Returns (seconds, compressed-KV bytes fully processed, threads, description).
    """
    import oracle
    from workloads import make_append_batch, make_queries, make_rows, referenced_tokens
    rb = ROW_BYTES[fmt]
    stride = 64 * rb
    pool = np.zeros(wl.num_blocks * stride, np.uint8)  # untouched pages stay unallocated
    ntok = wl.num_q if max_tokens is None else min(max_tokens, wl.num_q)
    tok = np.arange(ntok)
    sub_idx = wl.topk_idx[tok]
    seq, pos = referenced_tokens(wl)
    keep = np.isin(seq.astype(np.int64) * (1 << 32) + pos,
                   (np.repeat(wl.q_seq[tok], wl.topk).astype(np.int64) * (1 << 32)
                    + sub_idx.reshape(-1))[sub_idx.reshape(-1) >= 0])
    lat, rope = make_rows(wl, int(keep.sum()))
    oracle.append(lat, rope, seq[keep], pos[keep], wl.block_table, 64, pool, wl.num_blocks,
                  stride, fmt)
    ql, qr = make_queries(wl)
    H = wl.num_heads if heads is None else heads
    aseq, apos, alat, arope = make_append_batch(wl)
    threads = oracle.max_threads()
    t0 = time.perf_counter()
    oracle.append(alat[:ntok], arope[:ntok], aseq[:ntok], apos[:ntok], wl.block_table, 64, pool,
                  wl.num_blocks, stride, fmt)
    done = 0
    for t in tok:
        oracle.sparse_mla_decode(ql[t:t + 1, :H], qr[t:t + 1, :H], wl.q_seq[t:t + 1],
                                 sub_idx[t:t + 1], wl.block_table, wl.seq_lens, 64, pool,
                                 wl.num_blocks, stride, fmt, wl.sm_scale, nthreads=threads)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    secs = time.perf_counter() - t0
    rows = int((sub_idx[:done] >= 0).sum())
    kv_full = rows * rb * H / wl.num_heads
    desc = (f"{done} query tokens x {H} of {wl.num_heads} heads x top-{wl.topk} rows of the "
            f"{wl.name} workload (plus the oracle append of {ntok} new tokens), fp64 C oracle")
    return secs, kv_full, threads, desc


def cpu_model():
    """The host CPU as /proc/cpuinfo names it (x86 model name, or Arm implementer/part)."""
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
        return fields["model name"]
    parts = [f"{k} {fields[k]}" for k in ("CPU implementer", "CPU part", "CPU variant") if k in fields]
    return ", ".join(parts) or "unknown"


def run_cpu_table(args):
    """The fp64 oracle per config, 1 thread and all threads, on bounded samples.

    A sample is whole query tokens (all heads) until about `budget` seconds
    have passed; the full-config time is the sample time scaled by the valid
    rows of all tokens over those of the sample. The append configuration
    also times the oracle append of its new tokens.
    """
    import oracle
    from workloads import CONFIG_NAMES, make_append_batch, make_queries, make_rows, make_workload
    from workloads import referenced_tokens
    nmax = oracle.max_threads()
    model = cpu_model()
    for name in CONFIG_NAMES:
        wl = make_workload(name)
        fmt = 0
        rb = ROW_BYTES[fmt]
        stride = 64 * rb
        pool = np.zeros(wl.num_blocks * stride, np.uint8)
        seq, pos = referenced_tokens(wl)
        lat, rope = make_rows(wl, int(seq.size))
        oracle.append(lat, rope, seq, pos, wl.block_table, 64, pool, wl.num_blocks, stride, fmt)
        ql, qr = make_queries(wl)
        rows_all = int((wl.topk_idx >= 0).sum())
        for threads in sorted({1, nmax}):
            budget = 6.0 if threads == 1 else 3.0
            t0 = time.perf_counter()
            done = rows = 0
            for t in range(wl.num_q):
                oracle.sparse_mla_decode(ql[t:t + 1], qr[t:t + 1], wl.q_seq[t:t + 1],
                                         wl.topk_idx[t:t + 1], wl.block_table, wl.seq_lens, 64,
                                         pool, wl.num_blocks, stride, fmt, wl.sm_scale,
                                         nthreads=threads)
                done += 1
                rows += int((wl.topk_idx[t] >= 0).sum())
                if time.perf_counter() - t0 > budget:
                    break
            secs = time.perf_counter() - t0
            full_s = secs * rows_all / max(rows, 1)
            line = {"cpu_table": name, "threads": threads, "cpu_model": model,
                    "host_threads": nmax, "decode_s_full_config": round(full_s, 4),
                    "decode_us_per_row_head": round(secs / max(rows, 1) / wl.num_heads * 1e6, 4),
                    "sample": f"{done} of {wl.num_q} query tokens, all {wl.num_heads} heads, "
                              f"{rows} valid rows, fp64 C oracle, NVFP4 rows",
                    "config": describe(wl, fmt)}
            if name == "append_dense" and threads == 1:  # the oracle append is single-threaded
                aseq, apos, alat, arope = make_append_batch(wl)
                apool = np.zeros(wl.num_blocks * stride, np.uint8)
                t1 = time.perf_counter()
                oracle.append(alat, arope, aseq, apos, wl.block_table, 64, apool, wl.num_blocks,
                              stride, fmt)
                line["append_s"] = round(time.perf_counter() - t1, 4)
                line["append_tokens"] = int(aseq.size)
            print(json.dumps(line), flush=True)


def run_reference(args):
    from workloads import make_workload
    wl = make_workload(args.config)
    fmt = args.row_format
    # calibrate one (token, head) so that warmup + steps fit in about two minutes
    secs, _, threads, _ = oracle_sample(wl, fmt, 1e9, max_tokens=1, heads=1)
    per_head = max(secs, 1e-6)
    budget = 120.0 / max(args.steps + args.warmup, 1)
    heads = int(max(1, min(wl.num_heads, budget / per_head)))
    import oracle
    from workloads import make_queries
    # one bounded sample per step: `heads` heads of one query token, rotating tokens
    rb = ROW_BYTES[fmt]
    stride = 64 * rb
    pool = np.zeros(wl.num_blocks * stride, np.uint8)
    from workloads import make_rows, referenced_tokens
    seq, pos = referenced_tokens(wl)
    lat, rope = make_rows(wl, int(seq.size))
    oracle.append(lat, rope, seq, pos, wl.block_table, 64, pool, wl.num_blocks, stride, fmt)
    ql, qr = make_queries(wl)

    def step(i):
        t = i % wl.num_q
        oracle.sparse_mla_decode(ql[t:t + 1, :heads], qr[t:t + 1, :heads], wl.q_seq[t:t + 1],
                                 wl.topk_idx[t:t + 1], wl.block_table, wl.seq_lens, 64, pool,
                                 wl.num_blocks, stride, fmt, wl.sm_scale, nthreads=threads)
        return int((wl.topk_idx[t] >= 0).sum())

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    rows = 0
    for i in range(args.steps):
        rows += step(i)
    secs = time.perf_counter() - t0
    kv = rows * rb * heads / wl.num_heads
    value = kv / secs / 1e9
    sample = (f"per step: 1 query token x {heads} of {wl.num_heads} heads x top-{wl.topk} rows "
              f"of the {wl.name} workload; GB/s scaled by heads computed / {wl.num_heads}")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / max(args.steps, 1) * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": describe(wl, fmt),
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ main
def traffic_from_profiles(fmt, config):
    """DRAM bytes per decode launch from the committed ncu summary, if the kernel is unchanged."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    src = os.path.join(ROOT, "nvfp4_compressed_mla_gb300", "csrc", d.get("source", "decode.cu"))
    if not os.path.exists(src):
        return None
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    key = f"{config}/{fmt}"
    if d.get("source_sha256_16") != h or key not in d.get("per_launch_bytes", {}):
        return None
    return d["per_launch_bytes"][key]


def run_staged(args):
    """Fused NVFP4 decode vs the staged comparison path on the same inputs.

    The staged path is nvfp4_mla_stage_fp8 (selected rows re-encoded as FP8
    rows in a device buffer) followed by sparse_mla_decode over that buffer
    with FP8 rows. Both are timed as CUDA graphs of 100 steps over rotated
    layer caches (median of 5 replays after 20 warm-up steps).
    """
    import torch

    import nvfp4_compressed_mla_gb300 as nm
    from nvfp4_compressed_mla_gb300 import _native
    from workloads import all_tokens, make_workload, redraw_indices

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    lib = _native.load()
    peaks = load_peaks()
    wl = make_workload(args.config)
    stride = 64 * ROW_BYTES[0]
    alg = algorithmic(wl, 0)
    pool_bytes = wl.num_blocks * stride
    layers = args.layers or max(2, min(16, math.ceil(4 * 129e6 / max(alg["kv_bytes"], 1)) + 1))
    free, _ = torch.cuda.mem_get_info(dev)
    layers = max(1, min(layers, int(0.5 * free // max(pool_bytes, 1))))
    g = torch.Generator(device=dev)
    bt = torch.from_numpy(wl.block_table).to(dev)
    seq_lens = torch.from_numpy(wl.seq_lens).to(dev)
    q_seq = torch.from_numpy(wl.q_seq).to(dev)
    all_seq, all_pos = all_tokens(wl)
    sd = torch.from_numpy(all_seq).to(dev)
    pd = torch.from_numpy(all_pos).to(dev)
    L = []
    for li in range(layers):
        g.manual_seed(4242 + li)
        pool = torch.empty(pool_bytes, dtype=torch.uint8, device=dev)
        for s0 in range(0, all_seq.size, 1 << 20):
            e0 = min(s0 + (1 << 20), all_seq.size)
            lat = torch.randn((e0 - s0, 512), generator=g, device=dev).to(torch.bfloat16)
            rope = torch.randn((e0 - s0, 64), generator=g, device=dev).to(torch.bfloat16)
            nm.nvfp4_mla_append(lat, rope, sd[s0:e0], pd[s0:e0], bt, 64, pool, wl.num_blocks,
                                stride, 0)
        idx = wl.topk_idx if li == 0 else redraw_indices(wl, li)
        L.append(dict(pool=pool,
                      ql=torch.randn((wl.num_q, wl.num_heads, 512), generator=g,
                                     device=dev).to(torch.bfloat16),
                      qr=torch.randn((wl.num_q, wl.num_heads, 64), generator=g,
                                     device=dev).to(torch.bfloat16),
                      idx=torch.from_numpy(np.ascontiguousarray(idx)).to(dev)))
    H, topk = wl.num_heads, wl.topk
    out = torch.empty((wl.num_q, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((wl.num_q, H), dtype=torch.float32, device=dev)
    splits = lib.sparse_mla_decode_num_splits(wl.num_q, H, topk)
    ws = torch.empty(max(nm.sparse_mla_decode_workspace_size(wl.num_q, H, topk, splits), 16),
                     dtype=torch.uint8, device=dev)
    R = nm.nvfp4_mla_staged_rows_per_q(topk, 64)
    staged = torch.empty(wl.num_q * R * 576, dtype=torch.uint8, device=dev)
    sidx = torch.empty((wl.num_q, topk), dtype=torch.int32, device=dev)
    tb = nm.staged_fp8_tables(wl.num_q, topk, 64, dev)
    cap = torch.cuda.Stream(dev)
    sh = cap.cuda_stream

    def fused(li):
        d = L[li]
        return lib.sparse_mla_decode(
            d["ql"].data_ptr(), d["qr"].data_ptr(), q_seq.data_ptr(), d["idx"].data_ptr(),
            wl.num_q, H, topk, bt.data_ptr(), wl.num_seqs, wl.max_blocks_per_seq,
            seq_lens.data_ptr(), 64, d["pool"].data_ptr(), wl.num_blocks, stride, 0, wl.sm_scale,
            1.0, 1.0, out.data_ptr(), 0, lse.data_ptr(), ws.data_ptr(), ws.numel(), splits,
            None, sh)

    def stage(li):
        d = L[li]
        return lib.nvfp4_mla_stage_fp8(
            q_seq.data_ptr(), d["idx"].data_ptr(), wl.num_q, topk, bt.data_ptr(), wl.num_seqs,
            wl.max_blocks_per_seq, seq_lens.data_ptr(), 64, d["pool"].data_ptr(), wl.num_blocks,
            stride, 1.0, staged.data_ptr(), sidx.data_ptr(), None, sh)

    def staged_decode(li):
        d = L[li]
        return lib.sparse_mla_decode(
            d["ql"].data_ptr(), d["qr"].data_ptr(), tb["q_seq"].data_ptr(), sidx.data_ptr(),
            wl.num_q, H, topk, tb["block_table"].data_ptr(), wl.num_q, R // 64,
            tb["seq_lens"].data_ptr(), 64, staged.data_ptr(), tb["num_blocks"],
            tb["block_stride_bytes"], 1, wl.sm_scale, 1.0, 1.0, out.data_ptr(), 0,
            lse.data_ptr(), ws.data_ptr(), ws.numel(), splits, None, sh)

    def timed(fns):
        with torch.cuda.stream(cap):
            for i in range(20):
                for f in fns:
                    if f(i % layers):
                        raise RuntimeError("launch failed")
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            for i in range(100):
                for f in fns:
                    if f(i % layers):
                        raise RuntimeError("launch failed during capture")
        graph.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(cap)
            with torch.cuda.stream(cap):
                graph.replay()
            e1.record(cap)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return float(np.median(ts)) * 1e3 / 100

    t_fused = timed([fused])
    t_stage = timed([stage])
    t_staged = timed([stage, staged_decode])
    rows = wl.valid_slots()
    cfg = describe(wl, 0)
    cfg.update({"layers_rotated": layers, "num_splits": splits,
                "timing": "cuda graphs of 100 steps, median of 5 replays"})
    print(json.dumps({
        "comparison": "fused NVFP4 decode vs staged (selected rows -> FP8 buffer -> FP8 decode)",
        "fused_us": round(t_fused, 3),
        "staged_us": round(t_staged, 3),
        "stage_kernel_us": round(t_stage, 3),
        "staged_over_fused": round(t_staged / t_fused, 3),
        "stage_kernel_hbm_gbs": round(rows * (352 + 576) / (t_stage * 1e-6) / 1e9, 1),
        "stage_kernel_hbm_frac": round(rows * (352 + 576) / (t_stage * 1e-6) / 1e9
                                       / peaks["hbm_gbs"], 4),
        "config": cfg}), flush=True)


def run_sweep(args):
    """Decode µs/launch over a head sweep and at 15 query tokens x 16 heads x top-2048.

    Each point is timed as a CUDA graph of 100 decode launches that walk
    through enough layer caches (own pool rows, queries, top-k) that the
    rotation's selected rows exceed 4 x the 129 MB L2; the graph is replayed
    after 20 warm-up launches and the median of 5 replays is reported. If the
    capture fails, the same launches are timed back to back on the stream
    and the line says so. One JSON line per point.
    """
    import torch

    import nvfp4_compressed_mla_gb300 as nm
    from nvfp4_compressed_mla_gb300 import _native
    from workloads import all_tokens, make_workload, redraw_indices

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    lib = _native.load()
    peaks = load_peaks()
    fmt = args.row_format
    stride = 64 * ROW_BYTES[fmt]
    points = [("decode_batch", {"num_heads": h}) for h in (16, 32, 64, 128)]
    points.append(("multi_token", {"num_seqs": 1, "q_per_seq": 15, "num_heads": 16}))
    g = torch.Generator(device=dev)
    pools = {}
    n_launch, n_warm, n_rep = 100, 20, 5
    for name, kw in points:
        wl = make_workload(name, **kw)
        alg = algorithmic(wl, fmt)
        pool_bytes = wl.num_blocks * stride
        layers = max(2, min(64, math.ceil(4 * 129e6 / max(alg["kv_bytes"], 1)) + 1))
        key = (name, kw.get("num_seqs"))
        have = pools.get(key, [])
        free, _ = torch.cuda.mem_get_info(dev)
        layers = max(1, min(layers, len(have) + int(0.5 * free // max(pool_bytes, 1))))
        if len(have) < layers:  # pools do not depend on the head count: fill once, reuse
            all_seq, all_pos = all_tokens(wl)
            sd = torch.from_numpy(all_seq).to(dev)
            pd = torch.from_numpy(all_pos).to(dev)
            bt0 = torch.from_numpy(wl.block_table).to(dev)
            for li in range(len(have), layers):
                g.manual_seed(777 + li)
                pool = torch.empty(pool_bytes, dtype=torch.uint8, device=dev)
                for s0 in range(0, all_seq.size, 1 << 20):
                    e0 = min(s0 + (1 << 20), all_seq.size)
                    lat = torch.randn((e0 - s0, 512), generator=g, device=dev).to(torch.bfloat16)
                    rope = torch.randn((e0 - s0, 64), generator=g, device=dev).to(torch.bfloat16)
                    nm.nvfp4_mla_append(lat, rope, sd[s0:e0], pd[s0:e0], bt0, 64, pool,
                                        wl.num_blocks, stride, fmt)
                have.append(pool)
            pools[key] = have
        bt = torch.from_numpy(wl.block_table).to(dev)
        seq_lens = torch.from_numpy(wl.seq_lens).to(dev)
        q_seq = torch.from_numpy(wl.q_seq).to(dev)
        H = wl.num_heads
        per = []
        for li in range(layers):
            idx = wl.topk_idx if li == 0 else redraw_indices(wl, li)
            per.append(dict(
                ql=torch.randn((wl.num_q, H, 512), generator=g, device=dev).to(torch.bfloat16),
                qr=torch.randn((wl.num_q, H, 64), generator=g, device=dev).to(torch.bfloat16),
                idx=torch.from_numpy(np.ascontiguousarray(idx)).to(dev)))
        out = torch.empty((wl.num_q, H, 512), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((wl.num_q, H), dtype=torch.float32, device=dev)
        splits = lib.sparse_mla_decode_num_splits(wl.num_q, H, wl.topk)
        ws_bytes = nm.sparse_mla_decode_workspace_size(wl.num_q, H, wl.topk, splits)
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
        cap = torch.cuda.Stream(dev)

        def dec_args(li, sh):
            d = per[li]
            return (d["ql"].data_ptr(), d["qr"].data_ptr(), q_seq.data_ptr(), d["idx"].data_ptr(),
                    wl.num_q, H, wl.topk, bt.data_ptr(), wl.num_seqs, wl.max_blocks_per_seq,
                    seq_lens.data_ptr(), 64, have[li].data_ptr(), wl.num_blocks, stride, fmt,
                    wl.sm_scale, 1.0, 1.0, out.data_ptr(), 0, lse.data_ptr(), ws.data_ptr(),
                    ws.numel(), splits, None, sh)

        args_cap = [dec_args(i % layers, cap.cuda_stream) for i in range(n_launch)]
        with torch.cuda.stream(cap):
            for i in range(n_warm):
                if lib.sparse_mla_decode(*args_cap[i % n_launch]):
                    raise RuntimeError("decode failed")
        torch.cuda.synchronize()
        timing = "cuda graph of 100 launches, median of 5 replays"
        times = []
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=cap):
                for a in args_cap:
                    if lib.sparse_mla_decode(*a):
                        raise RuntimeError("a decode launch failed during capture")
            graph.replay()
            torch.cuda.synchronize()
            for _ in range(n_rep):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(cap)
                with torch.cuda.stream(cap):
                    graph.replay()
                e1.record(cap)
                torch.cuda.synchronize()
                times.append(e0.elapsed_time(e1))
        except RuntimeError as exc:  # capture refused: time the same launches eagerly
            torch.cuda.synchronize()
            timing = f"eager launches (graph capture failed: {str(exc).splitlines()[0][:80]})"
            times = []
            for _ in range(n_rep):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(cap)
                for a in args_cap:
                    lib.sparse_mla_decode(*a)
                e1.record(cap)
                torch.cuda.synchronize()
                times.append(e0.elapsed_time(e1))
        us = float(np.median(times)) * 1e3 / n_launch
        t = us * 1e-6
        cfg = describe(wl, fmt)
        cfg.update({"layers_rotated": layers, "num_splits": splits, "timing": timing})
        print(json.dumps({
            "sweep_point": f"{wl.num_q} q x {H} heads x top-{wl.topk}",
            "us_per_launch": round(us, 3),
            "kv_gbs": round(alg["kv_bytes"] / t / 1e9, 1),
            "hbm_frac": round(alg["bytes"] / t / 1e9 / peaks["hbm_gbs"], 4),
            "tensor_frac": round(alg["flops"] / t / 1e12 / peaks["bf16_tflops"], 4),
            "config": cfg}), flush=True)
        del per, out, lse, ws
        torch.cuda.empty_cache()


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return
    if args.cpu_table:
        if rank == 0:
            run_cpu_table(args)
        return
    if args.sweep:
        if rank == 0:
            run_sweep(args)
        return
    if args.staged:
        if rank == 0:
            run_staged(args)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, rank, world, local_rank)
    if rank != 0:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()
        return
    peaks = load_peaks()
    wl, alg, fmt = res["wl"], res["alg"], res["fmt"]
    K = args.steps
    ms_step = res["total_ms"] / K
    value = whole_job_gbs(alg["kv_bytes"], K, world, res["total_ms"])
    dec_s = res["decode_ms"] * 1e-3 / K
    achieved_tf = alg["flops"] / dec_s / 1e12
    achieved_gbs = alg["bytes"] / dec_s / 1e9
    bound = "tensor" if wl.num_heads * 1088 * 2 / ROW_BYTES[fmt] > \
        peaks["bf16_tflops"] * 1e3 / peaks["hbm_gbs"] else "hbm"
    if bound == "tensor":
        roof = {"bound": "tensor", "achieved": round(achieved_tf, 2), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(achieved_tf / peaks["bf16_tflops"], 4)}
    else:
        roof = {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved_gbs / peaks["hbm_gbs"], 4)}
    roof["traffic"] = traffic_from_profiles(fmt, wl.name)
    roof["peak_source"] = (f"{peaks['source']} (MEASURED_PEAKS.json burst; fp16 MMA = bf16 rate)"
                           if peaks["source"] == "measured" else "fallback")
    roof["kernel"] = "sparse_mla_decode"
    roof["hbm_frac"] = round(achieved_gbs / peaks["hbm_gbs"], 4)
    roof["tensor_frac"] = round(achieved_tf / peaks["bf16_tflops"], 4)
    cfg = describe(wl, fmt)
    cfg.update({"layers_rotated": res["layers"], "num_splits": res["splits"],
                "l2": f"inputs larger than L2: {res['layers']} layer caches rotated "
                      f"({res['layers'] - 1} x {alg['kv_bytes'] / 1e6:.1f} MB of other selected "
                      f"rows between reuses)",
                "parallelism": f"replicas x{world}",
                "cache_layout": ("BLHNC: one pool, each block holds every layer's 64-row page "
                                 "back to back" if args.blhnc else "one pool per layer")})
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": cfg,
        "us_per_launch": round(res["decode_ms"] * 1e3 / K, 3),
        "append_us_per_launch": round(res["append_ms"] * 1e3 / K, 3),
        "roofline": roof,
        "gpu_launches": res["launches_per_step"] * K,
        "clocks": res["clocks"],
    }
    if "e2e" in res:
        line["e2e"] = res["e2e"]
    if world == 1 and not args.no_cpu_baseline:
        secs, kv_full, threads, desc = oracle_sample(wl, fmt, budget_s=15.0)
        line["cpu_baseline"] = {"value": round(kv_full / secs / 1e9, 6), "unit": "GB/s",
                                "cores": threads, "kind": "oracle", "sample": desc}
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
