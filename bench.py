#!/usr/bin/env python3
"""Benchmark: split-KV decode attention on GB300 (one JSON line on stdout).

Default workload: MHA long-KV decode -- batch 1, 32 query heads = 32 kv heads,
head_dim 128, kv_len 65536, contiguous [S, H, D] bf16 K/V, scale 1/sqrt(128)
(1 GiB of K+V, larger than the 129 MB L2, so no flush is needed between
steps).  A step is one fd_decode call: the split kernel plus the LSE merge.
On one GPU the line also carries `workloads`: all five benchmark workloads
timed under the same protocol (CUDA-graph replay of back-to-back calls, the
split kernel timed by events the graph records).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1..5] [--impl ours|reference]
                  [--workloads 1,2,3,4,5|none]

Under torchrun each rank runs its own replica of the workload (the path
shards by request/head with no exchange), the timed region is bracketed by a
barrier and cudaDeviceSynchronize on every rank, and rank 0 prints the
whole-job throughput using the slowest rank's time.

`--impl reference` times the CPU oracle (the pages' method as plain fp64 C)
on the host cores instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import fd_synth as syn  # noqa: E402

METRIC = "decode-attn µs/call and achieved HBM TB/s (fraction of GB300 peak) on 1 GPU"
KERNEL_SOURCES = ["decode_attention_decoding_gb300/csrc/fd_kernels.cuh",
                  "decode_attention_decoding_gb300/csrc/fd_device.cuh",
                  "decode_attention_decoding_gb300/csrc/fd_sched.h"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "split_kernel_traffic.json")
TILE = 64
MAX_CTAS = 1024


# ---------------------------------------------------------------------------
# Algorithmic byte counts: K+V of the valid tokens once, q, O, LSE, and the
# workspace partials written once and read once
# ---------------------------------------------------------------------------

SEG_COST = 2   # the split schedule's cost of a segment start, in tiles (the library's kSegCostTiles)


def partial_count(lens, hkv, P, w=SEG_COST):
    """Number of (CTA, segment) partials the split writes: a host mirror of the
    library's schedule (contiguous runs of equal cost, a tile costing 1 and a
    segment start w more)."""
    nt = [(int(L) + TILE - 1) // TILE for L in lens]
    T = hkv * sum(nt)
    if T == 0:
        return 0
    C = T + w * hkv * sum(1 for k in nt if k)
    P = min(P, C)   # CTAs that take tiles
    n, first, starts = 0, 0, 0
    for k in nt:
        for _h in range(hkv):
            if k:
                starts += 1
                pos0 = first + w * starts
                c0, c1 = pos0 * P // C, (pos0 + k - 1) * P // C
                if c1 > c0:
                    n += c1 - c0 + 1
                first += k
    return n


def byte_counts(w, P):
    B, hq, d, ql = w.batch, w.num_q_heads, w.head_dim, w.q_len
    hkv, G = w.num_kv_heads, w.num_q_heads // w.num_kv_heads
    kv = w.kv_bytes()
    q = B * ql * hq * d * 2
    out = B * ql * hq * d * 4 + B * ql * hq * 4
    parts = partial_count(w.seq_lens, hkv, P)
    ws = parts * G * ql * (d + 1) * 4
    table = (sum((int(L) + w.page_size - 1) // w.page_size for L in w.seq_lens) * 4) if w.paged else 0
    return dict(kv=kv, q=q, out=out, ws_partials=parts, ws_once=ws, table=table, lens=B * 4,
                call=kv + q + out + 2 * ws,
                split=kv + q + ws + out)   # split reads K,V,q; writes partials or final O/LSE


def consumers_label(flags, w) -> str:
    """Which consumers the library's default choice runs for this workload."""
    G = w.num_q_heads // w.num_kv_heads * w.q_len   # query columns of a kv head
    fp8 = w.kv_dtype is not None
    row = w.head_dim * (1 if fp8 else 2)
    mma = "mma.sync fp16 on FP8 codes" if fp8 else "mma.sync bf16, P as two bf16 parts"
    if flags & 0x2:   # FD_FLAG_CUDA_CORES
        return "cuda cores"
    if w.paged and w.page_size < 8:   # no fusion; rows copied or gathered
        if G >= 2 and row >= 128:
            return f"tensor cores ({mma}), rows copied with cp.async"
        return "cuda cores" + (", rows gathered four per TMA load" if w.page_size <= 2 else "")
    short = row < 256 or (w.paged and w.page_size < 64)
    tiles = sum((int(L) + 63) // 64 for L in w.seq_lens) * w.num_kv_heads
    long_call = tiles / 152 >= 24
    fp8_single = fp8 and w.head_dim == 128 and G == 1   # paired at any length
    fused = short and (long_call or fp8_single) and any(f * w.head_dim <= 256 and w.num_kv_heads % f == 0 and
                                                        (G <= 16 if f == 2 else 4 * G <= 8) for f in (2, 4))
    if (G == 1 or row < 128) and not fused:
        return "cuda cores"
    tc5_shape = (fused and fp8 and w.head_dim == 128 and G <= 8 and w.num_kv_heads % 2 == 0
                 and (not w.paged or w.page_size >= 64))
    # FD_FLAG_TMEM_SCORES (0x80) forces the tcgen05 scores, FD_FLAG_NO_TMEM_SCORES (0x100) keeps the warp MMAs
    if tc5_shape and not flags & 0x100 and ((G <= 4 and tiles / (2 * 152) >= 24) or flags & 0x80):
        return "tensor cores (tcgen05 FP8 scores into TMEM, mma.sync fp16 P.V), fused kv heads"
    return f"tensor cores ({mma})" + (", fused kv heads" if fused else "")


def max_over_ranks(x: float, dist, device) -> float:
    """The largest value of x over all ranks (x itself without a process group)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tbs(bytes_per_call: int, world: int, ms_per_call_max: float) -> float:
    """Weak scaling: every rank processes one call per step; the slowest rank sets the time."""
    return world * bytes_per_call / (ms_per_call_max * 1e-3) / 1e12


def kernel_hash():
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def bench_workload(args):
    """The workload the arguments name: one of the five configurations, with
    an FP8 cache (--kv) and re-paged into pages of --page tokens when asked."""
    w = syn.make_config(args.config, kv_dtype=args.kv if args.kv != "bf16" else None, shrink=args.shrink,
                        head_dim=args.head_dim, q_len=args.q_len)
    if args.page:
        w = syn.repage(w, args.page, perm_seed=syn.seed_for(args.config, syn.TENSOR_PERM) + args.page)
    return w


def workload_name(args, w):
    """The workload's name: the configuration's, or the variant's (shrink,
    head_dim, q_len)."""
    variant = args.shrink > 1 or args.head_dim != 128 or args.q_len != 1
    return w.name if variant else syn.CONFIG_NAMES[args.config]


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.4)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t_start, t_end):
        """Median SM clock and the throttle reasons seen over the samples taken
        between t_start and t_end (wall clock; every sample if none fell there)."""
        if not self.lines:
            return None
        inside = [ln for ts, ln in self.lines if t_start <= ts <= t_end + 0.1]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in (inside or [ln for _, ln in self.lines]):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "samples_in_timed_region": len(inside)}


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------

class Resident:
    """One workload resident in HBM, called through the binding.  Workloads
    whose K/V fit twice in L2 rotate through copies whose total exceeds 2x L2,
    so every call streams its K/V from HBM."""

    def __init__(self, fd, w, dev, l2, flags):
        import torch
        self.fd, self.w, self.flags = fd, w, flags
        fp8 = w.kv_dtype is not None
        self.kv_opts = dict(kv_dtype=w.kv_dtype, k_scale=w.k_scale, v_scale=w.v_scale) if fp8 else {}

        def todev(bits):
            return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

        def todev_kv(codes):
            return torch.from_numpy(np.ascontiguousarray(codes)).to(dev) if fp8 else todev(codes)

        B, hq, d = w.batch, w.num_q_heads, w.head_dim
        self.q, k, v = todev(w.q), todev_kv(w.k), todev_kv(w.v)
        self.lens = torch.from_numpy(w.seq_lens.astype(np.int32)).to(dev)
        self.lens_h = torch.from_numpy(w.seq_lens.astype(np.int32))
        self.table = torch.from_numpy(w.block_table.astype(np.int32)).to(dev) if w.paged else None
        cap = w.max_blocks * w.page_size if w.paged else w.s_max
        self.ws = fd.make_workspace(B, hq, w.num_kv_heads, d, cap, w.page_size, dev, q_len=w.q_len)
        self.out = torch.empty(tuple(w.q.shape), dtype=torch.float32, device=dev)
        self.lse = torch.empty(tuple(w.q.shape[:-1]), dtype=torch.float32, device=dev)
        self.kv_alloc = w.k.nbytes + w.v.nbytes
        self.copies = 1
        if l2 and self.kv_alloc < 2 * l2:
            self.copies = int(np.ceil(2 * l2 / self.kv_alloc)) + 1
        self.kvs = [(k, v)] + [(k.clone(), v.clone()) for _ in range(self.copies - 1)]
        self.l2_note = (f"rotating {self.copies} K/V copies (> 2x L2)" if self.copies > 1
                        else f"inputs {self.kv_alloc / 2**20:.0f} MiB > L2 {l2 / 2**20:.0f} MiB, no flush")

    def step(self, i, events=None):
        w, fd = self.w, self.fd
        kk, vv = self.kvs[i % self.copies]
        if w.paged:
            fd.fd_decode_paged(self.q, kk, vv, self.table, self.lens, self.lens_h, scale=w.scale, out=self.out,
                               lse=self.lse, workspace=self.ws, split_events=events, flags=self.flags,
                               **self.kv_opts)
        else:
            fd.fd_decode(self.q, kk, vv, self.lens, self.lens_h, scale=w.scale, out=self.out, lse=self.lse,
                         workspace=self.ws, split_events=events, flags=self.flags, **self.kv_opts)

    def chunk(self, steps):
        """Calls per captured graph: 50, a whole number of K/V rotations."""
        c = self.copies
        return min(steps, 50 if c == 1 else c * max(1, 50 // c))


def capture_graph(dev, stream, fn, n):
    """A CUDA graph of fn(0) .. fn(n - 1), captured on a side stream."""
    import torch
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream(dev)
    cs.wait_stream(stream)
    with torch.cuda.stream(cs):
        with torch.cuda.graph(g, stream=cs):
            for i in range(n):
                fn(i)
    stream.wait_stream(cs)
    return g


def time_split_in_graph(res, dev, stream, chunk, calls):
    """The split and merge kernels' times (µs) from CUDA events that the graph
    itself records (the binding's split events become event nodes during
    capture) around every split launch of a graph of `chunk` back-to-back
    calls, replayed until `calls` calls were timed: split = its start to end
    event, merge = the split's end event to the next call's start event.
    An event node between two kernels stops the second from starting early
    (programmatic dependent launch), so each figure carries its kernel's
    launch latency, which the headline graph hides.
    Returns (split µs, merge µs, how)."""
    import torch
    chunk = max(2, chunk)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(chunk)]
    for a_, b_ in ev:          # torch creates the CUDA event on its first record
        a_.record(stream)
        b_.record(stream)
    torch.cuda.synchronize()

    def read(split, merge):
        split += [a_.elapsed_time(b_) * 1e3 for a_, b_ in ev]
        merge += [ev[i][1].elapsed_time(ev[i + 1][0]) * 1e3 for i in range(chunk - 1)]

    split, merge = [], []
    try:
        g = capture_graph(dev, stream, lambda i: res.step(i, ev[i]), chunk)
        g.replay()
        torch.cuda.synchronize()
        for _ in range(max(1, calls // chunk)):
            g.replay()
            torch.cuda.synchronize()
            read(split, merge)
        how = f"events in a CUDA graph of {chunk} calls, {len(split)} launches"
    except Exception as exc:   # report it and time eager launches instead
        torch.cuda.synchronize()
        split, merge = [], []
        for _ in range(max(1, min(calls, 1000) // chunk)):
            for i in range(chunk):
                res.step(i, ev[i])
            torch.cuda.synchronize()
            read(split, merge)
        how = f"eager launches ({type(exc).__name__}: {str(exc)[:120]})"
    return float(np.mean(split)), float(np.mean(merge)), how


def split_time_in_step(us_per_call, split_ev):
    """The split kernel's time for the roofline: its event time inside a
    graph, bounded by the headline graph's whole step (the kernel cannot take
    longer than the step; the events carry its launch latency, which
    programmatic dependent launch hides in the step)."""
    return min(split_ev, us_per_call)


def measure_workload(fd, w, dev, stream, l2, flags, P, peak_gbs, min_calls=1000, min_seconds=0.3, warmup=5):
    """µs per call (a CUDA graph of back-to-back calls, replayed) and the split
    kernel's time, for one workload; a `workloads` entry of the JSON line."""
    import torch
    res = Resident(fd, w, dev, l2, flags)
    for i in range(warmup):
        res.step(i)
    torch.cuda.synchronize()
    assert fd.fd_get_device_error(res.ws) == fd.FD_OK
    chunk = res.chunk(min_calls)
    g = capture_graph(dev, stream, res.step, chunk)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(2):
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    # at least min_calls calls and min_seconds of timed work (so the clock
    # sampler sees the timed region)
    est = e0.elapsed_time(e1) * 1e-3 / chunk
    reps = max(2, -(-min_calls // chunk), int(np.ceil(min_seconds / max(est * chunk, 1e-6))))
    with ClockSampler(dev.index or 0) as clk:
        t_wall0 = time.time()
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        t_wall1 = time.time()
    us = e0.elapsed_time(e1) / (reps * chunk) * 1e3
    split_ev, merge_ev, how = time_split_in_graph(res, dev, stream, chunk, min(min_calls, 500))
    split_us = split_time_in_step(us, split_ev)
    err = fd.fd_get_device_error(res.ws)
    bc = byte_counts(w, P)
    tbs = bc["call"] / (us * 1e-6) / 1e12
    split_gbs = bc["split"] / (split_us * 1e-6) / 1e9
    entry = {"us_per_call": us, "TB/s": tbs, "frac": tbs * 1e3 / peak_gbs,
             "split_us": split_us, "split_frac": split_gbs / peak_gbs, "split_event_us": split_ev,
             "merge_event_us": merge_ev, "split_timing": how,
             "consumers": consumers_label(flags, w), "bytes_per_call": bc["call"], "calls_timed": reps * chunk,
             "launch": f"cuda graph of {chunk} calls", "l2": res.l2_note, "clocks": clk.summary(t_wall0, t_wall1),
             "device_error": fd.fd_status_string(err)}
    del g, res
    torch.cuda.empty_cache()
    return entry


def run_ours(args, rank, world):
    import torch
    import decode_attention_decoding_gb300 as fd
    from decode_attention_decoding_gb300 import build as fdb
    fdb.build()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    w = bench_workload(args)
    B, hq, d = w.batch, w.num_q_heads, w.head_dim
    hkv = w.num_kv_heads
    fp8 = w.kv_dtype is not None
    props = torch.cuda.get_device_properties(dev)
    P = props.multi_processor_count
    l2 = getattr(props, "L2_cache_size", 0) or 0
    stream = torch.cuda.current_stream(dev)
    flags = (fd.FD_FLAG_CUDA_CORES if args.cuda_cores else 0) | \
        {"default": 0, "on": fd.FD_FLAG_TMEM_SCORES, "off": fd.FD_FLAG_NO_TMEM_SCORES}[args.tmem_scores]
    res = Resident(fd, w, dev, l2, flags)
    peaks, peak_src = measured_peaks()

    for i in range(args.warmup):
        res.step(i)
    torch.cuda.synchronize()
    assert fd.fd_get_device_error(res.ws) == fd.FD_OK

    K = args.steps
    # Headline: replay a CUDA graph of `chunk` back-to-back calls (the way a
    # serving loop issues decode steps); eager per-call time is reported too.
    chunk = res.chunk(K)
    graph, graph_error = None, None
    if not args.eager:
        try:
            graph = capture_graph(dev, stream, res.step, chunk)
            for _ in range(2):
                graph.replay()
            torch.cuda.synchronize()
        except Exception as exc:          # report it and time eager calls instead
            graph, graph_error = None, f"{type(exc).__name__}: {exc}"[:200]
            torch.cuda.synchronize()
    reps = max(1, K // chunk) if graph else K
    K = reps * chunk if graph else K
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        # The timed region: K back-to-back calls, nothing between them.
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        t_wall0 = time.time()
        e0.record(stream)
        if graph:
            for _ in range(reps):
                graph.replay()
        else:
            for i in range(K):
                res.step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        t_wall1 = time.time()
        if dist:
            dist.barrier()
    ms_total = e0.elapsed_time(e1)
    # The roofline's kernel time: events recorded by the graph around every
    # split launch (a separate timed pass, same calls, same stream), bounded
    # by the headline step.
    split_ev, merge_ev, split_how = time_split_in_graph(res, dev, stream, res.chunk(K), min(K, 2000))
    # eager calls (host marshalling + two launches per call)
    a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_eager = min(K, 500)
    torch.cuda.synchronize()
    a_.record(stream)
    for i in range(n_eager):
        res.step(i)
    b_.record(stream)
    torch.cuda.synchronize()
    eager_us = a_.elapsed_time(b_) / n_eager * 1e3
    ms_total = max_over_ranks(ms_total, dist, dev)
    ms_step = ms_total / K
    split_us = split_time_in_step(ms_step * 1e3, split_ev)
    bc = byte_counts(w, P)
    value_tbs = whole_job_tbs(bc["call"], world, ms_step)
    achieved_gbs = bc["split"] / (split_us * 1e-6) / 1e9
    traffic = None
    try:
        tj = json.load(open(TRAFFIC_FILE))
        if (tj.get("kernel_hash") == kernel_hash() and tj.get("workload") == workload_name(args, w)
                and not args.page and args.kv == "bf16" and not args.cuda_cores):
            traffic = tj.get("traffic_bytes_per_launch")
    except Exception:
        pass

    # End to end through the public API: pinned host inputs -> device, decode,
    # result -> host, every step.
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(fd, res, dev, stream, bc, world, dist, max(3, min(K, args.e2e_steps)))

    err = fd.fd_get_device_error(res.ws)
    headline_entry = {"us_per_call": ms_step * 1e3, "TB/s": value_tbs / world,
                      "frac": value_tbs * 1e3 / world / peaks["hbm_gbs"], "split_us": split_us,
                      "split_frac": achieved_gbs / peaks["hbm_gbs"], "split_event_us": split_ev,
                      "merge_event_us": merge_ev, "split_timing": split_how,
                      "consumers": consumers_label(flags, w), "bytes_per_call": bc["call"], "calls_timed": K,
                      "launch": f"cuda graph of {chunk} calls" if graph else "eager", "l2": res.l2_note,
                      "clocks": clk.summary(t_wall0, t_wall1), "device_error": fd.fd_status_string(err)}
    l2_note, copies = res.l2_note, res.copies
    del res, graph
    torch.cuda.empty_cache()

    # Every benchmark workload under the same protocol (one GPU only: under
    # torchrun the ranks run the headline replicas alone).
    workloads = None
    if (world == 1 and args.workloads != "none" and not args.page and args.shrink == 1 and args.head_dim == 128
            and args.q_len == 1):
        workloads = {}
        for c in [int(x) for x in args.workloads.split(",")]:
            name = syn.CONFIG_NAMES[c]
            if c == args.config:
                workloads[name] = headline_entry
                continue
            wc = syn.make_config(c, kv_dtype=args.kv if args.kv != "bf16" else None)
            workloads[name] = measure_workload(fd, wc, dev, stream, l2, flags, P, peaks["hbm_gbs"])
            del wc

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value_tbs, "unit": "TB/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_step, "us_per_call": ms_step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "frac_of_peak_hbm": value_tbs * 1e3 / world / peaks["hbm_gbs"],
            "dtype": "f32", "input_dtype": (f"bf16 q, FP8 {w.kv_dtype} K/V (scale {w.k_scale})" if fp8
                                            else "bf16"),
            "data": "synthetic (seeded N(0,1) bf16" + (", quantised once to FP8)" if fp8 else ")"),
            "impl": "ours",
            "config": {"workload": workload_name(args, w), "batch": B, "q_len": w.q_len, "num_q_heads": hq,
                       "num_kv_heads": hkv, "head_dim": d,
                       "kv_lens": ("uniform " + str(int(w.seq_lens[0]))) if len(set(w.seq_lens.tolist())) == 1
                       else f"ragged sum={int(w.seq_lens.sum())}",
                       "layout": f"paged P={w.page_size}" if w.paged else "contiguous",
                       "split_ctas": P, "parallelism": f"replicas x{world}",
                       "launch": headline_entry["launch"],
                       "graph_error": graph_error, "eager_us_per_call": eager_us, "l2": l2_note,
                       "kv_copies": copies},
            "bytes_per_call": bc["call"], "bytes_detail": bc,
            "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved_gbs / peaks["hbm_gbs"], "traffic": traffic,
                         "kernel": "fd::split_kernel", "split_us": split_us,
                         "split_us_how": "min(split kernel time from events recorded inside a CUDA graph, "
                                         "the headline step time)",
                         "split_event_us": split_ev, "merge_event_us": merge_ev, "split_timing": split_how,
                         "consumers": consumers_label(flags, w),
                         "peak_source": f"{peak_src} hbm_gbs (STREAM-style copy)"},
            "gpu_launches": 2 * K,        # split kernel + merge kernel per call
            "clocks": headline_entry["clocks"],
            "e2e": e2e,
            "cpu_baseline": cpu,
            "workloads": workloads,
            "device_error": fd.fd_status_string(err),
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_e2e(fd, res, dev, stream, bc, world, dist, steps):
    """The same metric through the public API with host buffers: every step
    copies q, K, V and the lengths from pinned host memory, decodes, and
    copies O and LSE back (whole tensors on the call's stream: on GB300 one
    pinned copy already runs at the host link's rate, and splitting it over
    streams and chunks only added synchronisation)."""
    import torch
    w = res.w
    fp8 = w.kv_dtype is not None
    hq_ = torch.from_numpy(np.ascontiguousarray(w.q).view(np.int16)).pin_memory()
    hk_, hv_ = (torch.from_numpy(np.ascontiguousarray(x).view(np.uint8 if fp8 else np.int16)).pin_memory()
                for x in (w.k, w.v))
    hl_ = res.lens_h.pin_memory()
    ho = torch.empty(tuple(w.q.shape), dtype=torch.float32).pin_memory()
    hlse = torch.empty(tuple(w.q.shape[:-1]), dtype=torch.float32).pin_memory()
    dq, dk, dv = (torch.empty(x.shape, dtype=x.dtype, device=dev) for x in (hq_, hk_, hv_))
    dl = torch.empty_like(res.lens)

    def e2e_step():
        dk.copy_(hk_, non_blocking=True)
        dv.copy_(hv_, non_blocking=True)
        dq.copy_(hq_, non_blocking=True)
        dl.copy_(hl_, non_blocking=True)
        qb = dq.view(torch.bfloat16)
        kb, vb = (dk, dv) if fp8 else (dk.view(torch.bfloat16), dv.view(torch.bfloat16))
        if w.paged:
            fd.fd_decode_paged(qb, kb, vb, res.table, dl, res.lens_h, scale=w.scale, out=res.out, lse=res.lse,
                               workspace=res.ws, **res.kv_opts)
        else:
            fd.fd_decode(qb, kb, vb, dl, res.lens_h, scale=w.scale, out=res.out, lse=res.lse, workspace=res.ws,
                         **res.kv_opts)
        ho.copy_(res.out, non_blocking=True)
        hlse.copy_(res.lse, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a.elapsed_time(b) / steps, dist, dev)
    h2d = hq_.nbytes + hk_.nbytes + hv_.nbytes + hl_.nbytes
    d2h = ho.numel() * 4 + hlse.numel() * 4
    out = {"value": whole_job_tbs(bc["call"], world, e2e_ms), "unit": "TB/s",
           "us_per_call": e2e_ms * 1e3, "h2d_bytes_per_step": int(h2d),
           "copies": "whole tensors, pinned host memory, on the call's stream",
           "d2h_bytes_per_step": int(d2h), "steps": steps}
    del dq, dk, dv, hk_, hv_
    return out


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------

def oracle_units(w, n_units):
    """The first n_units (request, kv head) units, each with every query row
    of its group over the whole kv length, and their algorithmic bytes: the
    unit's K+V rows once (as the GPU's count, not once per query row), plus
    its q rows, O rows and LSEs."""
    B, hq, hkv, d, ql = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.q_len
    G = hq // hkv
    units = [(b, g) for b in range(B) for g in range(hkv)][:max(1, n_units)]
    items = np.array([[b, i * hq + g * G + j, 0, -1] for b, g in units for i in range(ql) for j in range(G)],
                     dtype=np.int32)
    toks = sum(int(w.seq_lens[b]) for b, _ in units)
    by = toks * d * 2 * w.kv_elem_bytes + len(units) * ql * G * (d * 2 + d * 4 + 4)
    return items, by, len(units)


def time_oracle(w, items, threads):
    import oracle
    t0 = time.perf_counter()
    oracle.attend(w, items=items, threads=threads)
    return time.perf_counter() - t0


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith(("model name", "cpu part")):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or "unknown"


def oracle_rate(w, threads, seconds):
    """TB/s of the oracle on `threads` threads over a sample of units sized to
    take about `seconds`; returns (TB/s, seconds, units, repetitions)."""
    total_units = w.batch * w.num_kv_heads
    n = min(total_units, threads)
    items, by, n = oracle_units(w, n)
    dt = time_oracle(w, items, threads)
    n = int(min(total_units, max(n, n * seconds / max(dt, 1e-3))))
    items, by, n = oracle_units(w, n)
    reps, total, t = 0, 0, 0.0
    while t < seconds and reps < 1000:
        t += time_oracle(w, items, threads)
        total += by
        reps += 1
    return total / t / 1e12, t, n, reps


def cpu_baseline(w, seconds):
    """The fp64 oracle as it stands on the host cores: on every core, and on one."""
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    total_units = w.batch * w.num_kv_heads
    v_all, t_all, n_all, r_all = oracle_rate(w, threads, seconds * 0.6)
    v_one, t_one, n_one, r_one = oracle_rate(w, 1, seconds * 0.4)
    return {"value": v_all, "unit": "TB/s", "cores": threads, "kind": "oracle", "seconds": t_all,
            "cpu_model": cpu_model(),
            "sample": f"{n_all} of {total_units} (request, kv head) units, every query row of each over the "
                      f"whole kv length, x {r_all} repetitions, fp64 C oracle, {threads} threads; bytes = "
                      f"each unit's K+V once plus its q, O and LSE (the GPU's count)",
            "single_thread": {"value": v_one, "unit": "TB/s", "cores": 1, "seconds": t_one,
                              "sample": f"{n_one} units x {r_one} repetitions"}}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = bench_workload(args)
    threads = os.cpu_count() or 1
    total_units = w.batch * w.num_kv_heads
    budget = max(1.0, args.reference_budget_s / max(1, args.steps + args.warmup))
    n = min(total_units, threads)
    items, by, n = oracle_units(w, n)
    dt = time_oracle(w, items, threads)
    n = int(min(total_units, max(1, n * budget / max(dt, 1e-3))))
    items, by, n = oracle_units(w, n)
    for _ in range(args.warmup):
        time_oracle(w, items, threads)
    ts = [time_oracle(w, items, threads) for _ in range(args.steps)]
    t = float(np.sum(ts))
    value = args.steps * by / t / 1e12
    sample = (f"{n} of {total_units} (request, kv head) units per step, every query row of each over the whole "
              f"kv length, fp64 C oracle, {threads} threads; bytes = each unit's K+V once plus q, O, LSE")
    line = {"metric": METRIC, "value": value, "unit": "TB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "input_dtype": f"bf16 q, FP8 {w.kv_dtype} K/V" if w.kv_dtype else "bf16",
            "data": "synthetic (seeded N(0,1) bf16)", "impl": "reference",
            "config": {"workload": workload_name(args, w), "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": "TB/s", "cores": threads, "kind": "oracle",
                             "cpu_model": cpu_model(), "sample": sample},
            "e2e": {"value": value, "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", type=int, default=2, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--kv", default="bf16", choices=["bf16", "e4m3", "e5m2"],
                    help="K/V cache element type (FP8 caches are quantised from the same values)")
    ap.add_argument("--page", type=int, default=0,
                    help="re-page the workload's K/V into shuffled pages of this many tokens "
                         "(a divisor of 64 or a multiple of 64; 0 keeps its own layout)")
    ap.add_argument("--shrink", type=int, default=1,
                    help="divide the workload's lengths by this factor (a smaller case of the same launch "
                         "shape, for profiler captures; never the benchmark's own numbers)")
    ap.add_argument("--head-dim", type=int, default=128, choices=[64, 128, 256],
                    help="the workload with this head_dim (its lengths, heads and layout)")
    ap.add_argument("--q-len", type=int, default=1,
                    help="new query tokens per request (q [B, q_len, Hq, D], causal over the new tokens)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=40)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--eager", action="store_true", help="time eager calls instead of a CUDA graph")
    ap.add_argument("--cuda-cores", action="store_true",
                    help="force the CUDA-core consumers for GQA groups (comparison runs)")
    ap.add_argument("--tmem-scores", choices=("default", "on", "off"), default="default",
                    help="E4M3 caches with paired kv heads: tcgen05 scores into TMEM for up to 4 columns per kv "
                         "head (default), up to 8 (on), or never (off)")
    ap.add_argument("--workloads", default="1,2,3,4,5",
                    help="benchmark workloads also timed on one GPU for the line's `workloads` object "
                         "(comma-separated ids, or 'none')")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--reference-budget-s", type=float, default=120.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world)


if __name__ == "__main__":
    main()
