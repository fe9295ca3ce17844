#!/usr/bin/env python3
"""Benchmark: split-KV decode attention on GB300 (one JSON line on stdout).

Default workload: MHA long-KV decode -- batch 1, 32 query heads = 32 kv heads,
head_dim 128, kv_len 65536, contiguous [S, H, D] bf16 K/V, scale 1/sqrt(128)
(1 GiB of K+V, larger than the 129 MB L2, so no flush is needed between
steps).  A step is one fd_decode call: the split kernel plus the LSE merge.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1..5] [--impl ours|reference]

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

def partial_count(lens, hkv, P):
    """Number of (CTA, segment) partials the stream-K split writes (host mirror of fd_sched.h)."""
    nt = [(int(L) + TILE - 1) // TILE for L in lens]
    T = hkv * sum(nt)
    if T == 0:
        return 0
    base, rem = divmod(T, P)
    cut = rem * (base + 1)

    def cta(t):
        return t // (base + 1) if t < cut else rem + (t - cut) // base

    n = 0
    first = 0
    for b, k in enumerate(nt):
        for _h in range(hkv):
            if k:
                c0, c1 = cta(first), cta(first + k - 1)
                if c1 > c0:
                    n += c1 - c0 + 1
                first += k
    return n


def byte_counts(w, P):
    B, hq, d = w.q.shape
    hkv, G = w.num_kv_heads, w.num_q_heads // w.num_kv_heads
    kv = w.kv_bytes()
    q = B * hq * d * 2
    out = B * hq * d * 4 + B * hq * 4
    parts = partial_count(w.seq_lens, hkv, P)
    ws = parts * G * (d + 1) * 4
    table = (sum((int(L) + w.page_size - 1) // w.page_size for L in w.seq_lens) * 4) if w.paged else 0
    return dict(kv=kv, q=q, out=out, ws_partials=parts, ws_once=ws, table=table, lens=B * 4,
                call=kv + q + out + 2 * ws,
                split=kv + q + ws + out)   # split reads K,V,q; writes partials or final O/LSE


def consumers_label(args, w) -> str:
    """Which consumers the library's default choice runs for this workload."""
    G = w.num_q_heads // w.num_kv_heads
    fp8 = w.kv_dtype is not None
    row = w.head_dim * (1 if fp8 else 2)
    mma = "mma.sync fp16 on FP8 codes" if fp8 else "mma.sync bf16"
    if args.cuda_cores:
        return "cuda cores"
    if w.paged and w.page_size < 8:   # no fusion; rows copied or gathered
        if G >= 2 and row >= 128:
            return f"tensor cores ({mma}), rows copied with cp.async"
        return "cuda cores" + (", rows gathered four per TMA load" if w.page_size <= 2 else "")
    short = row < 256 or (w.paged and w.page_size < 64)
    tiles = sum((int(L) + 63) // 64 for L in w.seq_lens) * w.num_kv_heads
    long_call = tiles / 152 >= 24
    fused = short and long_call and any(f * w.head_dim <= 256 and w.num_kv_heads % f == 0 and
                                        (G <= 16 if f == 2 else 4 * G <= 8) for f in (2, 4))
    if (G == 1 or row < 128) and not fused:
        return "cuda cores"
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
    w = syn.make_config(args.config, kv_dtype=args.kv if args.kv != "bf16" else None)
    if args.page:
        w = syn.repage(w, args.page, perm_seed=syn.seed_for(args.config, syn.TENSOR_PERM) + args.page)
    return w


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
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t_start, t_end):
        if not self.lines:
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
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
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------

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
    B, hq, d = w.q.shape
    hkv = w.num_kv_heads
    fp8 = w.kv_dtype is not None
    kv_opts = dict(kv_dtype=w.kv_dtype, k_scale=w.k_scale, v_scale=w.v_scale) if fp8 else {}

    def todev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    def todev_kv(codes):
        if fp8:
            return torch.from_numpy(np.ascontiguousarray(codes)).to(dev)
        return todev(codes)

    q, k, v = todev(w.q), todev_kv(w.k), todev_kv(w.v)
    lens = torch.from_numpy(w.seq_lens.astype(np.int32)).to(dev)
    lens_h = torch.from_numpy(w.seq_lens.astype(np.int32))
    table = torch.from_numpy(w.block_table.astype(np.int32)).to(dev) if w.paged else None
    cap = w.max_blocks * w.page_size if w.paged else w.s_max
    ws = fd.make_workspace(B, hq, hkv, d, cap, w.page_size, dev)
    out = torch.empty((B, hq, d), dtype=torch.float32, device=dev)
    lse = torch.empty((B, hq), dtype=torch.float32, device=dev)
    props = torch.cuda.get_device_properties(dev)
    P = props.multi_processor_count
    l2 = getattr(props, "L2_cache_size", 0) or 0

    # L2 control: rotate through copies of K/V whose total exceeds 2x L2 when
    # one copy would fit in L2 (config 1); otherwise the inputs alone exceed L2.
    copies = 1
    kv_alloc = (w.k.nbytes + w.v.nbytes)
    if l2 and kv_alloc < 2 * l2:
        copies = int(np.ceil(2 * l2 / kv_alloc)) + 1
    kvs = [(k, v)] + [(k.clone(), v.clone()) for _ in range(copies - 1)]
    stream = torch.cuda.current_stream(dev)

    flags = fd.FD_FLAG_CUDA_CORES if args.cuda_cores else 0

    def step(i, events=None):
        kk, vv = kvs[i % copies]
        if w.paged:
            fd.fd_decode_paged(q, kk, vv, table, lens, lens_h, scale=w.scale, out=out, lse=lse, workspace=ws,
                               split_events=events, flags=flags, **kv_opts)
        else:
            fd.fd_decode(q, kk, vv, lens, lens_h, scale=w.scale, out=out, lse=lse, workspace=ws,
                         split_events=events, flags=flags, **kv_opts)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    assert fd.fd_get_device_error(ws) == fd.FD_OK

    K = args.steps
    # Headline: replay a CUDA graph of `chunk` back-to-back calls (the way a
    # serving loop issues decode steps); eager per-call time is reported too.
    chunk = min(K, 50 if copies == 1 else copies * max(1, 50 // copies))
    graph, graph_error = None, None
    if not args.eager:
        try:
            graph = torch.cuda.CUDAGraph()
            cap_stream = torch.cuda.Stream(dev)
            cap_stream.wait_stream(stream)
            with torch.cuda.stream(cap_stream):
                with torch.cuda.graph(graph, stream=cap_stream):
                    for i in range(chunk):
                        step(i)
            stream.wait_stream(cap_stream)
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
        # Timed region 1 (the headline): K back-to-back calls, nothing between them.
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
                step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        t_wall1 = time.time()
        if dist:
            dist.barrier()
        # Timed region 2 (the roofline): eager calls with CUDA events recorded
        # on the stream around every split-kernel launch.
        K2 = min(K, 2000)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K2)]
        for a_, b_ in ev:          # torch creates the CUDA event on first record
            a_.record(stream)
            b_.record(stream)
        torch.cuda.synchronize()
        for i in range(K2):
            step(i, ev[i])
        torch.cuda.synchronize()
    ms_total = e0.elapsed_time(e1)
    split_ms = [a_.elapsed_time(b_) for a_, b_ in ev]
    # eager calls without events (host marshalling + two launches per call)
    a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_eager = min(K, 500)
    torch.cuda.synchronize()
    a_.record(stream)
    for i in range(n_eager):
        step(i)
    b_.record(stream)
    torch.cuda.synchronize()
    eager_us = a_.elapsed_time(b_) / n_eager * 1e3
    ms_total = max_over_ranks(ms_total, dist, dev)
    ms_step = ms_total / K
    bc = byte_counts(w, P)
    value_tbs = whole_job_tbs(bc["call"], world, ms_step)
    split_avg_ms = float(np.mean(split_ms))
    peaks, peak_src = measured_peaks()
    achieved_gbs = bc["split"] / (split_avg_ms * 1e-3) / 1e9
    traffic = None
    try:
        tj = json.load(open(TRAFFIC_FILE))
        if (tj.get("kernel_hash") == kernel_hash() and tj.get("workload") == syn.CONFIG_NAMES[args.config]
                and not args.page and args.kv == "bf16"):
            traffic = tj.get("traffic_bytes_per_launch")
    except Exception:
        pass

    # End to end through the public API: pinned host inputs -> device, decode,
    # result -> host, every step.
    e2e = None
    if not args.no_e2e:
        hq_ = torch.from_numpy(np.ascontiguousarray(w.q).view(np.int16)).pin_memory()
        hk_, hv_ = (torch.from_numpy(np.ascontiguousarray(x).view(np.uint8 if fp8 else np.int16)).pin_memory()
                    for x in (w.k, w.v))
        hl_ = lens_h.pin_memory()
        ho = torch.empty((B, hq, d), dtype=torch.float32).pin_memory()
        hlse = torch.empty((B, hq), dtype=torch.float32).pin_memory()
        dq, dk, dv = (torch.empty(x.shape, dtype=x.dtype, device=dev) for x in (hq_, hk_, hv_))
        dl = torch.empty_like(lens)
        K2 = max(3, min(K, args.e2e_steps))

        # Host->device copies of the step's inputs on the call's stream, whole
        # tensors: on GB300 one pinned copy already runs at the link's rate
        # (~211 GB/s), and splitting it over streams and chunks only added
        # synchronisation (6.5 ms per step instead of 5.3 for workload 2).
        def e2e_step():
            dk.copy_(hk_, non_blocking=True)
            dv.copy_(hv_, non_blocking=True)
            dq.copy_(hq_, non_blocking=True)
            dl.copy_(hl_, non_blocking=True)
            qb = dq.view(torch.bfloat16)
            kb, vb = (dk, dv) if fp8 else (dk.view(torch.bfloat16), dv.view(torch.bfloat16))
            if w.paged:
                fd.fd_decode_paged(qb, kb, vb, table, dl, lens_h, scale=w.scale, out=out, lse=lse, workspace=ws,
                                   **kv_opts)
            else:
                fd.fd_decode(qb, kb, vb, dl, lens_h, scale=w.scale, out=out, lse=lse, workspace=ws, **kv_opts)
            ho.copy_(out, non_blocking=True)
            hlse.copy_(lse, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(K2):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(a.elapsed_time(b) / K2, dist, dev)
        h2d = hq_.nbytes + hk_.nbytes + hv_.nbytes + hl_.nbytes
        d2h = ho.numel() * 4 + hlse.numel() * 4
        e2e = {"value": whole_job_tbs(bc["call"], world, e2e_ms), "unit": "TB/s",
               "us_per_call": e2e_ms * 1e3, "h2d_bytes_per_step": int(h2d),
               "copies": "whole tensors, pinned host memory, on the call's stream",
               "d2h_bytes_per_step": int(d2h), "steps": K2}

    err = fd.fd_get_device_error(ws)
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
            "config": {"workload": syn.CONFIG_NAMES[args.config], "batch": B, "num_q_heads": hq,
                       "num_kv_heads": hkv, "head_dim": d,
                       "kv_lens": ("uniform " + str(int(w.seq_lens[0]))) if len(set(w.seq_lens.tolist())) == 1
                       else f"ragged sum={int(w.seq_lens.sum())}",
                       "layout": f"paged P={w.page_size}" if w.paged else "contiguous",
                       "split_ctas": P, "parallelism": f"replicas x{world}",
                       "launch": f"cuda graph of {chunk} calls" if graph else "eager",
                       "graph_error": graph_error, "eager_us_per_call": eager_us,
                       "l2": (f"rotating {copies} K/V copies (> 2x L2)" if copies > 1
                              else f"inputs {kv_alloc / 2**20:.0f} MiB > L2 {l2 / 2**20:.0f} MiB, no flush")},
            "bytes_per_call": bc["call"], "bytes_detail": bc,
            "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved_gbs / peaks["hbm_gbs"], "traffic": traffic,
                         "kernel": "fd::split_kernel", "split_us": split_avg_ms * 1e3,
                         "consumers": consumers_label(args, w),
                         "peak_source": f"{peak_src} hbm_gbs (STREAM-style copy)"},
            "gpu_launches": 2 * K,        # split kernel + merge kernel per call
            "clocks": clk.summary(t_wall0, t_wall1),
            "e2e": e2e,
            "cpu_baseline": cpu,
            "device_error": fd.fd_status_string(err),
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(w, n_rows):
    """The first n_rows (b, h) query rows over their whole length."""
    B, hq = w.batch, w.num_q_heads
    rows = [(b, h) for b in range(B) for h in range(hq)][:max(1, n_rows)]
    items = np.array([[b, h, 0, -1] for b, h in rows], dtype=np.int32)
    toks = sum(int(w.seq_lens[b]) for b, _ in rows)
    # bytes the oracle streams for these rows: K+V row per token (per query head)
    return items, toks * w.head_dim * 2 * w.kv_elem_bytes


def time_oracle(w, items, threads):
    import oracle
    t0 = time.perf_counter()
    oracle.attend(w, items=items, threads=threads)
    return time.perf_counter() - t0


def cpu_baseline(w, seconds):
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    total_rows = w.batch * w.num_q_heads
    # calibrate on a few rows, then size the sample to about `seconds`
    n = min(total_rows, threads)
    items, by = oracle_sample(w, n)
    dt = time_oracle(w, items, threads)
    n = int(min(total_rows, max(n, n * seconds / max(dt, 1e-3))))
    items, by = oracle_sample(w, n)
    reps, total, t = 0, 0, 0.0
    while t < seconds and reps < 1000:
        t += time_oracle(w, items, threads)
        total += by
        reps += 1
    return {"value": total / t / 1e12, "unit": "TB/s", "cores": threads, "kind": "oracle",
            "seconds": t,
            "sample": f"{n} of {total_rows} query rows (whole kv length each) x {reps} repetitions, "
                      f"fp64 C oracle, {threads} threads; bytes = K+V rows streamed per query row"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = bench_workload(args)
    threads = os.cpu_count() or 1
    total_rows = w.batch * w.num_q_heads
    budget = max(1.0, args.reference_budget_s / max(1, args.steps + args.warmup))
    n = min(total_rows, threads)
    items, by = oracle_sample(w, n)
    dt = time_oracle(w, items, threads)
    n = int(min(total_rows, max(1, n * budget / max(dt, 1e-3))))
    items, by = oracle_sample(w, n)
    for _ in range(args.warmup):
        time_oracle(w, items, threads)
    ts = [time_oracle(w, items, threads) for _ in range(args.steps)]
    t = float(np.sum(ts))
    value = args.steps * by / t / 1e12
    sample = (f"{n} of {total_rows} query rows per step (whole kv length each), fp64 C oracle, "
              f"{threads} threads")
    line = {"metric": METRIC, "value": value, "unit": "TB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "input_dtype": f"bf16 q, FP8 {w.kv_dtype} K/V" if w.kv_dtype else "bf16",
            "data": "synthetic (seeded N(0,1) bf16)", "impl": "reference",
            "config": {"workload": syn.CONFIG_NAMES[args.config], "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": "TB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
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
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=40)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--eager", action="store_true", help="time eager calls instead of a CUDA graph")
    ap.add_argument("--cuda-cores", action="store_true",
                    help="force the CUDA-core consumers for GQA groups (comparison runs)")
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
