"""Benchmark of the selected-index NoPE MLA paged decode on GB300.

A step is one full decode call (index resolution + query split, the decode kernel, the
log-sum-exp combine) over one batch of the workload, inputs resident in HBM. Steps are
captured into CUDA graphs and timed with CUDA events on the launching stream; each step
reads a different input replica and the replicas together exceed L2, so no step finds
its inputs in L2. Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Under torchrun each rank runs its own replicas on its own GPU (no data-path collective,
weak scaling); the time is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_mla_paged_gb300 import workloads as wl  # noqa: E402

METRIC = "sparse MLA decode µs/step; effective HBM TB/s & % roofline (1×GB300)"
UNIT = "us/step"
L2_BYTES = 129 * 1024 * 1024
WORKLOADS = {"tiny": 0, "decode_batch": 1, "ragged": 2, "pooled_128k": 3, "verify_k4": 4}
# The largest workload that fits one GPU (128 sequences x 128 heads over a 16M-token pool).
DEFAULT_WORKLOAD = "pooled_128k"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM bytes (read + write) of one decode-kernel launch of each workload, as counted by
# ncu (dram__bytes_read.sum + dram__bytes_write.sum) on the decode kernel as it is now. A
# workload absent here reports traffic null; an entry is dropped whenever the decode
# kernel changes, until it is counted again.
MEASURED_TRAFFIC = {"pooled_128k": 153921536, "ragged": 72731648, "verify_k4": 67966976, "decode_batch": 8965888}


# ----------------------------------------------------------------------------------------
# distributed plumbing (one process per GPU under torchrun)
# ----------------------------------------------------------------------------------------

def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws: int, backend: str):
    if ws > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend=backend)


def barrier(ws: int):
    if ws > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def shard_replicas(n_total: int, ws: int, rank: int):
    """Replica seeds owned by a rank: every rank runs the same per-rank batch size with
    its own inputs (weak scaling); seeds never collide across ranks."""
    return [rank * 100003 + i for i in range(n_total)]


# ----------------------------------------------------------------------------------------
# workload accounting (no decode arithmetic: counts of what a step must move)
# ----------------------------------------------------------------------------------------

def algorithmic_cost(w: wl.Workload) -> dict:
    """Bytes a step must move and flops it must do, per the decode's definition:
    each distinct selected token's 512-byte row once per sequence (twice when K and V are
    separate buffers), the BF16 queries and outputs, the selection rows and the touched
    block-table entries; 4*H*512 flops per selected token per row."""
    sel = w.sel_indices.to(torch.int64)
    R, W = sel.shape
    lens = w.seq_lens.to(torch.int64).reshape(R, 1)
    valid = (sel >= 0) & (sel < lens)
    key = torch.where(valid, sel, torch.full_like(sel, -1))
    per_row = torch.tensor([torch.unique(key[r][key[r] >= 0]).numel() for r in range(R)])
    seqs = w.num_seqs
    rps = w.rows_per_seq
    union_tokens, pages = 0, 0
    for s in range(seqs):
        ids = key[s * rps:(s + 1) * rps].reshape(-1)
        u = torch.unique(ids[ids >= 0])
        union_tokens += u.numel()
        pages += torch.unique(u // w.block_size).numel()
    kv = union_tokens * 512 * (1 if w.v_cache is None else 2)
    q = R * w.num_q_heads * 512 * 2
    out = q
    ids_b = R * W * 4
    bt = pages * 4
    flops = 4 * w.num_q_heads * 512 * int(per_row.sum())
    return {"bytes": kv + q + out + ids_b + bt, "kv_bytes": kv, "flops": flops,
            "selected_tokens": int(per_row.sum()), "union_tokens": union_tokens}


def event_ms(ev0: torch.cuda.Event, ev1: torch.cuda.Event) -> float:
    """Elapsed time between two events recorded by the library (inside a captured graph),
    read with the CUDA runtime's cudaEventElapsedTime (torch only times events it
    recorded itself)."""
    import ctypes
    global _LIBCUDART
    if _LIBCUDART is None:
        _LIBCUDART = ctypes.CDLL("libcudart.so.13")
        _LIBCUDART.cudaEventElapsedTime.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_void_p,
                                                    ctypes.c_void_p]
        _LIBCUDART.cudaEventElapsedTime.restype = ctypes.c_int
    ms = ctypes.c_float(0.0)
    rc = _LIBCUDART.cudaEventElapsedTime(ctypes.byref(ms), ev0.cuda_event, ev1.cuda_event)
    if rc != 0:
        raise RuntimeError(f"cudaEventElapsedTime failed ({rc})")
    return float(ms.value)


_LIBCUDART = None


def load_peaks() -> tuple[dict, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.proc = None
        self.lines = []
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        return time.time()

    def stop(self, t0: float, t1: float) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=2)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                rows.append((ts, float(parts[0]), float(parts[1]), parts[3:]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 - 0.06 <= r[0] <= t1 + 0.06] or rows
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median([r[1] for r in inside])), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside)}


# ----------------------------------------------------------------------------------------
# the CUDA arm
# ----------------------------------------------------------------------------------------

def make_replicas(idx: int, seeds, device, num_seqs=None):
    reps = [wl.config(idx, device=device, seed=wl.BASE_SEED + idx + 7919 * s, num_seqs=num_seqs) for s in seeds]
    return reps


def replica_count(idx: int) -> int:
    """Input replicas per GPU so that consecutive steps never share inputs in L2: the
    small workloads (under 20 MB a step) rotate 64 replicas, the large ones 2-4."""
    return {0: 64, 1: 64, 2: 4, 3: 2, 4: 4}[idx]


def run_cuda(args, ws_n, rank, local):
    import sparse_mla_paged_gb300.api as api

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    idx = WORKLOADS[args.workload]
    n_rep = args.replicas or replica_count(idx)
    reps = make_replicas(idx, shard_replicas(n_rep, ws_n, rank), device, args.seqs or None)
    w0 = reps[0]
    cost = algorithmic_cost(w0)
    verify = w0.base_lens is not None
    ws = api.alloc_workspace(w0.num_seqs, w0.rows_per_seq, w0.num_q_heads, w0.sel_width, args.ctas, device=device)
    outs = [torch.empty_like(r.q) for r in reps]
    stream = torch.cuda.Stream(device)
    K, W = args.steps, args.warmup

    def step(i, s, ev0=None, ev1=None):
        r = reps[i % n_rep]
        api.decode_workload(r, out=outs[i % n_rep], workspace=ws, num_ctas=args.ctas, verify=verify,
                            stream=s, ev_begin=ev0, ev_end=ev1, tile_tokens=args.tile, gather_mode=args.gather_mode)

    # warm-up, eager
    with torch.cuda.stream(stream):
        for i in range(max(W, 1)):
            step(i, stream)
    stream.synchronize()
    assert api.read_device_status(ws, stream) == 0, "device status after warm-up"

    # graphs of g steps (and a remainder graph) with events around every decode kernel
    g = min(K, args.graph_steps)
    reps_per_graph = K // g
    rem = K - reps_per_graph * g
    n_ev = g
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    for ev in ev_b + ev_e:                # creates the CUDA events (torch creates them lazily)
        ev.record(stream)
    stream.synchronize()
    assert all(ev.cuda_event for ev in ev_b + ev_e)

    def capture(n, base, with_events):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                for j in range(n):
                    if with_events:
                        step(base + j, stream, ev_b[base + j], ev_e[base + j])
                    else:
                        step(base + j, stream)
        return graph

    # `value` is timed on graphs without event nodes (an event record between two kernels
    # would cut the programmatic launch overlap); the decode-kernel durations come from a
    # second graph of the same steps with events around every decode kernel.
    main = capture(g, 0, False)
    tail = capture(rem, g, False) if rem else None
    timing = capture(g, 0, True)
    with torch.cuda.stream(stream):
        main.replay()                     # untimed replays: warm the graphs
        timing.replay()
    stream.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws_n)
    torch.cuda.synchronize()
    wall0 = time.time()
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for _ in range(reps_per_graph):
            main.replay()
        if tail is not None:
            tail.replay()
        t_end.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    wall1 = time.time()
    barrier(ws_n)
    with torch.cuda.stream(stream):
        timing.replay()
    stream.synchronize()
    kernel_ms = [event_ms(ev_b[j], ev_e[j]) for j in range(g)]
    clocks = sampler.stop(wall0, wall1)
    total_ms = t_start.elapsed_time(t_end)
    total_ms = max_over_ranks(total_ms, ws_n, device)
    us_per_step = total_ms * 1e3 / K
    kernel_us = float(np.mean(kernel_ms)) * 1e3

    # e2e: the C-ABI call with host buffers (pinned), copies inside the timed region
    e2e = run_e2e(api, reps, args, device, ws_n) if not args.skip_e2e else None

    peaks, peak_src = load_peaks()
    bw = float(peaks["hbm_gbs"])
    tf = float(peaks["bf16_tflops"])
    t_bytes = cost["bytes"] / (bw * 1e9)
    t_flops = cost["flops"] / (tf * 1e12)
    roof_us = max(t_bytes, t_flops) * 1e6
    bound = "hbm" if t_bytes >= t_flops else "tensor"
    if bound == "hbm":
        achieved = cost["bytes"] / (kernel_us * 1e-6) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": bw, "unit": "GB/s",
                "frac": round(achieved / bw, 4)}
    else:
        achieved = cost["flops"] / (kernel_us * 1e-6) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": tf, "unit": "TFLOP/s",
                "frac": round(achieved / tf, 4)}
    traffic = args.traffic if args.traffic is not None else MEASURED_TRAFFIC.get(args.workload)
    roof.update({"traffic": traffic, "peak_source": f"{peak_src} (MEASURED_PEAKS.json)" if
                 peak_src == "measured" else "fallback (6.8 TB/s, 1.9 PFLOP/s)",
                 "kernel": "decode_kernel", "kernel_us": round(kernel_us, 3),
                 "step_roofline_us": round(roof_us, 3), "step_frac": round(roof_us / us_per_step, 4)})
    launches_per_step = 3 if needs_combine(api, w0, args.ctas) else 2
    line = {
        "metric": METRIC, "value": round(us_per_step, 3), "unit": UNIT, "n_gpus": ws_n, "steps": K,
        "warmup": W, "ms_per_step": round(us_per_step / 1e3, 6), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
        "effective_tbs": round(ws_n * cost["bytes"] / (us_per_step * 1e-6) / 1e12, 4),
        "config": config_dict(w0, cost, n_rep, g, ws_n),
        "roofline": roof,
        "gpu_launches": K * launches_per_step,
        "clocks": clocks,
        "e2e": e2e,
    }
    line["_w0"] = w0
    return line


def config_dict(w: wl.Workload, cost: dict, n_rep: int, graph_steps: int, ws_n: int) -> dict:
    """The workload description printed by both arms (identical keys and values)."""
    return {"workload": w.name, "rows": w.rows, "heads": w.num_q_heads, "sel_width": w.sel_width,
            "block_size": w.block_size, "selected_tokens_per_step": cost["selected_tokens"],
            "algorithmic_bytes_per_step": cost["bytes"], "algorithmic_flops_per_step": cost["flops"],
            "l2": f"{n_rep} rotating input replicas per GPU, inputs of consecutive steps differ and "
                  f"exceed L2 together", "graph_steps": graph_steps,
            "parallelism": f"replicas x{ws_n}" if ws_n > 1 else "1 GPU"}


def needs_combine(api, w, ctas) -> bool:
    # The combine runs when some CTA boundary of the slot partition falls inside a unit.
    groups = (w.num_q_heads + 63) // 64
    T = w.rows * groups * w.sel_width
    ctas = api.decode_grid(w.num_seqs, w.rows_per_seq, w.num_q_heads, w.sel_width, ctas)
    return any((k * T // ctas) % w.sel_width != 0 for k in range(1, ctas))


def run_e2e(api, reps, args, device, ws_n):
    """Same metric through dsa_mla_decode_host: per step, H2D of q / block tables /
    seq_lens / selection from pinned memory, the decode, D2H of the output. Consecutive
    steps rotate over `--e2e-lanes` streams (default 3), each with its own device
    workspace and pinned host buffers, so that one step's copies overlap other steps'
    kernels, as a serving loop with that many requests in flight does. (At the pooled
    128K shape a step copies 17 MB each way; pinned copies run at about 0.2 TB/s per
    direction here, so with two lanes the loop is bound by the copies, with three by the
    kernels.)"""
    n = min(len(reps), 8)
    w0 = reps[0]
    verify = w0.base_lens is not None
    lanes = max(1, args.e2e_lanes)
    host = []
    for k in range(lanes):
        r = reps[k % n]
        lens = r.base_lens if verify else r.seq_lens
        host.append(dict(q=r.q.cpu().pin_memory(), bt=r.block_tables.cpu().pin_memory(),
                         sl=lens.cpu().pin_memory(), sel=r.sel_indices.cpu().pin_memory(),
                         out=torch.empty(r.q.shape, dtype=torch.bfloat16).pin_memory(), dev=r))
    nb = api.host_workspace_bytes(w0.num_seqs, w0.rows_per_seq, w0.num_q_heads, w0.sel_width,
                                  w0.block_tables.shape[0], w0.max_blocks_per_seq, int(verify), args.ctas)
    wss = [torch.zeros(nb, dtype=torch.uint8, device=device) for _ in range(lanes)]
    streams = [torch.cuda.Stream(device) for _ in range(lanes)]

    def call(i):
        h = host[i % lanes]
        r = h["dev"]
        vc = r.k_cache if r.v_cache is None else r.v_cache
        api.decode_host(h["q"], r.k_cache, vc, h["bt"], r.max_blocks_per_seq, h["sl"], h["sel"], r.num_seqs,
                        r.rows_per_seq, r.num_q_heads, r.block_size, r.cache_stride_bytes, r.k_scale, r.v_scale,
                        r.sm_scale, h["out"], wss[i % lanes], verify_rows=int(verify), num_ctas=args.ctas,
                        stream=streams[i % lanes])

    steps = max(1, min(args.steps, args.e2e_steps))
    # a lane's host buffers are reused by its next step, queued behind its copies
    for i in range(4):
        call(i)
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    done = [torch.cuda.Event() for _ in range(lanes)]
    barrier(ws_n)
    e0.record(streams[0])
    for s in streams[1:]:
        s.wait_event(e0)
    for i in range(steps):
        call(i)
    for k, s in enumerate(streams):
        done[k].record(s)
        streams[0].wait_event(done[k])
    e1.record(streams[0])
    streams[0].synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), ws_n, device)
    h = host[0]
    h2d = sum(t.numel() * t.element_size() for t in (h["q"], h["bt"], h["sl"], h["sel"]))
    d2h = h["out"].numel() * 2
    return {"value": round(ms * 1e3 / steps, 3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": steps,
            "api": f"dsa_mla_decode_host, {lanes} streams in rotation"}


# ----------------------------------------------------------------------------------------
# the CPU oracle: baseline and reference arm
# ----------------------------------------------------------------------------------------

def oracle_step_sample(w: wl.Workload, budget_s: float):
    """Times the oracle on whole rows of the workload until the budget is spent and
    returns (us per full step, rows timed, threads)."""
    import oracle

    oracle.build()
    threads = oracle.online_cores()
    rows_total = w.rows
    timed_rows, t_total = 0, 0.0
    order = np.random.default_rng(0).permutation(rows_total)
    i = 0
    while t_total < budget_s or timed_rows == 0:
        r = int(order[i % rows_total])
        t0 = time.perf_counter()
        oracle.decode_workload(w, rows=[r], threads=threads)
        t_total += time.perf_counter() - t0
        timed_rows += 1
        i += 1
        if timed_rows >= 4 * rows_total and t_total >= min(budget_s, 1.0):
            break
    per_row = t_total / timed_rows
    return per_row * rows_total * 1e6, timed_rows, threads


def cpu_sample_workload(w: wl.Workload) -> wl.Workload:
    """A CPU copy of a few sequences of w (only their pages), for timing the oracle."""
    seqs = sorted({0, w.num_seqs // 2, w.num_seqs - 1})
    sub, _ = w.subset(seqs)
    return sub


def cpu_baseline(w: wl.Workload, budget_s: float) -> dict:
    sub = cpu_sample_workload(w)
    us_sub, rows, threads = oracle_step_sample(sub, budget_s)
    us = us_sub / sub.rows * w.rows
    return {"value": round(us, 1), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{rows} whole decode rows (all {w.num_q_heads} heads each) drawn from "
                      f"{sub.num_seqs} sequences of the same inputs, timed and scaled to the "
                      f"{w.rows}-row step; float64 C oracle, {threads} threads over (row, head)"}


def run_reference(args, ws_n, rank):
    idx = WORKLOADS[args.workload]
    dev = "cuda" if (idx >= 2 and torch.cuda.is_available()) else "cpu"
    full = wl.config(idx, device=dev, num_seqs=args.seqs or None)
    cost = algorithmic_cost(full)
    n_rep = args.replicas or replica_count(idx)
    config = config_dict(full, cost, n_rep, min(args.steps, args.graph_steps), ws_n)
    w = cpu_sample_workload(full)
    scale = full.rows / w.rows
    budget = max(0.05, min(2.0, 90.0 / max(1, args.steps + args.warmup)))
    import oracle

    oracle.build()
    threads = oracle.online_cores()
    for _ in range(args.warmup):
        oracle_step_sample(w, budget)
    times = []
    rows_timed = 0
    for _ in range(args.steps):
        us, rows, _ = oracle_step_sample(w, budget)
        times.append(us * scale)
        rows_timed += rows
    value = float(np.mean(times))
    return {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws_n, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(value / 1e3, 3), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": config,
            "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"per step: whole decode rows timed for ~{budget:.2f} s and scaled to "
                                       f"the {full.rows}-row step ({rows_timed} rows over {args.steps} steps)"},
            "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ----------------------------------------------------------------------------------------
# component: the cache writer
# ----------------------------------------------------------------------------------------

def _time_in_graphs(call, steps, warmup, stream) -> tuple[float, int]:
    """Average device time of call(i) in microseconds: up to 256 calls captured in one CUDA
    graph, the graph replayed until `steps` calls ran; CUDA events on the launching stream."""
    with torch.cuda.stream(stream):
        for i in range(max(warmup, 3)):
            call(i)
    stream.synchronize()
    n = min(steps, 256)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            for i in range(n):
                call(i)
        graph.replay()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = max(1, steps // n)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            graph.replay()
        e1.record(stream)
    stream.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (reps * n), reps * n


def _hbm_roofline(nbytes: int, us: float) -> dict:
    peaks, _ = load_peaks()
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"bound": "hbm", "achieved": round(gbs, 1), "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
            "frac": round(gbs / float(peaks["hbm_gbs"]), 4)}


def run_latent_write(args):
    """Times dsa_latent_write (RMSNorm + cache scale + E4M3 into scattered slots of a 1 GiB
    pool) for `--rows` new tokens per call, 8 rotating input sets, in CUDA graphs. Bytes
    per row: 1 KiB of kv_a read, 512 B written, the slot; the 1 KiB weight once per call."""
    import sparse_mla_paged_gb300.api as api

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    rows, bs, pages = args.rows, 64, (1 << 30) // (64 * 512)
    g = torch.Generator(device=device)
    g.manual_seed(wl.BASE_SEED)
    cache = torch.zeros(pages * bs * 512, dtype=torch.uint8, device=device)
    sets = []
    for _ in range(8):
        x = torch.randn((rows, 512), generator=g, device=device).to(torch.bfloat16)
        slots = torch.randperm(pages * bs, generator=g, device=device)[:rows].to(torch.int64)
        sets.append((x, slots))
    w = (0.5 + torch.rand(512, generator=g, device=device)).to(torch.bfloat16)
    stream = torch.cuda.Stream(device)

    def call(i):
        x, sl = sets[i % 8]
        api.latent_write(x, w, sl, 1e-6, 0.05, bs, bs * 512, cache, stream=stream)

    us, calls = _time_in_graphs(call, args.steps, args.warmup, stream)
    nbytes = rows * (1024 + 512 + 8) + 1024
    return {"component": "latent_write", "rows": rows, "value": round(us, 3), "unit": "us/call",
            "bytes_per_call": nbytes, "calls": calls, "roofline": _hbm_roofline(nbytes, us)}


def run_select(args):
    """Times dsa_select_pools on the pooled 128K shape: `--rows` rows (default 128) of 32768
    pooled scores, 512 pools of 4 per row, every pool eligible; 16 rotating input sets
    (268 MB, above L2). Bytes per call: the scores and positions read, the ids written."""
    import sparse_mla_paged_gb300.api as api

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    rows, n_pools, kpool, topk = args.rows, 32768, 4, 512
    sets = [wl.pool_scores(rows, n_pools, kpool, device=device, seed=wl.BASE_SEED + i) for i in range(16)]
    outs = [torch.empty((rows, topk * kpool), dtype=torch.int32, device=device) for _ in range(2)]
    stream = torch.cuda.Stream(device)

    def call(i):
        sc, q = sets[i % 16]
        api.select_pools(sc, q, kpool, topk, out=outs[i % 2], stream=stream)

    us, calls = _time_in_graphs(call, args.steps, args.warmup, stream)
    nbytes = rows * (n_pools * 4 + 4 + topk * kpool * 4)
    return {"component": "select", "rows": rows, "n_pools": n_pools, "kpool": kpool, "index_topk": topk,
            "value": round(us, 3), "unit": "us/call", "bytes_per_call": nbytes, "calls": calls,
            "roofline": _hbm_roofline(nbytes, us)}


def run_absorb(args):
    """Times dsa_absorb_q and dsa_absorb_o (FP32 out) at the model size the pages' widths
    give: 64 heads, nope = vd = 256, kvl 512, q_lora_rank 2048, hidden 6144. Each is a
    batched BF16 GEMM; its roofline is the larger of its bytes (weights read, FP32 result
    written) over measured HBM and its flops over the measured dense BF16 peak. At K = 256
    both are HBM-bound (about 93 flops per byte)."""
    import sparse_mla_paged_gb300.api as api

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    H, nope, vd, kvl, ql, hidden = 64, 256, 256, 512, 2048, 6144
    q_b, kv_b, o_proj = wl.absorb_weights(H, nope, vd, kvl, ql, hidden, device=device)
    qa = torch.empty((H * kvl, ql), dtype=torch.float32, device=device)
    oa = torch.empty((hidden, H * kvl), dtype=torch.float32, device=device)
    stream = torch.cuda.Stream(device)
    peaks, _ = load_peaks()
    hbm, tensor = float(peaks["hbm_gbs"]), float(peaks["bf16_tflops"])
    res = {"component": "absorb", "heads": H, "nope": nope, "vd": vd, "kvl": kvl, "q_lora_rank": ql,
           "hidden": hidden, "unit": "us/call"}
    cases = (("absorb_q", lambda i: api.absorb_q(q_b, kv_b, H, nope, vd, out=qa, stream=stream),
              2.0 * H * kvl * ql * nope, 2 * H * nope * ql + 2 * H * nope * kvl + 4 * H * kvl * ql),
             ("absorb_o", lambda i: api.absorb_o(o_proj, kv_b, H, nope, vd, out=oa, stream=stream),
              2.0 * hidden * H * kvl * vd, 2 * hidden * H * vd + 2 * H * vd * kvl + 4 * hidden * H * kvl))
    for name, call, flops, nbytes in cases:
        us, calls = _time_in_graphs(call, min(args.steps, 512), args.warmup, stream)
        t_hbm, t_tensor = nbytes / (hbm * 1e3), flops / (tensor * 1e6)  # microseconds
        if t_hbm >= t_tensor:
            roof = {"bound": "hbm", "achieved": round(nbytes / (us * 1e3), 1), "peak": hbm, "unit": "GB/s"}
        else:
            roof = {"bound": "tensor", "achieved": round(flops / (us * 1e6), 1), "peak": tensor, "unit": "TFLOP/s"}
        roof["frac"] = round(max(t_hbm, t_tensor) / us, 4)
        res[name] = {"value": round(us, 2), "calls": calls, "flops_per_call": flops, "bytes_per_call": nbytes,
                     "tensor_tflops": round(flops / (us * 1e6), 1), "roofline": roof}
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=51200)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", choices=["cuda", "reference"], default="cuda")
    ap.add_argument("--workload", choices=list(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--ctas", type=int, default=0, help="decode grid size (0 = library default)")
    ap.add_argument("--tile", type=int, default=0, choices=[0, 64, 128],
                    help="decode tile in tokens (0 = library default)")
    ap.add_argument("--gather-mode", type=int, default=0, choices=[0, 1, 2],
                    help="0 = library default, 1 = per-thread copies, 2 = tensor-map gathers on dense pages")
    ap.add_argument("--replicas", type=int, default=0)
    ap.add_argument("--seqs", type=int, default=0,
                    help="sequences per batch (0 = the workload's own count); smaller batches serve "
                         "profiler captures of the same kernel")
    ap.add_argument("--graph-steps", type=int, default=256)
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--e2e-lanes", type=int, default=3, help="requests in flight (streams) for the e2e leg")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--component", choices=["latent_write", "select", "absorb"], default=None,
                    help="time one component of the path instead of the decode step (its own JSON line)")
    ap.add_argument("--rows", type=int, default=128, help="rows per call for --component latent_write / select")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per decode-kernel launch from an ncu capture of the current kernel")
    args = ap.parse_args()
    ws_n, rank, local = dist_info()

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, ws_n, rank)))
        return 0

    if not torch.cuda.is_available():
        print(json.dumps({"metric": METRIC, "error": "no CUDA device"}))
        return 1
    if args.component is not None:
        print(json.dumps({"latent_write": run_latent_write, "select": run_select,
                          "absorb": run_absorb}[args.component](args)))
        return 0
    init_dist(ws_n, "nccl")
    line = run_cuda(args, ws_n, rank, local)
    w0 = line.pop("_w0")
    if rank == 0:
        if not args.skip_cpu:
            line["cpu_baseline"] = cpu_baseline(w0, args.cpu_budget)
        print(json.dumps(line))
    if ws_n > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
