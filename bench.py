#!/usr/bin/env python3
"""Benchmark of the DSA indexer candidate-selection path on GB300.

One step = one pass of the whole path (block scores, block top-k + pin, clamp,
live-span mask, row top-k) over one batch: the fused dsa_select_topk launch on
the 1M-context prefill chunk (2048 rows x 1,048,576 fp32 logits, 8 GiB, larger
than L2, so no flush is needed between steps).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line on rank 0.  Under torchrun each rank processes its own
replica batch (weak scaling, no data-path collective); timing is the max over
ranks.  `--impl reference` times the CPU oracle instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wk  # noqa: E402

KERNEL_SRC = os.path.join(ROOT, "sparse_attention_indexer_live_gb300", "csrc", "dsa_select.cu")
PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_NOTE = os.path.join(ROOT, "profiles", "select_topk_kernel_prefill_1m.md")
FALLBACK_HBM_GBS = 6800.0
METRIC = "indexer select rows/s at W=1,048,576 (1M-context prefill chunk)"


# ---------------------------------------------------------------------------
# multi-rank plumbing (host only; the data path has no collective)

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return world, rank, local


def dist_init(backend: str):
    import torch.distributed as dist
    world, rank, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return world, rank


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_rows(rank: int, rows: int) -> np.ndarray:
    """Row ids whose data rank `rank` generates: each rank gets its own rows of
    the same shape (weak scaling), bounds shared."""
    return np.arange(rows, dtype=np.int32) + rank * rows


# ---------------------------------------------------------------------------
# accounting

def row_bounds(wl, starts, ends):
    r = np.arange(wl.rows)
    q = r // wl.row_repeat
    e = ends[q].astype(np.int64) - (wl.row_repeat - 1) + (r % wl.row_repeat)
    s = np.maximum(starts[q].astype(np.int64), 0) if starts is not None else np.zeros(wl.rows,
                                                                                     np.int64)
    return s, e


def algorithmic_bytes(wl, starts, ends, cand) -> np.ndarray:
    """Per-row minimum bytes of the path: read the live span when the values
    matter (more live blocks than Kb), write -inf over every non-kept column of
    [0, min(end, W)), write cand and topk, read the bounds."""
    W, B, Kb, K = wl.width, wl.block_size, wl.block_topk, wl.row_topk
    s, e = row_bounds(wl, starts, ends)
    ec = np.minimum(e, W)
    L = np.maximum(ec - s, 0)
    nb = (L + B - 1) // B
    out = np.zeros(wl.rows, dtype=np.int64)
    for r in range(wl.rows):
        c = cand[r].astype(np.int64)
        c = c[c >= 0]
        inside = s[r] + c * B < W
        live = np.unique(c[inside & (c < nb[r])])
        kept = int(np.minimum(B, ec[r] - (s[r] + live * B)).sum()) if len(live) else 0
        edge = bool((~inside).any())
        if edge and s[r] <= W - 1 < ec[r] and ((W - 1 - s[r]) // B) not in set(live.tolist()):
            kept += 1
        writes = max(int(ec[r]), 0) - kept
        read = 4 * int(L[r]) if nb[r] > Kb else 0
        out[r] = read + 4 * writes + 4 * (Kb + 1) + 4 * K + 8
    return out


def hbm_peak():
    try:
        with open(PEAKS) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, STREAM-style copy)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, one earlier GB300 measurement)"


def kernel_source_hash() -> str:
    with open(KERNEL_SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def committed_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source; else None."""
    try:
        txt = open(TRAFFIC_NOTE).read()
    except OSError:
        return None
    vals = {}
    for line in txt.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256") != kernel_source_hash():
        return None
    try:
        return int(vals["traffic_bytes_per_full_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# clocks

class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.lines = []
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        for t, line in self.lines:
            p = [x.strip() for x in line.split(",")]
            if len(p) < 10:
                continue
            try:
                rows.append((t, float(p[2]), float(p[3]), p[6:10]))
            except ValueError:
                continue
        inside = [r for r in rows if self.t0 and self.t1 and self.t0 <= r[0] <= self.t1]
        window = "timed region"
        if not inside:
            inside, window = rows, "run (timed region shorter than the 100 ms sample period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "window": "no nvidia-smi samples"}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3])
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside), "window": window}


# ---------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)

def oracle_rows_per_s(wl, rows, starts, ends, threads):
    """Time the oracle on the given rows (one row per task, `threads` host
    threads; the oracle releases the GIL inside its C code)."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    orc = oracle.default()
    data = wk.make_rows(wl, rows, starts, ends)
    s, e = row_bounds(wl, starts, ends)

    def one(i):
        r = int(rows[i]) % wl.rows
        orc.row(data[i], wl.width, int(s[r]), int(e[r]), wl.block_size, wl.block_topk,
                wl.row_topk, col_stride=wl.col_stride)

    t0 = time.perf_counter()
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(one, range(len(rows))))
    dt = time.perf_counter() - t0
    return len(rows) / dt, dt


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args, wl):
    world, rank = dist_init("gloo")
    if rank != 0:
        return
    starts, ends = wk.bounds(wl)
    cores = host_cores()
    rng = np.random.default_rng(0)
    per_step = min(cores, wl.rows)
    for _ in range(args.warmup):
        oracle_rows_per_s(wl, rng.choice(wl.rows, per_step, replace=False), starts, ends, cores)
    times = []
    for _ in range(args.steps):
        rows = rng.choice(wl.rows, per_step, replace=False)
        _, dt = oracle_rows_per_s(wl, rows, starts, ends, cores)
        times.append(dt)
    total = sum(times)
    value = per_step * args.steps / total
    sample = (f"{per_step} random rows of the workload per step (one per host core), "
              f"whole path per row, oracle as written")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config_block(wl),
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": cores, "kind": "oracle",
                         "sample": sample, "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_block(wl):
    return {"workload": f"{wl.name}: {wl.rows} rows x {wl.width} fp32 logits, "
                        f"B={wl.block_size}, block top-k={wl.block_topk} + newest-block pin, "
                        f"row top-k={wl.row_topk}; {wl.note}",
            "rows": wl.rows, "width": wl.width, "block_size": wl.block_size,
            "block_topk": wl.block_topk, "row_topk": wl.row_topk,
            "l2": f"inputs ({wl.rows * wl.row_stride * 4 / 2**30:.2f} GiB) larger than the "
                  f"129 MB L2, and L2 flushed (256 MB write) before every timed launch",
            "input": "fresh logits every timed step: restored from a pristine device copy "
                     "outside the launch's CUDA-event pair"}

# ---------------------------------------------------------------------------
# supplementary measurements (not the bench metric): latency-bound shapes and
# the scan-mode row top-k

def _events(torch, n):
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def measure_decode_graph(dsa, torch, dev, local, prefill):
    """The 1M-width graph-captured decode: 96 rows, median end ~600; one CUDA
    graph replay per step, warm and with L2 flushed."""
    peak, _ = hbm_peak()
    wl = wk.WORKLOADS["decode_1m"]
    x, starts, ends = wk.make_all(wl)
    logits = torch.from_numpy(x).to(dev)
    del x
    ends_d = torch.from_numpy(ends).to(dev)
    cand = torch.empty((wl.rows, wl.block_topk + 1), dtype=torch.int32, device=dev)
    topk = torch.empty((wl.rows, wl.row_topk), dtype=torch.int32, device=dev)
    plan = dsa.dsa_select_init(device=local, rows=wl.rows, width=wl.width,
                               block_size=wl.block_size, block_topk=wl.block_topk,
                               row_topk=wl.row_topk, row_repeat=wl.row_repeat)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    dsa.dsa_select_topk(plan, logits, None, ends_d, cand, topk, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dsa.dsa_select_topk(plan, logits, None, ends_d, cand, topk, stream=s)
    for _ in range(20):
        g.replay()
    torch.cuda.synchronize()
    n = 500
    e0, e1 = _events(torch, 2)
    e0.record()
    for _ in range(n):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    warm_us = e0.elapsed_time(e1) * 1e3 / n
    flush = torch.empty(64 << 20, dtype=torch.float32, device=dev)  # 256 MB > L2
    ev = _events(torch, 2 * 50)
    for i in range(50):
        flush.fill_(float(i))
        ev[2 * i].record()
        g.replay()
        ev[2 * i + 1].record()
    torch.cuda.synchronize()
    cold = [ev[2 * i].elapsed_time(ev[2 * i + 1]) * 1e3 for i in range(50)]
    # the two-call form (dsa_candidate_select, then the candidate-mode row
    # top-k) captured in one graph, warm
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=s):
        dsa.dsa_candidate_select(plan, logits, None, ends_d, cand, stream=s)
        dsa.dsa_row_topk(plan, logits, None, ends_d, cand, topk, stream=s)
    for _ in range(20):
        g2.replay()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(n):
        g2.replay()
    e1.record()
    torch.cuda.synchronize()
    two_us = e0.elapsed_time(e1) * 1e3 / n
    alg = int(algorithmic_bytes(wl, starts, ends, cand.cpu().numpy()).sum())
    full = wl.rows * wl.width * 4
    return {"rows": wl.rows, "us_per_replay_warm": warm_us,
            "us_per_replay_l2_flushed": statistics.median(cold),
            "us_per_replay_l2_flushed_min": min(cold),
            "us_per_replay_warm_two_calls": two_us,
            "algorithmic_bytes": alg, "achieved_gbs_warm": alg / (warm_us * 1e-6) / 1e9,
            "full_width_mask_bytes": full, "full_width_us_at_peak": full / (peak * 1e9) * 1e6,
            "ctas": plan.describe()["grid_select"]}


def measure_single_row(dsa, torch, dev, local, prefill):
    """One full 1M-column row (the pages' single-long-row case), fresh input
    every call."""
    wl1 = wk.WORKLOADS["prefill_1m"].with_(rows=1)
    x1 = wk.make_rows(wl1, [0], None, np.array([wl1.width], dtype=np.int32))
    l1 = torch.from_numpy(x1).to(dev)
    pristine = l1.clone()
    e1d = torch.tensor([wl1.width], dtype=torch.int32, device=dev)
    c1 = torch.empty((1, wl1.block_topk + 1), dtype=torch.int32, device=dev)
    t1 = torch.empty((1, wl1.row_topk), dtype=torch.int32, device=dev)
    p1 = dsa.dsa_select_init(device=local, rows=1, width=wl1.width, block_size=wl1.block_size,
                             block_topk=wl1.block_topk, row_topk=wl1.row_topk)
    for _ in range(3):
        l1.copy_(pristine)
        dsa.dsa_select_topk(p1, l1, None, e1d, c1, t1)
    ev = _events(torch, 40)
    for i in range(20):
        l1.copy_(pristine)
        ev[2 * i].record()
        dsa.dsa_select_topk(p1, l1, None, e1d, c1, t1)
        ev[2 * i + 1].record()
    torch.cuda.synchronize()
    us = statistics.median(ev[2 * i].elapsed_time(ev[2 * i + 1]) * 1e3 for i in range(20))
    a1 = int(algorithmic_bytes(wl1, None, np.array([wl1.width], dtype=np.int32),
                               c1.cpu().numpy()).sum())
    return {"us_per_call": us, "achieved_gbs": a1 / (us * 1e-6) / 1e9,
            "ctas": p1.describe()["grid_select"], "input": "fresh row every call"}


def measure_scan(dsa, torch, dev, local, prefill):
    """Scan-mode row top-k over the (masked) prefill logits."""
    wlp, plan_p, logits_p, ends_p, topk_p = prefill
    out_t = torch.empty_like(topk_p)
    dsa.dsa_row_topk(plan_p, logits_p, None, ends_p, None, out_t)
    e0, e1 = _events(torch, 2)
    e0.record()
    for _ in range(3):
        dsa.dsa_row_topk(plan_p, logits_p, None, ends_p, None, out_t)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / 3
    _, e = row_bounds(wlp, None, ends_p.cpu().numpy())
    L = np.minimum(e, wlp.width)
    scan_alg = int((4 * L + 4 * wlp.row_topk + 8).sum())
    peak, _ = hbm_peak()
    return {"ms_per_launch": ms, "rows_per_s": wlp.rows / (ms / 1e3),
            "achieved_gbs": scan_alg / (ms / 1e3) / 1e9,
            "frac": scan_alg / (ms / 1e3) / 1e9 / peak,
            "matches_fused": bool(torch.equal(out_t, topk_p))}


def measure_combine(dsa, torch, dev, local, prefill):
    """Top-k / sliding-window combine on the prefill chunk's top-k (20 launches
    in one CUDA graph)."""
    wlp, plan_p, logits_p, ends_p, topk_p = prefill
    window = 128
    comb = torch.empty((wlp.rows, wlp.row_topk + window), dtype=torch.int32, device=dev)
    us = _graph_timed(torch, lambda: dsa.dsa_combine_window(plan_p, None, ends_p, topk_p, window, comb))
    comb_alg = wlp.rows * (4 * wlp.row_topk + 4 * (wlp.row_topk + window) + 8)
    peak, _ = hbm_peak()
    return {"window": window, "us_per_launch": us, "achieved_gbs": comb_alg / (us * 1e-6) / 1e9,
            "frac": comb_alg / (us * 1e-6) / 1e9 / peak}


# supplementary measurements (not the bench metric), by name
EXTRAS = {
    "decode_1m_graph": measure_decode_graph,
    "single_row_1m": measure_single_row,
    "scan_topk_prefill_1m": measure_scan,
    "combine_window_prefill_1m": measure_combine,
    "indexer_producer": lambda dsa, torch, dev, local, prefill: measure_producer(dsa, torch, dev),
    "indexer_select_fused": lambda dsa, torch, dev, local, prefill: measure_fused(dsa, torch, dev),
    "indexer_select_fused_96x1m": lambda dsa, torch, dev, local, prefill: measure_fused(
        dsa, torch, dev, T=96, S=1 << 20),
    "grouped_sparse_attention": lambda dsa, torch, dev, local, prefill: measure_attention(
        dsa, torch, dev),
    "grouped_sparse_attention_ranges": lambda dsa, torch, dev, local, prefill: measure_attention_ranges(
        dsa, torch, dev),
}


def measure_extras(dsa, torch, dev, local, prefill, names=None):
    return {name: fn(dsa, torch, dev, local, prefill) for name, fn in EXTRAS.items()
            if names is None or name in names}


def fp8_peak_tflops():
    """Measured bf16 burst (MEASURED_PEAKS.json) x the nominal fp8 / bf16
    dense ratio of 2 (4.5 / 2.25 PFLOP/s); fallback 1.9 PFLOP/s bf16."""
    try:
        with open(PEAKS) as f:
            return 2.0 * float(json.load(f)["bf16_tflops"]), "2 x measured bf16 burst"
    except Exception:
        return 2.0 * 1900.0, "2 x fallback bf16 (1.9 PFLOP/s)"


def measure_producer(dsa, torch, dev, T=608, S=131072):
    """FP8 indexer logits on the tensor cores (causal spans)."""
    q, k, ks, w, _, ends = wk.indexer_inputs(T, S, seed=11)
    qd, kd = torch.from_numpy(q).to(dev), torch.from_numpy(k).to(dev)
    ksd, wd = torch.from_numpy(ks).to(dev), torch.from_numpy(w).to(dev)
    en = torch.from_numpy(ends).to(dev)
    out = torch.empty((T, S), dtype=torch.float32, device=dev)
    for _ in range(3):
        dsa.dsa_indexer_logits(qd, kd, ksd, wd, None, en, out)
    e0, e1 = _events(torch, 2)
    e0.record()
    for _ in range(10):
        dsa.dsa_indexer_logits(qd, kd, ksd, wd, None, en, out)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / 10
    pairs = int(np.minimum(ends, S).astype(np.int64).sum())
    flops = 2.0 * pairs * 64 * 128
    peak, src = fp8_peak_tflops()
    tf = flops / (ms / 1e3) / 1e12
    return {"queries": T, "keys": S, "ms_per_launch": ms, "tflops": tf, "peak_tflops": peak,
            "frac": tf / peak, "peak_source": src, "status": dsa.dsa_indexer_status()}


def measure_fused(dsa, torch, dev, T=608, S=131072, B=8, Kb=256, K=2048):
    """The producer fused with the selection (dsa_indexer_select) against the
    two-step path (dsa_indexer_logits, then dsa_select_topk) on the same causal
    queries; both give the same cand / topk."""
    q, k, ks, w, _, ends = wk.indexer_inputs(T, S, seed=11)
    qd, kd = torch.from_numpy(q).to(dev), torch.from_numpy(k).to(dev)
    ksd, wd = torch.from_numpy(ks).to(dev), torch.from_numpy(w).to(dev)
    en = torch.from_numpy(ends).to(dev)
    plan = dsa.dsa_select_init(rows=T, width=S, block_size=B, block_topk=Kb, row_topk=K)
    logits = torch.empty((T, S), dtype=torch.float32, device=dev)
    cand2 = torch.empty((T, Kb + 1), dtype=torch.int32, device=dev)
    topk2 = torch.empty((T, K), dtype=torch.int32, device=dev)
    ws_bytes = dsa.dsa_indexer_select_workspace(plan)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    cand = torch.empty((T, Kb + 1), dtype=torch.int32, device=dev)
    topk = torch.empty((T, K), dtype=torch.int32, device=dev)

    def two_step():
        dsa.dsa_indexer_logits(qd, kd, ksd, wd, None, en, logits)
        dsa.dsa_select_topk(plan, logits, None, en, cand2, topk2)

    def fused():
        dsa.dsa_indexer_select(plan, qd, kd, ksd, wd, en, ws, cand, topk)

    res = {"queries": T, "keys": S, "block_size": B, "block_topk": Kb, "row_topk": K}
    for name, fn in (("two_step", two_step), ("fused", fused)):
        for _ in range(3):
            fn()
        e0, e1 = _events(torch, 2)
        e0.record()
        for _ in range(10):
            fn()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / 10
        res[name] = {"us_per_call": us, "rows_per_s": T / (us * 1e-6)}
    res["fused_workspace_bytes"] = int(ws_bytes)
    res["two_step_logits_bytes"] = int(T * S * 4)
    res["same_result"] = bool(torch.equal(cand, cand2) and torch.equal(topk, topk2))
    res["status"] = dsa.dsa_indexer_status()
    return res


def _graph_timed(torch, f, reps=20):
    """us per call of f, with reps calls captured in one CUDA graph: the replay
    times the kernels, not the host's launch rate."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            f()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(reps):
            f()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = _events(torch, 2)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / reps


def measure_attention_ranges(dsa, torch, dev, T=2048, H=8, Sr=1 << 20, blk=128, window=512):
    """The range form of the grouped attention (dsa_sparse_attention_ranges)
    on a compressed-prefix-plus-window selection: keys [0, Sc) hold one
    compressed entry per `blk` positions, keys [Sc, Sc + Sr) the raw
    positions; the T tokens are the last T positions of the context, and
    token t at position p attends to the compressed entries [0, (p + 1) / blk)
    and the raw window [p - window + 1, p] -- two ranges, no index lists."""
    Sc = Sr // blk
    S = Sc + Sr
    q, k, v, _ = wk.attention_inputs(T, H, S, 8, seed=22, G=128 // H)
    pos = Sr - T + np.arange(T)
    ranges = np.zeros((T, 2, 2), dtype=np.int32)
    ranges[:, 0, 1] = (pos + 1) // blk
    ranges[:, 1, 0] = Sc + np.maximum(0, pos - window + 1)
    ranges[:, 1, 1] = Sc + pos + 1
    select = Sc + window
    qd, kd, vd = (torch.from_numpy(x.view(np.int16)).to(dev) for x in (q, k, v))
    rd = torch.from_numpy(ranges).to(dev)
    cfg = dsa.ranges_attention_cfg(qd, kd, rd, select)
    ws = torch.zeros(dsa.dsa_sparse_attention_ranges_workspace(cfg, 2), dtype=torch.uint8, device=dev)
    o = torch.empty((T, H, 128), dtype=torch.float32, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    scale = 1.0 / math.sqrt(128)
    us_union = _graph_timed(torch, lambda: dsa.dsa_group_union_ranges(cfg, rd, ws))
    us = _graph_timed(torch, lambda: dsa.dsa_sparse_attention_ranges(cfg, qd, kd, vd, rd, scale, ws, o, lse))
    G = 128 // H
    groups = -(-T // G)
    cap = G * select
    rec = 16 + 2 * ((cap * 4 + 15) & ~15)
    wsn = ws.cpu().numpy()
    union = np.array([int(wsn[g * rec:g * rec + 4].view(np.int32)[0]) for g in range(groups)])
    sel = (ranges[:, :, 1] - ranges[:, :, 0]).sum(axis=1)
    u_tot = float(union.sum())
    union_bytes = 16.0 * T + groups * 16 + 8.0 * u_tot
    attn_bytes = 4.0 + 8.0 * u_tot + T * H * 128 * 2 + 2 * 256 * u_tot + T * H * (128 * 4 + 4)
    hbm, hbm_src = hbm_peak()
    useful = 2.0 * H * float(sel.sum()) * (128 + 128)
    us_attn = us - us_union
    return {"tokens": T, "heads": H, "group": G, "keys": S, "compressed": Sc, "window": window,
            "ranges_per_token": 2, "us_per_call": us, "us_union": us_union, "us_attention": us_attn,
            "tokens_per_s": T / (us * 1e-6), "union_over_selection": float(union.mean() / sel.mean()),
            "roofline": {"bound": "hbm", "unit": "GB/s", "peak": hbm, "peak_source": hbm_src,
                         "bytes_per_call": union_bytes + attn_bytes,
                         "achieved": (union_bytes + attn_bytes) / (us * 1e-6) / 1e9,
                         "frac": (union_bytes + attn_bytes) / (us * 1e-6) / 1e9 / hbm,
                         "attention_kernel_frac": attn_bytes / (us_attn * 1e-6) / 1e9 / hbm},
            "useful_tflops": useful / (us * 1e-6) / 1e12, "status": dsa.dsa_sparse_attention_status()}


def measure_attention(dsa, torch, dev, T=2048, H=8, S=1 << 20, Kc=2048, own=0.05):
    """Grouped masked sparse attention (dsa_sparse_attention): union build plus
    attention, on T tokens whose neighbours share most of their selection.

    The path is bound by HBM: every union position's key and value rows
    (2 x 256 bytes) are gathered once per group.  Algorithmic bytes: the
    union reads the selections and writes each group's record (count, keys,
    masks); the attention reads the records, Q and the gathered rows and
    writes o and lse."""
    q, k, v, idx = wk.attention_inputs(T, H, S, Kc, seed=21, own=own, G=128 // H)
    qd, kd, vd = (torch.from_numpy(x.view(np.int16)).to(dev) for x in (q, k, v))
    idd = torch.from_numpy(idx).to(dev)
    cfg = dsa.attention_cfg(qd, kd, idd)
    ws = torch.zeros(dsa.dsa_sparse_attention_workspace(cfg), dtype=torch.uint8, device=dev)
    o = torch.empty((T, H, 128), dtype=torch.float32, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    scale = 1.0 / math.sqrt(128)

    timed = lambda f: _graph_timed(torch, f)
    us_union = timed(lambda: dsa.dsa_group_union(cfg, idd, ws))
    us = timed(lambda: dsa.dsa_sparse_attention(cfg, qd, kd, vd, idd, scale, ws, o, lse))
    G = 128 // H
    groups = -(-T // G)
    cap = G * Kc
    rec = 16 + 2 * ((cap * 4 + 15) & ~15)
    wsn = ws.cpu().numpy()
    union = np.array([int(wsn[g * rec:g * rec + 4].view(np.int32)[0]) for g in range(groups)])
    sel = (idx >= 0).sum(axis=1)
    useful = 2.0 * H * float(sel.sum()) * (128 + 128)
    tiles = np.ceil(union / 128.0)
    executed = 2.0 * 128 * float((tiles * 128).sum()) * (128 + 128)
    u_tot = float(union.sum())
    union_bytes = 4.0 * T * Kc + groups * 16 + 8.0 * u_tot
    attn_bytes = 4.0 + 8.0 * u_tot + T * H * 128 * 2 + 2 * 256 * u_tot + T * H * (128 * 4 + 4)
    hbm, hbm_src = hbm_peak()
    peak = None
    try:
        with open(PEAKS) as f:
            peak = float(json.load(f)["bf16_tflops"])
    except Exception:
        peak = 1900.0
    us_attn = us - us_union
    return {"tokens": T, "heads": H, "group": G, "keys": S, "select": Kc, "neighbour_own_fraction": own,
            "us_per_call": us, "us_union": us_union, "us_attention": us_attn,
            "tokens_per_s": T / (us * 1e-6),
            "union_over_selection": float(union.mean() / sel.mean()),
            "roofline": {"bound": "hbm", "unit": "GB/s", "peak": hbm, "peak_source": hbm_src,
                         "bytes_per_call": union_bytes + attn_bytes,
                         "achieved": (union_bytes + attn_bytes) / (us * 1e-6) / 1e9,
                         "frac": (union_bytes + attn_bytes) / (us * 1e-6) / 1e9 / hbm,
                         "attention_kernel_frac": attn_bytes / (us_attn * 1e-6) / 1e9 / hbm,
                         "union_kernel_frac": union_bytes / (us_union * 1e-6) / 1e9 / hbm},
            "useful_tflops": useful / (us * 1e-6) / 1e12, "executed_tflops": executed / (us * 1e-6) / 1e12,
            "bf16_peak_tflops": peak, "status": dsa.dsa_sparse_attention_status()}


# ---------------------------------------------------------------------------
# our arm

def run_ours(args, wl):
    import torch

    import sparse_attention_indexer_live_gb300 as dsa
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist_init("nccl")
    dev = torch.device("cuda", local)
    dsa.build()
    dsa.load()

    starts, ends = wk.bounds(wl)
    rows = replica_rows(rank, wl.rows)
    host = torch.empty((wl.rows, wl.row_stride), dtype=torch.float32, pin_memory=True)
    wk.fill_rows(wl, rows, host.numpy(), starts, ends, bound_rows=np.arange(wl.rows))
    logits = host.to(dev)
    ends_h = torch.from_numpy(ends).pin_memory()
    ends_d = ends_h.to(dev)
    starts_d = None
    cand = torch.empty((wl.rows, wl.block_topk + 1), dtype=torch.int32, device=dev)
    topk = torch.empty((wl.rows, wl.row_topk), dtype=torch.int32, device=dev)
    plan = dsa.dsa_select_init(device=local, rows=wl.rows, width=wl.width,
                               block_size=wl.block_size, block_topk=wl.block_topk,
                               row_topk=wl.row_topk, row_repeat=wl.row_repeat)
    stream = torch.cuda.current_stream()

    def step():
        dsa.dsa_select_topk(plan, logits, starts_d, ends_d, cand, topk, stream=stream)

    visible = os.environ.get("CUDA_VISIBLE_DEVICES")
    clocks = ClockSampler(visible.split(",")[local].strip() if visible else str(local))
    clocks.start()
    # Every timed launch sees fresh logits, as every real prefill or decode step
    # does: before each launch the buffer is restored from a pristine device
    # copy and L2 is flushed (a 256 MB write), both outside the launch's event
    # pair, so the launch starts cold on unmasked input.
    pristine = logits.clone()
    flush = torch.empty(64 << 20, dtype=torch.float32, device=dev)

    def restore():
        logits.copy_(pristine)
        flush.zero_()

    first = torch.cuda.Event(enable_timing=True)
    first_end = torch.cuda.Event(enable_timing=True)
    restore()
    first.record(stream)
    step()
    first_end.record(stream)
    torch.cuda.synchronize()
    first_ms = first.elapsed_time(first_end)
    cand_h = cand.cpu().numpy()
    for _ in range(max(args.warmup - 1, 0)):
        restore()
        step()
    torch.cuda.synchronize()

    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    clocks.mark("t0")
    for i in range(args.steps):
        restore()
        ev0[i].record(stream)
        step()
        ev1[i].record(stream)
    torch.cuda.synchronize()
    clocks.mark("t1")
    barrier()
    launch_ms = [ev0[i].elapsed_time(ev1[i]) for i in range(args.steps)]
    total_ms = max_over_ranks(sum(launch_ms), dev)
    clocks.stop()
    # the same launch repeated on the buffer it has already masked (the path
    # leaves it unchanged): a secondary figure, not the headline
    reps = min(args.steps, 50)
    m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step()
    m0.record(stream)
    for _ in range(reps):
        step()
    m1.record(stream)
    torch.cuda.synchronize()
    masked_ms = m0.elapsed_time(m1) / reps
    del pristine, flush

    # end to end through the public API: pinned host logits -> device, the
    # fused call, cand + topk -> pinned host, every step.  The rows go in
    # chunks: the copy of chunk c + 1 (a second stream) overlaps the call on
    # chunk c, and each chunk's outputs go back as soon as its call is done.
    e2e = None
    if args.e2e_steps > 0:
        cand_ref, topk_ref = cand.clone(), topk.clone()
        cand_out = torch.empty(cand.shape, dtype=torch.int32, pin_memory=True)
        topk_out = torch.empty(topk.shape, dtype=torch.int32, pin_memory=True)
        rep = wl.row_repeat
        chunks = max(1, min(args.e2e_chunks, wl.rows // rep))
        per = -(-(wl.rows // rep) // chunks) * rep
        pieces = []
        for r0 in range(0, wl.rows, per):
            r1 = min(r0 + per, wl.rows)
            pl = dsa.dsa_select_init(device=local, rows=r1 - r0, width=wl.width,
                                     block_size=wl.block_size, block_topk=wl.block_topk,
                                     row_topk=wl.row_topk, row_repeat=rep)
            pieces.append((r0, r1, pl, torch.cuda.Event()))
        copier = torch.cuda.Stream()

        def e2e_step():
            copier.wait_stream(stream)  # the previous step's calls are done with the rows
            for r0, r1, pl, ev in pieces:
                with torch.cuda.stream(copier):
                    logits[r0:r1].copy_(host[r0:r1], non_blocking=True)
                    ends_d[r0 // rep:-(-r1 // rep)].copy_(ends_h[r0 // rep:-(-r1 // rep)],
                                                          non_blocking=True)
                    ev.record(copier)
                stream.wait_event(ev)
                dsa.dsa_select_topk(pl, logits[r0:r1], None, ends_d[r0 // rep:-(-r1 // rep)],
                                    cand[r0:r1], topk[r0:r1], stream=stream)
                cand_out[r0:r1].copy_(cand[r0:r1], non_blocking=True)
                topk_out[r0:r1].copy_(topk[r0:r1], non_blocking=True)

        e2e_step()  # warm-up (plans, copies)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), dev)
        h2d = host.numel() * 4 + ends_h.numel() * 4
        d2h = cand_out.numel() * 4 + topk_out.numel() * 4
        same = bool(torch.equal(cand_out, cand_ref.cpu()) and torch.equal(topk_out, topk_ref.cpu()))
        e2e = {"value": wl.rows * world * args.e2e_steps / (e2e_ms / 1e3), "unit": "rows/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e2e_ms / args.e2e_steps, "steps": args.e2e_steps,
               "chunks": len(pieces), "matches_single_call": same}

    if rank != 0:
        return
    alg = algorithmic_bytes(wl, starts, ends, cand_h)
    alg_launch = int(alg.sum())
    avg_launch_s = statistics.mean(launch_ms) / 1e3
    peak, peak_src = hbm_peak()
    achieved = alg_launch / avg_launch_s / 1e9
    traffic = committed_traffic()
    value = wl.rows * world * args.steps / (total_ms / 1e3)
    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded Philox4x32-10 N(0,1) logits with 64 planted +6 sigma "
                "spikes per row)",
        "config": config_block(wl),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "select_kernel<true> (fused dsa_select_topk)",
                     "algorithmic_bytes_per_launch": alg_launch, "peak_source": peak_src,
                     "avg_launch_ms": avg_launch_s * 1e3,
                     "min_launch_ms": min(launch_ms), "max_launch_ms": max(launch_ms),
                     "first_pass_ms": first_ms,
                     "input": "fresh (unmasked) logits for every timed launch, L2 flushed",
                     "masked_input_ms": masked_ms},
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clocks.summary(),
    }
    if args.extras:
        line["extras"] = measure_extras(dsa, torch, dev, local,
                                        (wl, plan, logits, ends_d, topk), args.extra)
    if args.cpu_rows > 0:
        cores = host_cores()
        rng = np.random.default_rng(1)
        sample = rng.choice(wl.rows, min(args.cpu_rows, wl.rows), replace=False)
        v, dt = oracle_rows_per_s(wl, sample, starts, ends, cores)
        one = sample[:max(1, min(16, len(sample)))]
        v1, dt1 = oracle_rows_per_s(wl, one, starts, ends, 1)
        line["cpu_baseline"] = {"value": v, "unit": "rows/s", "cores": min(cores, len(sample)),
                                "kind": "oracle",
                                "sample": f"{len(sample)} random rows of the workload, whole "
                                          f"path per row, rows in parallel over the host "
                                          f"cores, {dt:.1f} s wall",
                                "single_thread": {"value": v1, "unit": "rows/s", "cores": 1,
                                                  "sample": f"{len(one)} of those rows on one "
                                                            f"thread, {dt1:.1f} s wall"},
                                "cpu_model": cpu_model()}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="prefill_1m", choices=sorted(wk.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--e2e-chunks", type=int, default=8,
                    help="row chunks of the end-to-end step (copy of one overlaps the call on another)")
    ap.add_argument("--producer-only", nargs=2, type=int, metavar=("QUERIES", "KEYS"),
                    help="time only the tensor-core indexer-logits producer and print its JSON")
    ap.add_argument("--fused-only", nargs=2, type=int, metavar=("QUERIES", "KEYS"),
                    help="time only the fused producer + selection against the two-step path")
    ap.add_argument("--attention-only", action="store_true",
                    help="time only the grouped masked sparse attention and print its JSON")
    ap.add_argument("--attention-ranges-only", action="store_true",
                    help="time only the range form of the grouped attention and print its JSON")
    ap.add_argument("--no-extras", dest="extras", action="store_false",
                    help="skip the supplementary decode / single-row / scan-mode timings")
    ap.add_argument("--extra", action="append", choices=sorted(EXTRAS),
                    help="run only the named supplementary timing (repeatable)")
    ap.add_argument("--rows", type=int, default=None,
                    help="override the workload's row count (smaller profiling cases)")
    ap.add_argument("--cpu-rows", type=int, default=384,
                    help="rows of the oracle CPU baseline sample (0 = skip)")
    args = ap.parse_args()
    if args.warmup < 1:
        ap.error("--warmup must be >= 1")
    if args.attention_only:
        import torch

        import sparse_attention_indexer_live_gb300 as dsa
        dsa.build()
        dsa.load()
        print(json.dumps(measure_attention(dsa, torch, torch.device("cuda:0"))), flush=True)
        return
    if args.attention_ranges_only:
        import torch

        import sparse_attention_indexer_live_gb300 as dsa
        dsa.build()
        dsa.load()
        print(json.dumps(measure_attention_ranges(dsa, torch, torch.device("cuda:0"))), flush=True)
        return
    if args.producer_only or args.fused_only:
        import torch

        import sparse_attention_indexer_live_gb300 as dsa
        dsa.build()
        dsa.load()
        fn, (T, S) = ((measure_producer, args.producer_only) if args.producer_only
                      else (measure_fused, args.fused_only))
        print(json.dumps(fn(dsa, torch, torch.device("cuda:0"), T=T, S=S)), flush=True)
        return
    wl = wk.WORKLOADS[args.workload]
    if args.rows is not None:
        wl = wl.with_(rows=args.rows)
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
