"""Benchmark of the paged MLA KV-cache gather on GB300.

Metric: effective gather GB/s = (entry bytes read + entry bytes written) per
call / device time, and its fraction of the measured HBM copy peak. A step is
one gather call (the whole hot path: plan, page mapping, block-table lookups,
data movement) over one batch of synthetic input.

Default workload: single-60K raw gather (1 request of 60,000 tokens, block
size 64, 576-element bf16 entries, 1024 shuffled blocks). Inputs are resident
in HBM. Consecutive steps rotate over several identical replicas of the inputs
whose combined footprint is more than four times the L2 cache, so no step
finds its data in L2 (no flush inside the timed region). A second, separate
measurement ("cold") flushes L2 by writing a 512 MB buffer before every call
and reports the median call time, the way the page measured its kernels.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--config 60k|tiny|300k|skew8|skew64_raw|skew64_dequant]
Under torchrun (N > 1) every rank runs its own replica of the workload (weak
scaling, no collective on the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import re
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_mla_kv_cache_gb300 import workloads as W  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
METRIC = "effective gather GB/s (read+write / device time) and % of GB300 HBM peak"
# committed ncu summary of the dominant kernel per workload
PROFILE_FILES = {
    "60k": "gather_bulk_single60k.md",
    "300k": "gather_bulk_single300k.md",
    "skew8": "gather_tma_convert_skew8.md",
    "skew64_raw": "gather_bulk_skew64_raw.md",
    "skew64_dequant": "gather_tma_convert_skew64_dequant.md",
}
KERNEL_SRC = os.path.join(ROOT, "paged_mla_kv_cache_gb300", "csrc", "pmg_gather.cu")


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(x: float, device) -> float:
    """Max over ranks of a per-rank float (the timed region's length); the
    tensor lives on `device` (cuda for NCCL, cpu for gloo)."""
    if not torch.distributed.is_initialized() or torch.distributed.get_world_size() == 1:
        return float(x)
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def weak_value(bytes_per_step: int, steps: int, max_ms: float, world: int) -> float:
    """Whole-job GB/s: every rank moved bytes_per_step per step; the job took the
    slowest rank's time."""
    return world * bytes_per_step * steps / (max_ms * 1e-3) / 1e9


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_code_hash(text: str) -> str:
    """sha256 of the kernel source with comments and blank lines removed, so a
    comment edit does not count as a kernel change."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    lines = [line.rstrip() for line in text.splitlines() if line.strip()]
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()


def profiled_traffic(config: str):
    """DRAM bytes per launch from the committed ncu summary of this workload, if
    it was taken on the current kernel code (else None)."""
    name = PROFILE_FILES.get(config)
    if name is None:
        return None
    try:
        text = open(os.path.join(ROOT, "profiles", name)).read()
    except OSError:
        return None
    m_sha = re.search(r"kernel_code_sha256:\s*([0-9a-f]{64})", text)
    m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    if not (m_sha and m_tr):
        return None
    sha = kernel_code_hash(open(KERNEL_SRC).read())
    return int(m_tr.group(1)) if sha == m_sha.group(1) else None


class ClockSampler:
    """nvidia-smi clock and throttle samples while the timed region runs."""

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.proc = None
        self.path = None
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index),
                 "--query-gpu=clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                 "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                 "clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", str(period_ms)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def workload_config(wl: W.Workload) -> dict:
    """The keys that name the workload, shared by both arms."""
    return {"workload": wl.name, "num_reqs": wl.num_reqs, "total_tokens": wl.total_tokens,
            "block_size": wl.block_size, "entry_size": wl.entry_size, "num_blocks": wl.num_blocks,
            "cache_dtype": wl.src_dtype, "out_dtype": wl.dst_dtype, "bytes_per_step": wl.algorithmic_bytes()}


def make_workload(name: str) -> W.Workload:
    return W.CONFIGS[name]()


class DeviceInputs:
    """One replica of a workload's inputs and output, resident on the device."""

    def __init__(self, wl: W.Workload, device):
        self.cache_full = wl.cache.to(device)
        self.cache = self.cache_full[:, :, :wl.entry_size]
        self.bt = wl.block_table.to(device)
        self.cu = wl.cu_seq_lens.to(device)
        self.ss = None if wl.seq_starts is None else wl.seq_starts.to(device)
        self.scale = torch.tensor([wl.scale], dtype=torch.float32, device=device)
        self.dst = torch.empty((wl.total_tokens, wl.entry_size), dtype=W.TORCH_DTYPES[wl.dst_dtype], device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)

    def nbytes(self):
        return self.cache_full.numel() * self.cache_full.element_size() + self.dst.numel() * self.dst.element_size()


def run_ours(args, wl: W.Workload, ws: int, rank: int, local: int):
    from paged_mla_kv_cache_gb300 import binding
    from paged_mla_kv_cache_gb300.build import build_library
    build_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    alg_bytes = wl.algorithmic_bytes()

    base = DeviceInputs(wl, dev)
    nrep = max(2, math.ceil(4 * L2_BYTES / base.nbytes()))
    reps = [base] + [DeviceInputs(wl, dev) for _ in range(nrep - 1)]

    # one scheduling workspace serves every call on this stream
    ws_buf = None if args.no_workspace else binding.new_workspace(dev)

    if args.entry == "tokens":
        # the per-token entry point: each output row names its request
        cu_h = wl.cu_seq_lens.numpy()
        t2s_h = np.full(wl.total_tokens, -1, np.int32)
        for r in range(wl.num_reqs):
            t2s_h[cu_h[r]:min(cu_h[r + 1], wl.total_tokens)] = r
        for r in reps:
            r.t2s = torch.from_numpy(t2s_h).to(dev)

    def step(k, strm=None, options=None):
        r = reps[k % nrep]
        opts = args.options if options is None else options
        if args.entry == "tokens":
            binding.gather_tokens(r.cache, r.dst, r.bt, r.t2s, r.cu, r.scale, r.err, num_reqs=wl.num_reqs,
                                  stream=stream if strm is None else strm, options=opts, workspace=ws_buf)
        else:
            binding.gather(r.cache, r.dst, r.bt, r.cu, r.ss, r.scale, r.err, num_reqs=wl.num_reqs,
                           stream=stream if strm is None else strm, options=opts, workspace=ws_buf)

    path, unit = binding.select_path(base.cache, base.dst, base.bt, base.cu, num_reqs=wl.num_reqs,
                                     options=args.options)
    if args.entry == "tokens":
        path = "per-token " + ("SIMT" if path != "bulk" else "bulk")
    for k in range(args.warmup):
        step(k)
    torch.cuda.synchronize(dev)

    # The timed steps are replayed from CUDA graphs of our launches so that the
    # host's per-call cost (argument marshalling, launch) stays off the clock.
    def capture(n, options=None):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cs = torch.cuda.current_stream()
            for k in range(n):
                step(k, cs, options)
        return g

    per_graph = min(args.steps, nrep * max(1, 120 // nrep))
    g_main = capture(per_graph)
    n_main, rem = divmod(args.steps, per_graph)
    g_rem = capture(rem) if rem else None
    g_main.replay()
    torch.cuda.synchronize(dev)
    if ws > 1:
        torch.distributed.barrier()

    # --- timed region: K steps -----------------------------------------------
    sampler = ClockSampler(local)
    time.sleep(0.15)  # let the sampler start
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    start.record(stream)
    for _ in range(n_main):
        g_main.replay()
    if g_rem is not None:
        g_rem.replay()
    end.record(stream)
    torch.cuda.synchronize(dev)
    if ws > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    ms = reduce_max(start.elapsed_time(end), dev)
    for r in reps:
        flag = int(r.err.item())
        if flag != 0:
            raise RuntimeError(f"gather reported data errors (flag {flag}) on valid inputs")

    ms_per_step = ms / args.steps
    value = weak_value(alg_bytes, args.steps, ms, ws)
    # the gather is the only kernel of a step: its average launch duration is
    # the timed region over the steps (inter-launch gaps included)
    per_launch_ms = ms_per_step

    # --- the same steps with the early-metadata promise (reported beside) -----
    early = None
    if not args.quick and args.entry == "gather" and not (args.options & 8):
        opts = args.options | 8
        n_e = min(args.steps, 3000)
        pg = min(n_e, per_graph)
        g_e = capture(pg, opts)
        g_e.replay()
        torch.cuda.synchronize(dev)
        reps_e = max(1, n_e // pg)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps_e):
            g_e.replay()
        b.record(stream)
        torch.cuda.synchronize(dev)
        ms_e = reduce_max(a.elapsed_time(b), dev)
        steps_e = reps_e * pg
        v_e = weak_value(alg_bytes, steps_e, ms_e, ws)
        peak_e, _ = measured_peak()
        early = {"value": round(v_e, 1), "unit": "GB/s", "frac": round(alg_bytes / (ms_e / steps_e * 1e-3) / 1e9 / peak_e, 4),
                 "per_launch_us": round(ms_e / steps_e * 1e3, 2), "steps": steps_e,
                 "options": "PMG_OPT_EARLY_METADATA (caller promises no running kernel writes the metadata)"}
        del g_e

    # --- cold: flush L2 (write 512 MB) before each call, median -------------
    cold = None
    if not args.quick:
        flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
        times = []
        for k in range(30):
            flush.fill_(k & 0xFF)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            step(k)
            b.record(stream)
            torch.cuda.synchronize(dev)
            times.append(a.elapsed_time(b))
        med = statistics.median(times)
        cold = {"median_us": round(med * 1e3, 2), "gbs": round(alg_bytes / (med * 1e-3) / 1e9, 1),
                "flush": "512 MB write before each call"}
        del flush

    # --- end to end: host buffers through the public binding -----------------
    e2e = None
    if not args.quick:
        e2e = run_e2e(wl, dev, stream, alg_bytes, steps=min(max(args.steps // 200, 5), 40), ws=ws)

    peak, peak_kind = measured_peak()
    achieved = alg_bytes / (per_launch_ms * 1e-3) / 1e9
    result = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if wl.src_dtype == wl.dst_dtype == "bf16" else f"{wl.src_dtype}->{wl.dst_dtype}",
        "data": "synthetic (seeded N(0,1) cache, seeded block-id permutation)",
        "config": {
            **workload_config(wl),
            "path": path if args.options == 0 else f"{path} (options {args.options})",
            "schedule": ("static" if args.no_workspace else "dynamic (workspace)")
                        + (", early metadata" if args.early_metadata else ""),
            "l2": f"{nrep} rotating input replicas ({sum(r.nbytes() for r in reps) / 1e6:.0f} MB) > 4x L2; no flush",
            "parallelism": f"replicas x{ws}",
        },
        "roofline": {
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": profiled_traffic(args.config),
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback",
            "per_launch_us": round(per_launch_ms * 1e3, 2),
        },
        "clocks": clocks,
        "gpu_launches": args.steps,
        "cold": cold,
        "early_metadata": early,
        "e2e": e2e,
    }
    return result


def run_e2e(wl, dev, stream, alg_bytes, steps, ws):
    """Same metric through the public binding with inputs and output in pinned
    host memory: every step copies its inputs host -> device, gathers, and
    copies the output device -> host."""
    from paged_mla_kv_cache_gb300 import binding
    h_cache = wl.cache.pin_memory()
    h_bt = wl.block_table.pin_memory()
    h_cu = wl.cu_seq_lens.pin_memory()
    h_ss = None if wl.seq_starts is None else wl.seq_starts.pin_memory()
    h_scale = torch.tensor([wl.scale], dtype=torch.float32).pin_memory()
    h_out = torch.empty((wl.total_tokens, wl.entry_size), dtype=W.TORCH_DTYPES[wl.dst_dtype]).pin_memory()
    d_cache = torch.empty_like(wl.cache, device=dev)
    d_bt = torch.empty_like(wl.block_table, device=dev)
    d_cu = torch.empty_like(wl.cu_seq_lens, device=dev)
    d_ss = None if h_ss is None else torch.empty_like(h_ss, device=dev)
    d_scale = torch.empty(1, dtype=torch.float32, device=dev)
    d_out = torch.empty(h_out.shape, dtype=h_out.dtype, device=dev)
    d_err = torch.zeros(1, dtype=torch.int32, device=dev)
    d_ws = binding.new_workspace(dev)
    h2d = sum(t.numel() * t.element_size() for t in (h_cache, h_bt, h_cu, h_scale) + ((h_ss,) if h_ss is not None else ()))
    d2h = h_out.numel() * h_out.element_size()

    def one():
        d_cache.copy_(h_cache, non_blocking=True)
        d_bt.copy_(h_bt, non_blocking=True)
        d_cu.copy_(h_cu, non_blocking=True)
        if d_ss is not None:
            d_ss.copy_(h_ss, non_blocking=True)
        d_scale.copy_(h_scale, non_blocking=True)
        binding.gather(d_cache[:, :, :wl.entry_size], d_out, d_bt, d_cu, d_ss, d_scale, d_err,
                       num_reqs=wl.num_reqs, stream=stream, workspace=d_ws)
        h_out.copy_(d_out, non_blocking=True)

    for _ in range(2):
        one()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        one()
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b) / steps
    return {"value": round(ws * alg_bytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 4), "steps": steps}


def oracle_sample(wl: W.Workload, rows: int):
    """A bounded sample of the workload for the CPU oracle: the first `rows`
    output rows of each request's share, as one smaller call of the same shape."""
    from oracle import gather as og
    cache = W.tensor_bits(wl.cache)
    cache_view = np.lib.stride_tricks.as_strided(
        cache, shape=(cache.shape[0], cache.shape[1], wl.entry_size), strides=cache.strides)
    frac = min(1.0, rows / max(wl.rows, 1))
    lens = [int(math.ceil(L * frac)) for L in wl.lens]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    dst = wl.new_dst(row_stride=None)[:T] if T <= wl.total_tokens else None
    bt = wl.block_table.numpy()
    ss = None if wl.seq_starts is None else wl.seq_starts.numpy()
    sample_bytes = T * wl.entry_size * (W.ELEM_BYTES[wl.src_dtype] + W.ELEM_BYTES[wl.dst_dtype])

    def run():
        return og.gather(cache_view, bt, cu, ss, wl.num_reqs, T, wl.block_size, wl.entry_size, wl.src_dtype,
                         wl.dst_dtype, wl.scale, dst)
    return run, sample_bytes, T


def cpu_baseline(wl: W.Workload, budget_s: float = 10.0):
    """The oracle as it stands, single-threaded on a host core, repeated over the
    full workload (or a prefix sample if one call would exceed the budget)."""
    run, nbytes, rows = oracle_sample(wl, wl.rows)
    t0 = time.perf_counter()
    run()
    t1 = time.perf_counter() - t0
    if t1 > budget_s / 3:
        run, nbytes, rows = oracle_sample(wl, int(wl.rows * budget_s / 3 / t1))
    n, t0 = 0, time.perf_counter()
    while True:
        run()
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (n >= 3 and el >= budget_s / 2 and el / n * (n + 1) > budget_s):
            break
    gbs = nbytes * n / el / 1e9
    return {"value": round(gbs, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} full oracle calls over {rows} of {wl.rows} rows in {el:.1f} s "
                      f"({platform.machine()}, single thread)"}


def run_reference(args, wl, ws, rank):
    """The reference arm: the CPU oracle timed on host cores, each step a bounded
    sample of the workload so that warmup + steps end within a few minutes."""
    if rank != 0:
        return None
    run_full, nbytes_full, _ = oracle_sample(wl, wl.rows)
    t0 = time.perf_counter()
    run_full()
    t_full = time.perf_counter() - t0
    budget = 90.0
    per_step = budget / max(args.steps + args.warmup, 1)
    rows = max(64, min(wl.rows, int(wl.rows * per_step / max(t_full, 1e-9))))
    run, nbytes, rows = oracle_sample(wl, rows)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    el = time.perf_counter() - t0
    value = nbytes * args.steps / el / 1e9
    sample = f"{rows} of {wl.rows} rows per step ({platform.machine()}, single thread)"
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.src_dtype, "data": "synthetic",
        "config": {**workload_config(wl), "path": "CPU oracle (per-token loop)"},
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="60k", choices=sorted(W.CONFIGS))
    ap.add_argument("--quick", action="store_true", help="skip the cold, e2e and CPU-baseline legs")
    ap.add_argument("--options", type=int, default=0, help="PMG_OPT_* bits passed to every call (path sweeps)")
    ap.add_argument("--early-metadata", action="store_true",
                    help="pass PMG_OPT_EARLY_METADATA (the caller's promise that no running kernel writes the "
                         "metadata): planning overlaps the previous call's tail")
    ap.add_argument("--entry", choices=["gather", "tokens"], default="gather",
                    help="gather: the page gather (default); tokens: the per-token indexed gather")
    ap.add_argument("--no-workspace", action="store_true",
                    help="static work split (no scheduling workspace) for comparison")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.early_metadata:
        args.options |= 8  # PMG_OPT_EARLY_METADATA
    ws, rank, local = dist_env()
    if ws > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if args.impl == "ours" else "gloo"
        torch.distributed.init_process_group(backend=backend, device_id=torch.device("cuda", local)
                                             if backend == "nccl" else None)
    wl = make_workload(args.config)
    if args.impl == "reference":
        res = run_reference(args, wl, ws, rank)
    else:
        res = run_ours(args, wl, ws, rank, local)
        if rank == 0 and not args.quick:
            res["cpu_baseline"] = cpu_baseline(wl)
        elif rank == 0:
            res["cpu_baseline"] = None
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
