"""Benchmark of the paged MLA KV-cache gather on GB300.

Metric: effective gather GB/s = (entry bytes read + entry bytes written) per
call / device time, and its fraction of the measured HBM copy peak. A step is
one gather call (the whole hot path: plan, page mapping, block-table lookups,
data movement) over one batch of synthetic input.

Headline workload: single-300K raw gather (1 request of 300,000 tokens, block
size 64, 576-element bf16 entries, 5000 shuffled blocks), the largest of the
named single-GPU workloads. Inputs are resident in HBM. Consecutive steps
rotate over identical replicas of the inputs whose combined footprint is more
than four times the L2 cache, so no step finds its data in L2 (no flush inside
the timed region). The K timed steps are replayed from CUDA graphs; the region
of exactly K steps is timed several times (so that the clock sampler sees the
GPU under load even for small K) and the median region gives the line's value.

Beside the headline the line carries:
  per_config  every named target workload (single-60K, single-300K, skew-8,
              skew-64 raw and dequant, and a 1M-token fp32 copy whose output
              offsets pass 2^31 bytes): steady-state GB/s and fraction of
              peak, per-launch time, and two "cold" medians with L2 flushed
              before every call, the page's cold-cache way of timing its
              kernels: "cold" writes a 512 MB buffer, "cold_clean" also reads
              it back (so L2 holds clean lines of another buffer).
  e2e         the same metric through the public binding with pinned host
              buffers, host<->device copies inside the timed region.
  cpu_baseline  the CPU oracle on the host cores (single thread, and all cores
              as concurrent oracle calls over disjoint row ranges).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--config 300k|60k|tiny|skew8|skew64_raw|skew64_dequant|fp32_1m]
Under torchrun (N > 1) every rank runs its own replica of the workload (weak
scaling, no collective on the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import concurrent.futures
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
HEADLINE = "300k"
PER_CONFIG = ["60k", "300k", "skew8", "skew64_raw", "skew64_dequant", "fp32_1m"]
# Committed ncu captures of the dominant kernel per workload: DRAM bytes over
# several consecutive launches of the timed step, divided by the launch count.
PROFILE_FILES = {
    "60k": "gather_bulk_single60k.md",
    "300k": "gather_bulk_single300k.md",
    "skew8": "gather_tma_convert_skew8.md",
    "skew64_raw": "gather_bulk_skew64_raw.md",
    "skew64_dequant": "gather_tma_convert_skew64_dequant.md",
    "fp32_1m": "gather_bulk_fp32_1m.md",
    # the per-token entry point (--entry tokens) on the same kernels in token mode
    "tokens_skew8": "gather_tma_convert_tokens_skew8.md",
    "tokens_60k": "gather_bulk_tokens_single60k.md",
}
KERNEL_SRC = os.path.join(ROOT, "paged_mla_kv_cache_gb300", "csrc", "pmg_gather.cu")
# how L2 is kept out of the steady-state figure; one statement for both arms
L2_POLICY = ("each GPU step reads and writes inputs/outputs not touched by the previous steps "
             "(rotating replicas, >= 4x L2 in all), no flush in the timed region; the cold figures flush "
             "L2 before every call")


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
    """DRAM read and write bytes per launch from the committed ncu capture of
    this workload (consecutive launches of the timed step), if it was taken on
    the current kernel code; else None. This is a stored capture, not a
    measurement of this run: the line labels it so."""
    name = PROFILE_FILES.get(config)
    if name is None:
        return None
    try:
        text = open(os.path.join(ROOT, "profiles", name)).read()
    except OSError:
        return None
    m_sha = re.search(r"kernel_code_sha256:\s*([0-9a-f]{64})", text)
    m_rd = re.search(r"dram_read_bytes_per_launch:\s*([0-9]+)", text)
    m_wr = re.search(r"dram_write_bytes_per_launch:\s*([0-9]+)", text)
    m_n = re.search(r"launches_captured:\s*([0-9]+)", text)
    if not (m_sha and m_rd and m_wr):
        return None
    if kernel_code_hash(open(KERNEL_SRC).read()) != m_sha.group(1):
        return None
    return {"read": int(m_rd.group(1)), "write": int(m_wr.group(1)),
            "source": f"committed ncu capture profiles/{name}: dram__bytes_read.sum and dram__bytes_write.sum "
                      f"over {m_n.group(1) if m_n else 'several'} consecutive launches of the timed step, "
                      f"per launch (same kernel code hash)"}


def cpu_facts():
    """Host core count and CPU model of the machine the oracle runs on."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if model is None:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith(("model name", "cpu part")):
                    model = line.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    return {"nproc": os.cpu_count(), "cpu_model": model or "unknown", "machine": platform.machine()}


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
                 "clocks_event_reasons.sw_power_cap,utilization.gpu",
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
        sm, mx, busy, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                f_sm, f_mx = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            sm.append(f_sm)
            mx.append(f_mx)
            try:
                busy.append(float(parts[7]) > 0)
            except ValueError:
                busy.append(False)
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        loaded = [s for s, b in zip(sm, busy) if b]
        return {"sm_mhz": statistics.median(loaded or sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm), "samples_under_load": len(loaded),
                "period_ms": 50}


def workload_config(wl: W.Workload) -> dict:
    """The keys that name the workload; both arms print exactly this dict."""
    return {"workload": wl.name, "num_reqs": wl.num_reqs, "total_tokens": wl.total_tokens,
            "block_size": wl.block_size, "entry_size": wl.entry_size, "num_blocks": wl.num_blocks,
            "cache_dtype": wl.src_dtype, "out_dtype": wl.dst_dtype, "bytes_per_step": wl.algorithmic_bytes(),
            "l2": L2_POLICY}


def make_workload(name: str) -> W.Workload:
    return W.CONFIGS[name]()


def dtype_label(wl: W.Workload) -> str:
    return wl.src_dtype if wl.src_dtype == wl.dst_dtype else f"{wl.src_dtype}->{wl.dst_dtype}"


def kernel_of(path: str, wl: W.Workload, entry: str) -> str:
    """The kernel a call on this path launches: the TMA path ("bulk") has a
    byte-copy kernel and a converting kernel; the SIMT paths one kernel per
    entry point."""
    if path == "bulk":
        return "gather_bulk_kernel" if wl.src_dtype == wl.dst_dtype else "gather_tma_convert_kernel"
    if path == "none":
        return "none"
    return "gather_tokens_kernel" if entry == "tokens" else "gather_simt_kernel"


class DeviceInputs:
    """One replica of a workload's inputs and output, resident on the device."""

    def __init__(self, wl: W.Workload, device, cache=None, dst_offset: int = 0):
        self.cache_full = wl.cache.to(device) if cache is None else cache
        self.cache = self.cache_full[:, :, :wl.entry_size]
        self.bt = wl.block_table.to(device)
        self.cu = wl.cu_seq_lens.to(device)
        self.ss = None if wl.seq_starts is None else wl.seq_starts.to(device)
        self.scale = torch.tensor([wl.scale], dtype=torch.float32, device=device)
        # dst_offset > 0: the output is rows [dst_offset, dst_offset + T) of a
        # larger workspace, as one rank's slice before a context-parallel
        # all-gather; rows below it are filled with a sentinel and must stay so
        self.dst_full = torch.empty((dst_offset + wl.total_tokens, wl.entry_size),
                                    dtype=W.TORCH_DTYPES[wl.dst_dtype], device=device)
        if dst_offset > 0:
            self.dst_full[:dst_offset].view(torch.uint8).fill_(0x5A)
        self.dst = self.dst_full[dst_offset:]
        self.dst_offset = dst_offset
        self.err = torch.zeros(1, dtype=torch.int32, device=device)

    def nbytes(self):
        return self.cache_full.numel() * self.cache_full.element_size() + self.dst.numel() * self.dst.element_size()


class Runner:
    """A workload on the device: replicas, one scheduling workspace, the call."""

    def __init__(self, wl: W.Workload, dev, stream, args, dst_offset: int = 0):
        from paged_mla_kv_cache_gb300 import binding
        self.binding = binding
        self.wl, self.dev, self.stream, self.args = wl, dev, stream, args
        base = DeviceInputs(wl, dev, dst_offset=dst_offset)
        self.nrep = max(2, math.ceil(4 * L2_BYTES / base.nbytes()))
        self.reps = [base] + [DeviceInputs(wl, dev, dst_offset=dst_offset) for _ in range(self.nrep - 1)]
        self.ws_buf = None if args.no_workspace else binding.new_workspace(dev)
        if args.entry == "tokens":
            # the per-token entry point: each output row names its request
            cu_h = wl.cu_seq_lens.numpy()
            t2s_h = np.full(wl.total_tokens, -1, np.int32)
            for r in range(wl.num_reqs):
                t2s_h[cu_h[r]:min(cu_h[r + 1], wl.total_tokens)] = r
            for r in self.reps:
                r.t2s = torch.from_numpy(t2s_h).to(dev)
        path, _ = binding.select_path(base.cache, base.dst, base.bt, base.cu, num_reqs=wl.num_reqs,
                                      options=args.options)
        self.path = ("per-token " + path) if args.entry == "tokens" else path
        self.kernel = kernel_of(path, wl, args.entry)

    def footprint_mb(self):
        return sum(r.nbytes() for r in self.reps) / 1e6

    def step(self, k, strm=None, options=None):
        r = self.reps[k % self.nrep]
        b = self.binding
        opts = self.args.options if options is None else options
        s = self.stream if strm is None else strm
        if self.args.entry == "tokens":
            b.gather_tokens(r.cache, r.dst, r.bt, r.t2s, r.cu, r.scale, r.err, num_reqs=self.wl.num_reqs,
                            stream=s, options=opts, workspace=self.ws_buf)
        else:
            b.gather(r.cache, r.dst, r.bt, r.cu, r.ss, r.scale, r.err, num_reqs=self.wl.num_reqs,
                     stream=s, options=opts, workspace=self.ws_buf)

    def capture(self, n, options=None):
        """A CUDA graph of n consecutive steps (our launches only)."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cs = torch.cuda.current_stream()
            for k in range(n):
                self.step(k, cs, options)
        return g

    def graphs_for(self, steps, options=None):
        per_graph = min(steps, self.nrep * max(1, 120 // self.nrep))
        n_main, rem = divmod(steps, per_graph)
        g_main = self.capture(per_graph, options)
        g_rem = self.capture(rem, options) if rem else None
        g_main.replay()
        if g_rem is not None:
            g_rem.replay()
        torch.cuda.synchronize(self.dev)
        return g_main, n_main, g_rem

    def timed_region(self, graphs, world):
        """One region of exactly the graphs' steps, events on our stream,
        barrier + synchronize on both sides. Returns ms (max over ranks)."""
        g_main, n_main, g_rem = graphs
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(self.dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(self.stream)
        for _ in range(n_main):
            g_main.replay()
        if g_rem is not None:
            g_rem.replay()
        b.record(self.stream)
        torch.cuda.synchronize(self.dev)
        if world > 1:
            torch.distributed.barrier()
        return reduce_max(a.elapsed_time(b), self.dev)

    def cold(self, iters=50, read_back=False):
        """Median call time with L2 flushed before each call, outside the event
        pair: a 512 MB buffer is written (the page's cold-cache protocol), and
        with read_back it is then read back too, so that L2 holds clean lines
        of another buffer and no write-back of the flush lands in the call."""
        flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=self.dev)
        sink = torch.empty((), dtype=torch.int64, device=self.dev)
        times = []
        for k in range(iters):
            flush.fill_(k & 0xFF)
            if read_back:
                torch.sum(flush.view(torch.int64), dim=0, out=sink)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(self.stream)
            self.step(k)
            b.record(self.stream)
            torch.cuda.synchronize(self.dev)
            times.append(a.elapsed_time(b))
        del flush
        times.sort()
        med = statistics.median(times)
        alg = self.wl.algorithmic_bytes()
        peak, _ = measured_peak()
        return {"median_us": round(med * 1e3, 2), "mean_us": round(statistics.fmean(times) * 1e3, 2),
                "p10_us": round(times[len(times) // 10] * 1e3, 2),
                "p90_us": round(times[(9 * len(times)) // 10] * 1e3, 2), "iters": iters,
                "gbs": round(alg / (med * 1e-3) / 1e9, 1), "frac": round(alg / (med * 1e-3) / 1e9 / peak, 4),
                "flush": ("512 MB written then read back" if read_back else "512 MB written")
                         + " before each call, outside the event pair"}

    def check_flags(self):
        for r in self.reps:
            flag = int(r.err.item())
            if flag != 0:
                raise RuntimeError(f"{self.wl.name}: gather reported data errors (flag {flag}) on valid inputs")
            if r.dst_offset > 0 and not bool((r.dst_full[:r.dst_offset].view(torch.uint8) == 0x5A).all()):
                raise RuntimeError(f"{self.wl.name}: rows below the output offset were written")

    def close(self):
        del self.reps
        torch.cuda.empty_cache()


def steady(runner: Runner, steps: int, world: int, min_total_ms: float = 0.0, max_repeats: int = 1,
           options=None):
    """Median over repeats of a region of exactly `steps` steps."""
    graphs = runner.graphs_for(steps, options)
    regions = [runner.timed_region(graphs, world)]
    want = 1 if max_repeats <= 1 else max(5, min(max_repeats, math.ceil(min_total_ms / max(regions[0], 1e-6))))
    while len(regions) < want:
        regions.append(runner.timed_region(graphs, world))
    del graphs
    return regions


def run_per_config(args, dev, stream, world, headline=None):
    """Steady state and cold figures for every named target workload."""
    peak, _ = measured_peak()
    out = {}
    for name in PER_CONFIG:
        if headline is not None and name == args.config:
            out[name] = headline
            continue
        wl = make_workload(name)
        r = Runner(wl, dev, stream, args)
        for k in range(max(args.warmup, 3)):
            r.step(k)
        torch.cuda.synchronize(dev)
        alg = wl.algorithmic_bytes()
        # about 30 ms of steps per region, median of 5 regions
        est = alg / (peak * 0.8e9) * 1e3
        n = int(min(3000, max(30, 30.0 / est)))
        regions = steady(r, n, world, max_repeats=5, min_total_ms=0.0)
        ms = statistics.median(regions) / n
        cold = r.cold()
        cold_clean = r.cold(read_back=True)
        r.check_flags()
        tr = profiled_traffic(name)
        out[name] = {"workload": wl.name, "bytes_per_step": alg, "dtype": dtype_label(wl), "path": r.path,
                     "kernel": r.kernel,
                     "dram_traffic_per_launch": None if tr is None else {"read": tr["read"], "write": tr["write"],
                                                                         "source": tr["source"]},
                     "steady": {"gbs": round(alg / (ms * 1e-3) / 1e9, 1),
                                "frac": round(alg / (ms * 1e-3) / 1e9 / peak, 4),
                                "per_launch_us": round(ms * 1e3, 2), "steps_per_region": n,
                                "regions": len(regions)},
                     "cold": cold, "cold_clean": cold_clean}
        r.close()
        del wl
    # the 300K gather as one rank's slice of a context-parallel workspace:
    # rows [T, 2T) of 2T rows (rank 1 of 2), replayed from CUDA graphs like
    # every steady-state figure here
    wl = make_workload("300k")
    T = wl.total_tokens
    r = Runner(wl, dev, stream, args, dst_offset=T)
    for k in range(max(args.warmup, 3)):
        r.step(k)
    torch.cuda.synchronize(dev)
    alg = wl.algorithmic_bytes()
    n = 200
    regions = steady(r, n, world, max_repeats=5, min_total_ms=0.0)
    ms = statistics.median(regions) / n
    r.check_flags()
    out["300k_cp_slice"] = {"workload": wl.name + ", written at rows [T, 2T) of a 2T-row workspace",
                            "bytes_per_step": alg, "dtype": dtype_label(wl), "path": r.path, "kernel": r.kernel,
                            "dst_offset_rows": T,
                            "steady": {"gbs": round(alg / (ms * 1e-3) / 1e9, 1),
                                       "frac": round(alg / (ms * 1e-3) / 1e9 / peak, 4),
                                       "per_launch_us": round(ms * 1e3, 2), "steps_per_region": n,
                                       "regions": len(regions)},
                            "rows_below_offset": "sentinel intact after every replica's steps"}
    r.close()
    return out


def run_ours(args, wl: W.Workload, ws: int, rank: int, local: int):
    from paged_mla_kv_cache_gb300.build import build_library
    build_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    alg_bytes = wl.algorithmic_bytes()
    runner = Runner(wl, dev, stream, args)
    for k in range(args.warmup):
        runner.step(k)
    torch.cuda.synchronize(dev)

    # --- timed regions: exactly K steps each, repeated so that the clock
    # sampler (50 ms period) sees the GPU under load --------------------------
    graphs = runner.graphs_for(args.steps)
    runner.timed_region(graphs, ws)  # untimed: settles the replays
    sampler = ClockSampler(local)
    time.sleep(0.15)  # let the sampler start
    regions = [runner.timed_region(graphs, ws)]
    repeats = max(3, min(args.max_repeats, math.ceil(args.min_timed_ms / max(regions[0], 1e-6))))
    while len(regions) < repeats:
        regions.append(runner.timed_region(graphs, ws))
    clocks = sampler.stop()
    del graphs
    runner.check_flags()
    ms = statistics.median(regions)
    ms_per_step = ms / args.steps
    value = weak_value(alg_bytes, args.steps, ms, ws)
    # the gather is the only kernel of a step: its average launch duration is
    # the region over the steps (inter-launch gaps included)
    per_launch_ms = ms_per_step

    # --- the same steps with the early-metadata promise (reported beside) -----
    early = None
    if not args.quick and args.entry == "gather" and not (args.options & 8):
        n_e = min(max(args.steps, 200), 3000)
        reg = steady(runner, n_e, ws, options=args.options | 8)
        ms_e = reg[0]
        peak_e, _ = measured_peak()
        early = {"value": round(weak_value(alg_bytes, n_e, ms_e, ws), 1), "unit": "GB/s",
                 "frac": round(alg_bytes / (ms_e / n_e * 1e-3) / 1e9 / peak_e, 4),
                 "per_launch_us": round(ms_e / n_e * 1e3, 2), "steps": n_e,
                 "options": "PMG_OPT_EARLY_METADATA (caller promises no running kernel writes the metadata)"}

    cold = None if args.quick else runner.cold()
    cold_clean = None if args.quick else runner.cold(read_back=True)
    peak, peak_kind = measured_peak()
    achieved = alg_bytes / (per_launch_ms * 1e-3) / 1e9
    # the committed capture of this entry point on this workload, default options only
    profile_key = args.config if args.entry == "gather" else f"tokens_{args.config}"
    tr_h = profiled_traffic(profile_key) if args.options == 0 else None
    headline_entry = {"workload": wl.name, "bytes_per_step": alg_bytes, "dtype": dtype_label(wl),
                      "path": runner.path, "kernel": runner.kernel,
                      "dram_traffic_per_launch": None if tr_h is None else {"read": tr_h["read"], "write": tr_h["write"],
                                                                            "source": tr_h["source"]},
                      "steady": {"gbs": round(achieved, 1), "frac": round(achieved / peak, 4),
                                 "per_launch_us": round(per_launch_ms * 1e3, 2), "steps_per_region": args.steps,
                                 "regions": len(regions)},
                      "cold": cold, "cold_clean": cold_clean}
    footprint = runner.footprint_mb()
    nrep = runner.nrep
    runner.close()

    per_config = None
    if not args.quick and rank == 0 and not args.no_per_config:
        per_config = run_per_config(args, dev, stream, 1, headline=headline_entry)

    # --- end to end: host buffers through the public binding -----------------
    e2e = None
    if not args.quick:
        e2e = run_e2e(wl, dev, stream, alg_bytes, steps=20, ws=ws)

    traffic = tr_h
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
        "dtype": dtype_label(wl),
        "data": "synthetic (seeded N(0,1) cache, seeded block-id permutation)",
        "config": workload_config(wl),
        "path": runner.path if args.options == 0 else f"{runner.path} (options {args.options})",
        "kernel": runner.kernel,
        "schedule": ("static" if args.no_workspace else "dynamic (workspace)")
                    + (", early metadata" if args.early_metadata else ""),
        "parallelism": f"replicas x{ws}",
        "timing": {"regions": len(regions), "steps_per_region": args.steps,
                   "region_ms": {"min": round(min(regions), 4), "median": round(ms, 4), "max": round(max(regions), 4)},
                   "mean_value": round(weak_value(alg_bytes, args.steps * len(regions), sum(regions), ws), 1),
                   "replicas": f"{nrep} input replicas ({footprint:.0f} MB)",
                   "how": "value = bytes x K / median over regions of the device time of exactly K steps "
                          "(CUDA events on the launching stream, barrier + synchronize on both sides)"},
        "roofline": {
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": None if traffic is None else traffic["read"] + traffic["write"],
            "traffic_read": None if traffic is None else traffic["read"],
            "traffic_write": None if traffic is None else traffic["write"],
            "traffic_source": None if traffic is None else traffic["source"],
            "algorithmic_bytes": alg_bytes,
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, burst copy)" if peak_kind == "measured"
                           else "fallback",
            "per_launch_us": round(per_launch_ms * 1e3, 2),
        },
        "clocks": clocks,
        "gpu_launches": args.steps,
        "gpu_launches_note": "our kernel launches inside one timed region (one per step)",
        "cold": cold,
        "cold_clean": cold_clean,
        "early_metadata": early,
        "per_config": per_config,
        "e2e": e2e,
    }
    return result


def run_e2e(wl, dev, stream, alg_bytes, steps, ws):
    """Same metric through the public binding with inputs and output in pinned
    host memory: every step copies all of its inputs host -> device, gathers,
    and copies its whole output device -> host, inside the timed region.

    Steps are pipelined the way a serving loop would run them: two device
    buffer sets, input copies on one stream, the gather on the benchmark's
    stream, output copies on a third, ordered by events. Step k + 1's input
    copy then overlaps step k's output copy (the host link is full duplex).
    `serial` times the same steps one after another on one stream."""
    from paged_mla_kv_cache_gb300 import binding
    h_cache = wl.cache.pin_memory()
    h_bt = wl.block_table.pin_memory()
    h_cu = wl.cu_seq_lens.pin_memory()
    h_ss = None if wl.seq_starts is None else wl.seq_starts.pin_memory()
    h_scale = torch.tensor([wl.scale], dtype=torch.float32).pin_memory()
    h_out = torch.empty((wl.total_tokens, wl.entry_size), dtype=W.TORCH_DTYPES[wl.dst_dtype]).pin_memory()
    h_in = [h_cache, h_bt, h_cu, h_scale] + ([h_ss] if h_ss is not None else [])

    class Set:
        def __init__(self):
            self.inp = [torch.empty_like(t, device=dev) for t in h_in]
            self.out = torch.empty(h_out.shape, dtype=h_out.dtype, device=dev)
            self.err = torch.zeros(1, dtype=torch.int32, device=dev)
            self.ws = binding.new_workspace(dev)
            self.copied = torch.cuda.Event()
            self.gathered = torch.cuda.Event()
            self.drained = torch.cuda.Event()

        def gather(self, strm):
            cache, bt, cu, scale = self.inp[:4]
            ss = self.inp[4] if h_ss is not None else None
            binding.gather(cache[:, :, :wl.entry_size], self.out, bt, cu, ss, scale, self.err,
                           num_reqs=wl.num_reqs, stream=strm, workspace=self.ws)

    sets = [Set(), Set()]
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = h_out.numel() * h_out.element_size()

    def pipelined_step(k):
        b = sets[k % 2]
        with torch.cuda.stream(s_in):
            if k >= 2:
                s_in.wait_event(b.gathered)  # step k - 2 no longer reads this set's inputs
            for d, h in zip(b.inp, h_in):
                d.copy_(h, non_blocking=True)
            b.copied.record(s_in)
        stream.wait_event(b.copied)
        if k >= 2:
            stream.wait_event(b.drained)  # step k - 2's output has left this set's buffer
        b.gather(stream)
        b.gathered.record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(b.gathered)
            h_out.copy_(b.out, non_blocking=True)
            b.drained.record(s_out)

    def serial_step():
        b = sets[0]
        with torch.cuda.stream(stream):
            for d, h in zip(b.inp, h_in):
                d.copy_(h, non_blocking=True)
            b.gather(stream)
            h_out.copy_(b.out, non_blocking=True)

    def timed(fn):
        torch.cuda.synchronize(dev)
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s_in)
        stream.wait_event(a)
        s_out.wait_event(a)
        fn()
        # the end event follows every stream's last operation
        for st in (s_in, s_out):
            ev = torch.cuda.Event()
            ev.record(st)
            stream.wait_event(ev)
        e.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(e) / steps

    def run_pipelined():
        for k in range(steps):
            pipelined_step(k)

    def run_serial():
        for _ in range(steps):
            serial_step()

    for k in range(4):
        pipelined_step(k)
    serial_step()
    torch.cuda.synchronize(dev)
    # three regions of `steps` steps each, median (one region can catch a
    # host-side stall while the steps are being queued)
    ms_all = [timed(run_pipelined) for _ in range(3)]
    ms_serial_all = [timed(run_serial) for _ in range(3)]
    ms, ms_serial = statistics.median(ms_all), statistics.median(ms_serial_all)
    for b in sets:
        if int(b.err.item()) != 0:
            raise RuntimeError("e2e: gather reported data errors on valid inputs")
    return {"value": round(ws * alg_bytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 4), "steps": steps,
            "regions_ms_per_step": [round(x, 4) for x in ms_all],
            "how": "pinned host buffers; two device buffer sets; input copies, gather and output copies on "
                   "three streams ordered by events, so step k + 1's input copy overlaps step k's output copy",
            "serial": {"value": round(ws * alg_bytes / (ms_serial * 1e-3) / 1e9, 1),
                       "ms_per_step": round(ms_serial, 4),
                       "regions_ms_per_step": [round(x, 4) for x in ms_serial_all],
                       "how": "the same steps one after another on one stream"}}


def sample_call(wl: W.Workload, rows: int):
    """A bounded sample of the workload for the CPU oracle: the first
    ceil(len_r * rows / total) rows of every request, as one smaller call of the
    same shape. Returns (args for oracle.gather, bytes, rows)."""
    cache = W.tensor_bits(wl.cache)
    cache_view = np.lib.stride_tricks.as_strided(
        cache, shape=(cache.shape[0], cache.shape[1], wl.entry_size), strides=cache.strides)
    frac = min(1.0, rows / max(wl.rows, 1))
    lens = [int(math.ceil(L * frac)) for L in wl.lens]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    bt = wl.block_table.numpy()
    ss = None if wl.seq_starts is None else wl.seq_starts.numpy()
    nbytes = T * wl.entry_size * (W.ELEM_BYTES[wl.src_dtype] + W.ELEM_BYTES[wl.dst_dtype])
    return dict(cache=cache_view, bt=bt, cu=cu, ss=ss, T=T), nbytes, T


def split_rows(call: dict, parts: int):
    """The sample call cut into `parts` calls over disjoint output row ranges
    (each a plain oracle call: the requests overlapping the range, their row
    ranges clipped and their starts advanced by the rows cut off)."""
    cu, T = call["cu"].astype(np.int64), call["T"]
    R = len(cu) - 1
    ss = np.zeros(R, np.int64) if call["ss"] is None else call["ss"].astype(np.int64)
    out = []
    bounds = np.linspace(0, T, parts + 1).astype(np.int64)
    for a, b in zip(bounds[:-1], bounds[1:]):
        if b <= a:
            continue
        rs = [r for r in range(R) if cu[r] < b and cu[r + 1] > a]
        c_lo = np.array([max(cu[r], a) for r in rs], np.int64)
        c_hi = np.array([min(cu[r + 1], b) for r in rs], np.int64)
        sub_cu = np.concatenate([[0], np.cumsum(c_hi - c_lo)]).astype(np.int32)
        sub_ss = np.array([ss[r] + (c_lo[i] - cu[r]) for i, r in enumerate(rs)], np.int32)
        out.append(dict(cache=call["cache"], bt=np.ascontiguousarray(call["bt"][rs]), cu=sub_cu, ss=sub_ss,
                        T=int(b - a), row0=int(a)))
    return out


def oracle_runner(wl: W.Workload, call: dict):
    from oracle import gather as og
    dst = wl.new_dst()[:call["T"]] if call["T"] <= wl.total_tokens else None

    def run(c=call, d=dst):
        return og.gather(c["cache"], c["bt"], c["cu"], c["ss"], len(c["cu"]) - 1, c["T"], wl.block_size,
                         wl.entry_size, wl.src_dtype, wl.dst_dtype, wl.scale, d)
    return run


def time_oracle(run, budget_s):
    n, t0 = 0, time.perf_counter()
    while True:
        run()
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (n >= 3 and el >= budget_s / 2 and el / n * (n + 1) > budget_s):
            return n, el


def cpu_baseline(wl: W.Workload, budget_s: float = 10.0):
    """The oracle as it stands on the host cores: single-threaded, repeated over
    the full workload (or a prefix sample if one call would exceed a third of
    the budget); then the same sample as concurrent oracle calls over disjoint
    row ranges, one per core (the oracle's C loop runs outside the GIL)."""
    facts = cpu_facts()
    call, nbytes, rows = sample_call(wl, wl.rows)
    run = oracle_runner(wl, call)
    t0 = time.perf_counter()
    run()
    t1 = time.perf_counter() - t0
    if t1 > budget_s / 3:
        call, nbytes, rows = sample_call(wl, int(wl.rows * budget_s / 3 / t1))
        run = oracle_runner(wl, call)
    n, el = time_oracle(run, budget_s)
    gbs = nbytes * n / el / 1e9
    res = {"value": round(gbs, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": f"{n} oracle calls over {rows} of {wl.rows} rows in {el:.1f} s, single thread",
           **facts}
    cores = facts["nproc"] or 1
    if cores > 1:
        parts = split_rows(call, cores)
        runs = [oracle_runner(wl, c) for c in parts]
        with concurrent.futures.ThreadPoolExecutor(max_workers=len(runs)) as pool:
            def all_parts():
                list(pool.map(lambda f: f(), runs))
            m, el_m = time_oracle(all_parts, budget_s / 2)
        res["all_cores"] = {"value": round(nbytes * m / el_m / 1e9, 3), "unit": "GB/s", "cores": len(runs),
                            "kind": f"oracle, {len(runs)} cores",
                            "sample": f"{m} passes over the same {rows} rows split into {len(runs)} concurrent "
                                      f"oracle calls (disjoint row ranges) in {el_m:.1f} s"}
    return res


def run_reference(args, wl, ws, rank):
    """The reference arm: the CPU oracle timed on host cores, each step a bounded
    sample of the workload so that warmup + steps end within a few minutes."""
    if rank != 0:
        return None
    call, _, _ = sample_call(wl, wl.rows)
    run_full = oracle_runner(wl, call)
    t0 = time.perf_counter()
    run_full()
    t_full = time.perf_counter() - t0
    budget = 90.0
    per_step = budget / max(args.steps + args.warmup, 1)
    rows = max(64, min(wl.rows, int(wl.rows * per_step / max(t_full, 1e-9))))
    call, nbytes, rows = sample_call(wl, rows)
    run = oracle_runner(wl, call)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    el = time.perf_counter() - t0
    value = nbytes * args.steps / el / 1e9
    facts = cpu_facts()
    sample = f"{rows} of {wl.rows} rows per step (prefix of every request), single thread"
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype_label(wl), "data": "synthetic",
        "config": workload_config(wl),
        "path": "CPU oracle (per-token loop)",
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample,
                         **facts},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=HEADLINE, choices=sorted(W.CONFIGS))
    ap.add_argument("--quick", action="store_true",
                    help="skip the per-config, cold, early-metadata, e2e and CPU-baseline legs")
    ap.add_argument("--no-per-config", action="store_true", help="skip the per-config leg only")
    ap.add_argument("--min-timed-ms", type=float, default=600.0,
                    help="repeat the K-step region until the regions add up to this much device time")
    ap.add_argument("--max-repeats", type=int, default=400)
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
    if args.steps < 1:
        ap.error("--steps must be >= 1")
    if args.early_metadata:
        args.options |= 8  # PMG_OPT_EARLY_METADATA
    ws, rank, local = dist_env()
    if ws > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if args.impl == "ours" else "gloo"
        torch.distributed.init_process_group(backend=backend, device_id=torch.device("cuda", local)
                                             if backend == "nccl" else None)
    if args.impl == "reference":
        res = run_reference(args, make_workload(args.config), ws, rank) if rank == 0 else None
    else:
        wl = make_workload(args.config)
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
