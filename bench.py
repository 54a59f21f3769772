#!/usr/bin/env python3
"""Benchmark of the grouped NVFP4 block-scaled GEMM (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Metric: microseconds per grouped call. Also reported: effective TFLOP/s and
TB/s, and the fraction of the roofline max(2*sum(M*N*K) / FP4 peak,
algorithmic bytes / HBM peak).

The default workload is the MoE-shaped g=8 problem with M = 80,176,128,72,64,248,96,160,
N = 4096 and K = 7168 (seed 1111). It is the largest of the leaderboard shapes and the
first line of the timing table on page 1 of the pages. The inputs are synthetic, from
`gen` (SplitMix64): uniform E2M1 nibbles, and E4M3 scales uniform over
the codes 0x20..0x40.

Timing (ours):
 * Inputs are resident in HBM, with scales prepacked. Warm-up calls run first,
   and the device table is cached by then.
 * Before every timed call, L2 is flushed: a 2 x L2 buffer is written, then a
   second 2 x L2 buffer is read, so that the call starts with an L2 holding
   neither its inputs nor dirty lines.
 * Each call is timed alone with CUDA events on the launching stream.
   `value` is the mean over K calls; median, min and max are also reported.
 * e2e runs the same call through the public API from pinned HOST buffers with
   row-major scales. Each timed step copies A, B, SFA and SFB host->device,
   runs the GEMM (which reads row-major scales itself where K % 256 == 0, else
   after a prepack launch), and copies C device->host.
 * With the default workload on one GPU, the line also carries `other_workloads`:
   the other four workloads timed the same way, not part of `value`
   (--no-other-workloads skips them).
 * Outside the timed region: `prepack` (every SFA and SFB of the workload through
   nvfp4_prepack_scales_batch, one launch, L2 flushed before each call, with its
   bytes and roofline fraction; the same launch over one scale row after a flush,
   the fixed cost of any flushed call; and `chained`: back-to-back calls over
   rotating operand sets larger than L2 from one CUDA graph, beside a plain
   device-to-device copy of the same bytes) and `cold_call` (calls that miss the
   table cache, against calls that hit it).
 * `clocks`: SM clock, power and clock-event reasons of the GPU in use, sampled
   every 5 ms through NVML during the timed region.
 * Under torchrun (N > 1) every rank runs its own replica on its own GPU (weak
   scaling; the path has no exchange step). Timing is the max over ranks, and
   `value` = that time divided by N (aggregate time per grouped call). With
   --split groups|n the ranks instead share ONE call (strong scaling): whole
   groups, or N ranges of every group, each rank writing its own outputs (C stays
   sharded, nothing crosses between ranks); `value` = the slowest rank's time.
--impl reference times the CPU oracle (the plain C reference restated from the
pages) on bounded samples of the same workload.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import gen  # noqa: E402

NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_FP4_TFLOPS = 13500.0  # dense NVFP4, GB300
# The pages' best leaderboard time for each workload, us per grouped call, on B200
# (page 1, the timing table at the head of submission 495528): another machine's
# number, reported as context through vs_baseline, not a target.
PAGES_BEST_US = {"moe_g8_n4096_k7168": 47.5, "moe_g8_n7168_k2048": 45.0, "g2_n3072_k4096": 14.3,
                 "g2_n4096_k1536": 10.5}
KERNEL_CHOICE = {"auto": 0, "pair": 1, "single": 2, "swapab": 3, "swapab_pair": 4}  # values of NVFP4_OPT_CTA_PAIR
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = ["block_scaled_fp4_persistent_gb300/csrc/gemm_kernel.cuh",
                  "block_scaled_fp4_persistent_gb300/csrc/pair_kernel.cuh",
                  "block_scaled_fp4_persistent_gb300/csrc/ptx.cuh",
                  "block_scaled_fp4_persistent_gb300/csrc/table.h"]


# ------------------------------------------------------------------ helpers --

def workload_stats(groups):
    flops = sum(2 * g.M * g.N * g.K for g in groups)
    nbytes = sum(g.M * g.K // 2 + g.N * g.K // 2 + g.M * g.K // 16 + g.N * g.K // 16 + 2 * g.M * g.N for g in groups)
    return flops, nbytes


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def roofline_terms(groups, peaks):
    flops, nbytes = workload_stats(groups)
    fp4_tflops = peaks["bf16_tflops"] * NOMINAL_FP4_TFLOPS / NOMINAL_BF16_TFLOPS
    t_fp4_us = flops / (fp4_tflops * 1e12) * 1e6
    t_hbm_us = nbytes / (peaks["hbm_gbs"] * 1e9) * 1e6
    return flops, nbytes, fp4_tflops, t_fp4_us, t_hbm_us


def kernel_source_hash():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel, workload):
    """dram read+write bytes per launch from the committed ncu summary of this
    kernel on this workload, or None when that summary was taken on other kernel
    sources."""
    path = os.path.join(ROOT, "profiles", f"{kernel.split('<')[0]}_{workload}.txt")
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line and not line.startswith(" "):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    if fields.get("kernel_sources_sha256_16") != kernel_source_hash():
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def gpu_pci_id(local_rank):
    """The PCI bus id of the CUDA device in use ("dddddddd:bb:dd.0"), which names the same GPU
    to NVML and nvidia-smi whatever CUDA_VISIBLE_DEVICES maps; None where torch lacks it."""
    import torch
    p = torch.cuda.get_device_properties(local_rank)
    try:
        return "%08x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
    except AttributeError:
        return None


class ClockSampler:
    """SM clock, power and clock-event reasons of the GPU in use, sampled every few
    milliseconds while running: through NVML (libnvidia-ml, read-only queries) where it
    loads, else nvidia-smi every 200 ms. window_begin()/window_end() bracket the timed
    region; the summary covers the samples inside it, or, where the region was shorter
    than one period, the samples of the whole run (said in `window`)."""

    NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                    0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    SMI_QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                 "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                 "clocks_event_reasons.sw_power_cap")

    def __init__(self, pci_id, period_s=0.005):
        self.pci_id = pci_id
        self.period_s = period_s
        self.samples = []  # (t, sm_mhz, max_mhz, power_w, [reasons])
        self.source = None
        self.windows = []
        self._stop = threading.Event()
        self._thread = None
        self._proc = None

    def _nvml(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        if self.pci_id is None or lib.nvmlDeviceGetHandleByPciBusId_v2(self.pci_id.encode(), ctypes.byref(h)) != 0:
            raise OSError("no NVML handle for the device")
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        clk, mx, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()

        def read():
            lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk))      # NVML_CLOCK_SM
            lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
            lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw))
            get_reasons(h, ctypes.byref(rs))
            names = [n for bit, n in self.NVML_REASONS.items() if rs.value & bit]
            return float(clk.value), float(mx.value), pw.value / 1000.0, names
        read()
        return read

    def _loop(self, read):
        while not self._stop.is_set():
            try:
                self.samples.append((time.perf_counter(),) + read())
            except Exception:
                pass
            self._stop.wait(self.period_s)

    def _smi_loop(self):
        for line in self._proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                names = [n for n, v in zip(["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                            "sw_power_cap"], parts[3:7]) if v.lower() == "active"]
                self.samples.append((time.perf_counter(), float(parts[0]), float(parts[1]), float(parts[2]), names))
            except ValueError:
                continue

    def __enter__(self):
        try:
            read = self._nvml()
            self.source = "nvml"
            self._thread = threading.Thread(target=self._loop, args=(read,), daemon=True)
        except OSError:
            try:
                cmd = ["nvidia-smi", f"--query-gpu={self.SMI_QUERY}", "--format=csv,noheader,nounits", "-lms", "200"]
                if self.pci_id:
                    cmd[1:1] = ["-i", self.pci_id]
                self._proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.source = "nvidia-smi"
                self._thread = threading.Thread(target=self._smi_loop, daemon=True)
            except OSError:
                self._thread = None
        if self._thread is not None:
            self._thread.start()
        return self

    def window_begin(self):
        self.windows.append([time.perf_counter(), None])

    def window_end(self):
        if self.windows:
            self.windows[-1][1] = time.perf_counter()

    def __exit__(self, *exc):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=2)

    def summary(self):
        inside = [x for x in self.samples if any(a <= x[0] <= (b or a) for a, b in self.windows)]
        window = "timed region"
        if not inside:
            inside, window = list(self.samples), "whole run (the timed region was shorter than one sample period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": self.source}
        reasons = sorted({n for x in inside for n in x[4]})
        return {"sm_mhz": statistics.median(x[1] for x in inside), "sm_max_mhz": max(x[2] for x in inside),
                "power_w_max": round(max(x[3] for x in inside), 1), "reasons": reasons, "samples": len(inside),
                "window": window, "source": self.source, "period_ms": (self.period_s * 1e3 if self.source == "nvml"
                                                                      else 200), "gpu_pci": self.pci_id}


# --------------------------------------------------------- distributed glue --

def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


def reduce_max(value: float, world: int):
    """Max of `value` over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------- CPU oracle leg --

def _row_slices(groups, start, count):
    """`count` output rows taken cyclically from row `start` of the concatenation of all groups'
    rows, as sub-groups (consecutive rows of one group stay together)."""
    total = sum(g.M for g in groups)
    offs = np.cumsum([0] + [g.M for g in groups])
    picked = {}
    for j in range(min(count, total)):
        r = (start + j) % total
        gi = int(np.searchsorted(offs, r, side="right") - 1)
        picked.setdefault(gi, []).append(r - int(offs[gi]))
    sub = []
    for gi, rows in picked.items():
        g = groups[gi]
        idx = np.array(sorted(rows))
        sub.append(gen.GroupInputs(len(idx), g.N, g.K, g.A[idx], g.B, g.SFA[idx], g.SFB))
    return sub


def oracle_sample(groups, start, rows, threads):
    """Runs the oracle on `rows` output rows. Returns (seconds, multiply-adds, threads used)."""
    import oracle
    sub = _row_slices(groups, start, rows)
    t0 = time.perf_counter()
    oracle.grouped_gemm(sub, nthreads=threads)
    dt = time.perf_counter() - t0
    return dt, sum(g.M * g.N * g.K for g in sub), min(threads, max(g.M for g in sub))


def oracle_rows_for(groups, budget_s, threads):
    """How many rows one sample may take to stay near budget_s (at least 1)."""
    dt, _, _ = oracle_sample(groups, 0, 1, threads)
    waves = int(budget_s / max(dt, 1e-4))
    rows = max(1, threads * waves) if waves >= 1 else 1
    return min(rows, sum(g.M for g in groups))


def time_oracle(groups, target_s, threads):
    """The oracle on a row sample sized to about target_s seconds, scaled to one full grouped
    call by multiply-adds. Returns (us per call, sample description, threads used)."""
    rows = oracle_rows_for(groups, target_s, threads)
    dt, macs, used = oracle_sample(groups, 0, rows, threads)
    macs_full = sum(g.M * g.N * g.K for g in groups)
    desc = (f"{min(rows, sum(g.M for g in groups))} of {sum(g.M for g in groups)} output rows (all N, all K), "
            f"{dt:.2f} s; time scaled by full/sampled multiply-adds")
    return dt * 1e6 * macs_full / macs, desc, used


# ---------------------------------------------------------------- our arm ---

def time_prepack(groups, dev, stream, flush, steps, peaks):
    """nvfp4_prepack_scales_batch over every SFA and SFB of the workload (one launch), L2
    flushed before each call, CUDA events around it. The result must equal the per-operand
    prepack's bit for bit."""
    import torch
    import block_scaled_fp4_persistent_gb300 as nv
    srcs, dsts, rows, Ks, singles = [], [], [], [], []
    for g in groups:
        for sf, r in ((g.SFA, g.M), (g.SFB, g.N)):
            t = torch.from_numpy(np.ascontiguousarray(sf)).to(dev)
            srcs.append(t)
            dsts.append(torch.empty(max(1, nv.nvfp4_prepacked_scale_bytes(r, g.K)), dtype=torch.uint8, device=dev))
            rows.append(r)
            Ks.append(g.K)
            singles.append(nv.prepack_scales(t, g.K))
    args = ([t.data_ptr() for t in srcs], rows, Ks, [t.data_ptr() for t in dsts])
    for _ in range(3):
        flush()
        nv.nvfp4_prepack_scales_batch(*args, stream)
    torch.cuda.synchronize()
    for a, b in zip(dsts, singles):
        if not torch.equal(a, b):
            raise RuntimeError("batched prepack differs from the per-operand prepack")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e0, e1 in ev:
        flush()
        e0.record(stream)
        nv.nvfp4_prepack_scales_batch(*args, stream)
        e1.record(stream)
    torch.cuda.synchronize()
    us = statistics.fmean(a.elapsed_time(b) for a, b in ev) * 1e3
    read = sum(r * k // 16 for r, k in zip(rows, Ks))
    written = sum(nv.nvfp4_prepacked_scale_bytes(r, k) for r, k in zip(rows, Ks))
    gbs = (read + written) / (us * 1e-6) / 1e9

    # the fixed cost of any flushed call: the same launch over one 16-byte scale row
    one_src = torch.zeros(16, dtype=torch.uint8, device=dev)
    one_dst = torch.empty(512, dtype=torch.uint8, device=dev)
    one = ([one_src.data_ptr()], [1], [64], [one_dst.data_ptr()])
    ev1 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e0, e1 in ev1:
        flush()
        e0.record(stream)
        nv.nvfp4_prepack_scales_batch(*one, stream)
        e1.record(stream)
    torch.cuda.synchronize()
    floor_us = statistics.fmean(a.elapsed_time(b) for a, b in ev1) * 1e3

    # chained: back-to-back calls over rotating operand sets that together exceed L2 three
    # times (so each call reads its operands from HBM), captured once in a CUDA graph so that
    # the host's launch cost does not starve the GPU; beside it, a plain device-to-device copy
    # of the same read bytes under the same conditions
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n_sets = max(2, -(-3 * l2 // max(1, read + written)))
    sets = [args]
    held = []
    for _ in range(n_sets - 1):
        s_src = [t.clone() for t in srcs]
        s_dst = [torch.empty_like(t) for t in dsts]
        held.append((s_src, s_dst))
        sets.append(([t.data_ptr() for t in s_src], rows, Ks, [t.data_ptr() for t in s_dst]))
    words = read // 4
    copies = [(torch.empty(words, dtype=torch.int32, device=dev), torch.empty(words, dtype=torch.int32, device=dev))
              for _ in range(n_sets)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())

    def chained(body):
        with torch.cuda.stream(side):
            body()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            body()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        per = []
        for _ in range(20):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(side):
                e0.record(side)
                graph.replay()
                e1.record(side)
            torch.cuda.synchronize()
            per.append(e0.elapsed_time(e1) * 1e3 / n_sets)
        return statistics.fmean(per)

    def prepack_all():
        for a in sets:
            nv.nvfp4_prepack_scales_batch(*a, side.cuda_stream)

    def copy_all():
        for a, b in copies:
            b.copy_(a)

    chained_us = chained(prepack_all)
    copy_us = chained(copy_all)
    torch.cuda.synchronize()
    for (_, s_dst) in held:
        for a, b in zip(s_dst, dsts):
            if not torch.equal(a, b):
                raise RuntimeError("chained prepack differs from the timed one")
    cgbs = (read + written) / (chained_us * 1e-6) / 1e9
    return {"value": round(us, 3), "unit": "us", "steps": steps, "operands": len(rows), "launches": 1,
            "algorithmic_bytes": read + written, "read_bytes": read, "written_bytes": written,
            "achieved_gbs": round(gbs, 1), "frac": round(gbs / peaks["hbm_gbs"], 4),
            "what": "nvfp4_prepack_scales_batch of every SFA and SFB of the workload, L2 flushed before each call",
            "flushed_floor_us": round(floor_us, 3),
            "chained": {"value": round(chained_us, 3), "unit": "us", "achieved_gbs": round(cgbs, 1),
                        "frac": round(cgbs / peaks["hbm_gbs"], 4), "sets": n_sets,
                        "copy_same_bytes_us": round(copy_us, 3),
                        "what": f"back-to-back calls over {n_sets} operand sets (together 3x L2), one CUDA graph; "
                                f"copy_same_bytes_us: a device-to-device copy of the {read} read bytes, same conditions"}}


def time_cold_calls(keep, stream, flush, reps):
    """Calls that miss the table cache (each with a fresh C buffer, so a new table is built:
    tensor maps encoded, tile lists built, table uploaded) against calls that hit it: host time
    until the call returns, and event time of the call on the stream (upload included)."""
    import torch
    import block_scaled_fp4_persistent_gb300 as nv

    def probs_with(Cs):
        return [nv.problem(A, B, SFA, SFB, C) for (A, B, SFA, SFB, _), C in zip(keep, Cs)]

    out = {}
    alive = []  # every C of the misses stays allocated, so no pointer (and no table key) repeats
    for kind in ("miss", "hit"):
        fixed = [torch.empty_like(k[4]) for k in keep]
        host, gpu = [], []
        for i in range(reps):
            Cs = [torch.empty_like(k[4]) for k in keep] if kind == "miss" else fixed
            alive.append(Cs)
            probs = probs_with(Cs)
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            t0 = time.perf_counter()
            nv.nvfp4_grouped_gemm(probs, stream)
            host.append((time.perf_counter() - t0) * 1e6)
            e1.record(stream)
            torch.cuda.synchronize()
            if kind == "hit" and i == 0:
                host.clear()  # the first call of the fixed set is itself a miss
                continue
            gpu.append(e0.elapsed_time(e1) * 1e3)
        out[kind] = {"host_us": round(statistics.median(host), 1), "gpu_us": round(statistics.median(gpu), 3)}
    out["reps"] = reps
    out["what"] = ("miss: every call with a new C pointer builds and uploads a new table (the cache holds 32, so "
                   "misses also evict); hit: the same call repeated. host_us = time until the call returns; "
                   "gpu_us = event time on the stream (table upload and kernel), L2 flushed before each call")
    return out


def shard_inputs(groups, world, rank, mode):
    """This rank's share of one call (block_scaled_fp4_persistent_gb300.shard's plans) as
    host inputs: whole groups, or every group cut to this rank's range of B's rows (and
    its scale rows); the rank's C is its column block of each group's C."""
    from block_scaled_fp4_persistent_gb300 import shard
    shapes = [(g.M, g.N, g.K) for g in groups]
    if mode == "groups":
        return [groups[i] for i in shard.shard_groups(shapes, world)[rank]]
    return [gen.GroupInputs(groups[gi].M, n1 - n0, groups[gi].K, groups[gi].A, groups[gi].B[n0:n1], groups[gi].SFA,
                            groups[gi].SFB[n0:n1]) for gi, n0, n1 in shard.shard_n(shapes, world)[rank]]


def run_ours(args, groups, rank, world, local_rank):
    import torch
    import block_scaled_fp4_persistent_gb300 as nv
    with ClockSampler(gpu_pci_id(local_rank)) as clocks:
        return _run_ours(args, groups, rank, world, local_rank, clocks)


def _run_ours(args, groups, rank, world, local_rank, clocks):
    import torch
    import block_scaled_fp4_persistent_gb300 as nv

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    peaks, peak_kind = load_peaks()
    flops, nbytes, fp4_tflops, t_fp4_us, t_hbm_us = roofline_terms(groups, peaks)

    # inputs resident in HBM, scales prepacked
    keep, probs = [], []
    for g in groups:
        A = torch.from_numpy(g.A).to(dev)
        B = torch.from_numpy(g.B).to(dev)
        SFA = nv.prepack_scales(torch.from_numpy(g.SFA).to(dev), g.K)
        SFB = nv.prepack_scales(torch.from_numpy(g.SFB).to(dev), g.K)
        C = torch.empty((g.M, g.N), dtype=torch.float16, device=dev)
        keep.append((A, B, SFA, SFB, C))
        probs.append(nv.problem(A, B, SFA, SFB, C))
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_w = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
    flush_r = torch.ones(2 * l2 // 4, dtype=torch.float32, device=dev)
    sink = torch.zeros(1, dtype=torch.float32, device=dev)

    def flush():
        flush_w.fill_(1.0)
        torch.sum(flush_r, dim=(0,), keepdim=True, out=sink)

    for _ in range(args.warmup):
        flush()
        nv.nvfp4_grouped_gemm(probs, stream)
    torch.cuda.synchronize()
    kernel = nv.nvfp4_last_kernel()
    launches_per_call = nv.nvfp4_last_launches()  # this library's kernels per grouped call (the same every call)
    st, detail = nv.nvfp4_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {st} {detail}")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    fl_starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    clocks.window_begin()
    w0 = time.perf_counter()
    for i in range(args.steps):
        fl_starts[i].record(stream)
        flush()
        starts[i].record(stream)
        nv.nvfp4_grouped_gemm(probs, stream)
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - w0
    clocks.window_end()
    st, detail = nv.nvfp4_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {st} {detail}")
    per_call_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    flush_ms = [s.elapsed_time(e) for s, e in zip(fl_starts, starts)]
    mean_us = statistics.fmean(per_call_ms) * 1e3
    med_us = statistics.median(per_call_ms) * 1e3
    mean_us_all = reduce_max(mean_us, world)

    # Chained calls, for callers that run grouped GEMMs back to back: batches of
    # back-to-back calls with programmatic dependent launch on (each call may set up
    # while the one before finishes), L2 flushed before each batch only. Reported beside
    # the headline, which flushes L2 before every call and launches without it.
    chain_calls, chain_batches = 20, max(3, min(50, args.steps // 20))
    nv.nvfp4_set_option(nv.NVFP4_OPT_PDL, 1)
    try:
        for _ in range(2):
            nv.nvfp4_grouped_gemm(probs, stream)
        torch.cuda.synchronize()
        ch_starts = [torch.cuda.Event(enable_timing=True) for _ in range(chain_batches)]
        ch_ends = [torch.cuda.Event(enable_timing=True) for _ in range(chain_batches)]
        for i in range(chain_batches):
            flush()
            ch_starts[i].record(stream)
            for _ in range(chain_calls):
                nv.nvfp4_grouped_gemm(probs, stream)
            ch_ends[i].record(stream)
        torch.cuda.synchronize()
    finally:
        nv.nvfp4_set_option(nv.NVFP4_OPT_PDL, 0)
    st, detail = nv.nvfp4_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {st} {detail}")
    chain_us = reduce_max(statistics.fmean(s.elapsed_time(e) for s, e in zip(ch_starts, ch_ends)) * 1e3 / chain_calls,
                          world)
    working_set = nbytes  # inputs + C of one call, algorithmic bytes

    # End to end: host buffers, row-major scales, every step's copies inside the timed
    # region. A step's inputs sit in one pinned host arena and cross in one copy (the host
    # link carries ~210 GB/s however the bytes are cut, but every copy has a fixed cost),
    # and its results come back in one copy. Device arenas are double-buffered over three
    # streams, so step i+1's inputs cross while step i computes and returns its result.
    e2e_steps = max(1, min(args.steps, args.e2e_steps))

    def packed(sizes):
        offs, off = [], 0
        for n in sizes:
            offs.append(off)
            off = (off + n + 255) // 256 * 256
        return offs, off

    in_offs, in_bytes = packed([a.nbytes for g in groups for a in (g.A, g.B, g.SFA, g.SFB)])
    out_offs, out_bytes = packed([g.M * g.N * 2 for g in groups])
    h_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    for i, arr in enumerate(a for g in groups for a in (g.A, g.B, g.SFA, g.SFB)):
        h_in[in_offs[i]:in_offs[i] + arr.nbytes].copy_(torch.from_numpy(np.ascontiguousarray(arr).reshape(-1).view(np.uint8)))
    h_out = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
    d_in = [torch.empty(in_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    d_out = [torch.empty(out_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    e2e_probs = []
    for b in range(2):
        pi, po = d_in[b].data_ptr(), d_out[b].data_ptr()
        e2e_probs.append([nv.Nvfp4Problem(g.M, g.N, g.K, nv.NVFP4_SF_ROWMAJOR, pi + in_offs[4 * j], pi + in_offs[4 * j + 1],
                                          pi + in_offs[4 * j + 2], pi + in_offs[4 * j + 3], po + out_offs[j])
                          for j, g in enumerate(groups)])
    h2d, d2h = sum(a.nbytes for g in groups for a in (g.A, g.B, g.SFA, g.SFB)), sum(g.M * g.N * 2 for g in groups)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        b = i % 2
        s_in.wait_event(ev_comp[b])  # the GEMM that last read d_in[b] is done
        with torch.cuda.stream(s_in):
            d_in[b].copy_(h_in, non_blocking=True)
        ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])  # the copy that last read d_out[b] is done
        nv.nvfp4_grouped_gemm(e2e_probs[b], stream)
        ev_comp[b].record(stream)
        s_out.wait_event(ev_comp[b])
        with torch.cuda.stream(s_out):
            h_out.copy_(d_out[b], non_blocking=True)
        ev_out[b].record(s_out)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(s_out)  # after the last step's result copy, which follows everything else
    torch.cuda.synchronize()
    barrier(world)
    e2e_us = reduce_max(e0.elapsed_time(e1) * 1e3 / e2e_steps, world)
    e2e_launches = nv.nvfp4_last_launches()  # kernels per grouped call on this path
    st, detail = nv.nvfp4_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {st} {detail}")
    # the e2e result must match the resident-input result bit for bit
    for j, (g, (_, _, _, _, C)) in enumerate(zip(groups, keep)):
        hC = h_out[out_offs[j]:out_offs[j] + g.M * g.N * 2].view(torch.int16).view(g.M, g.N)
        if not torch.equal(C.cpu().view(torch.int16), hC):
            raise RuntimeError("e2e output differs from the resident-input output")

    # outside the timed region: the prepack on its own, and table-cache misses
    prepack = time_prepack(groups, dev, stream, flush, min(args.steps, 200), peaks)
    cold = time_cold_calls(keep, stream, flush, 40)

    achieved_gbs = nbytes / (mean_us * 1e-6) / 1e9
    roof_us = max(t_fp4_us, t_hbm_us)
    out = {
        "metric": "us per grouped call (NVFP4 block-scaled grouped GEMM, fp16 out)",
        # replicas: N calls finish in the slowest rank's time, so one call costs that / N;
        # shards: one call finishes in the slowest rank's time
        "value": round(mean_us_all / (world if args.split == "replicas" else 1), 3),
        "unit": "us",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(mean_us_all / 1e3, 6),
        "higher_is_better": False,
        "scaling": "weak" if args.split == "replicas" else "strong",
        "vs_baseline": (round(mean_us_all / (world if args.split == "replicas" else 1) / PAGES_BEST_US[args.workload], 4)
                        if args.workload in PAGES_BEST_US else None),
        "vs_baseline_ref": ({"value": PAGES_BEST_US[args.workload], "unit": "us", "hardware": "B200",
                             "what": "the pages' best leaderboard time for this workload (context, not the target)"}
                            if args.workload in PAGES_BEST_US else None),
        "dtype": "e2m1 x e2m1 (ue4m3 block-16 scales), fp32 accumulate, fp16 out",
        "data": "synthetic (SplitMix64 seeded generator; shapes and distributions of the leaderboard workload)",
        "config": {"workload": args.workload, "g": len(groups), "M": [g.M for g in groups],
                   "N": [g.N for g in groups], "K": [g.K for g in groups], "seed": gen.WORKLOADS[args.workload]["seed"],
                   "kernel_choice": args.kernel,
                   "scales": "prepacked 128x4 blocked layout", "l2": "flushed before every timed call "
                   "(2xL2 write, then 2xL2 read)", "parallelism": (f"replicas x{world}" if args.split == "replicas"
                                   else f"one call in {args.split} shards x{world} (rank 0's share below)")},
        "median_us": round(med_us, 3),
        "min_us": round(min(per_call_ms) * 1e3, 3),
        "max_us": round(max(per_call_ms) * 1e3, 3),
        "tflops": round(flops / (mean_us * 1e-6) / 1e12, 2),
        "tbs": round(achieved_gbs / 1e3, 4),
        "roofline_us": round(roof_us, 3),
        "roofline_fraction": round(roof_us / mean_us, 4),
        "roofline_terms_us": {"fp4": round(t_fp4_us, 3), "hbm": round(t_hbm_us, 3),
                              "fp4_peak_tflops": round(fp4_tflops, 1),
                              "fp4_peak_kind": f"{peak_kind} bf16 x nominal fp4/bf16 ratio 6"},
        "roofline": {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved_gbs / peaks["hbm_gbs"], 4), "peak_kind": f"{peak_kind} (copy bandwidth)",
                     "algorithmic_bytes_per_launch": nbytes, "traffic": profiled_traffic(kernel, args.workload),
                     "kernel": kernel},
        "gpu_launches": launches_per_call * args.steps,
        "time_share": {"gemm": round(sum(per_call_ms) / (sum(per_call_ms) + sum(flush_ms)), 4),
                       "l2_flush": round(sum(flush_ms) / (sum(per_call_ms) + sum(flush_ms)), 4)},
        "timed_region_wall_s": round(wall, 3),
        "clocks": clocks.summary(),
        "prepack": prepack,
        "cold_call": cold,
        "chained": {"value": round(chain_us / (world if args.split == "replicas" else 1), 3), "unit": "us",
                    "calls_per_batch": chain_calls,
                    "batches": chain_batches, "pdl": True,
                    "l2": ("flushed before each batch only; one call's inputs and C (%.0f MB) %s L2 (%.0f MB)"
                           % (working_set / 1e6, "exceed" if working_set > l2 else "fit in", l2 / 1e6))},
        "e2e": {"value": round(e2e_us / (world if args.split == "replicas" else 1), 3), "unit": "us", "steps": e2e_steps,
                "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "gpu_launches_per_step": e2e_launches,
                "h2d_gbs": round(h2d / (e2e_us * 1e-6) / 1e9, 1) if e2e_us > 0 else None,
                "h2d_note": "the copy in is the whole step: this box's host link carries ~210 GB/s host to device "
                            "(copy engine and SM loads of mapped pinned memory alike)",
                "path": "one pinned host arena of A/B/row-major SFA/SFB -> one H2D copy -> nvfp4_grouped_gemm (the GEMM "
                        "kernel reads the row-major scales itself where K % 256 == 0, else a prepack launch first) -> "
                        "one D2H copy of C; device arenas double-buffered over three streams, so step i+1's copy in "
                        "overlaps step i's GEMM and copy out"},
    }
    return out


def time_flushed(groups, steps, warmup, local_rank):
    """The headline protocol (L2 flushed before every call, CUDA events around each call)
    on another workload, for the line's other_workloads key: mean us per call and the kernel."""
    import torch
    import block_scaled_fp4_persistent_gb300 as nv

    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    keep, probs = [], []
    for g in groups:
        A = torch.from_numpy(g.A).to(dev)
        B = torch.from_numpy(g.B).to(dev)
        SFA = nv.prepack_scales(torch.from_numpy(g.SFA).to(dev), g.K)
        SFB = nv.prepack_scales(torch.from_numpy(g.SFB).to(dev), g.K)
        C = torch.empty((g.M, g.N), dtype=torch.float16, device=dev)
        keep.append((A, B, SFA, SFB, C))
        probs.append(nv.problem(A, B, SFA, SFB, C))
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_w = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
    flush_r = torch.ones(2 * l2 // 4, dtype=torch.float32, device=dev)
    sink = torch.zeros(1, dtype=torch.float32, device=dev)

    def flush():
        flush_w.fill_(1.0)
        torch.sum(flush_r, dim=(0,), keepdim=True, out=sink)

    for _ in range(warmup):
        flush()
        nv.nvfp4_grouped_gemm(probs, stream)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        flush()
        starts[i].record(stream)
        nv.nvfp4_grouped_gemm(probs, stream)
        ends[i].record(stream)
    torch.cuda.synchronize()
    st, detail = nv.nvfp4_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {st} {detail}")
    return statistics.fmean(s.elapsed_time(e) for s, e in zip(starts, ends)) * 1e3, nv.nvfp4_last_kernel()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="moe_g8_n4096_k7168", choices=sorted(gen.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--split", default="replicas", choices=["replicas", "groups", "n"],
                    help="N > 1: every rank runs its own replica of the call (weak scaling, the default), or "
                         "its share of ONE call: whole groups, or N ranges of every group (strong scaling)")
    ap.add_argument("--kernel", default="auto", choices=sorted(KERNEL_CHOICE),
                    help="kernel kind (NVFP4_OPT_CTA_PAIR): the library's automatic choice by default")
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="budget of the oracle timing sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip timing the second MoE workload beside the default one")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local_rank = dist_env()
    if world != args.gpus:
        if world == 1 and args.gpus > 1:
            ap.error("--gpus > 1 needs torchrun (one process per GPU)")
    w = gen.WORKLOADS[args.workload]

    if args.impl == "reference":
        if rank != 0:
            return 0
        groups = gen.make_problem_set(w["seed"], w["Ms"], w["Ns"], w["Ks"])
        threads = os.cpu_count() or 1
        flops, nbytes = workload_stats(groups)
        macs_full = flops // 2
        budget = max(0.02, 90.0 / (args.steps + args.warmup))
        rows = oracle_rows_for(groups, budget, threads)
        cursor = 0
        for _ in range(args.warmup):
            oracle_sample(groups, cursor, rows, threads)
            cursor += rows
        samples, used = [], 1
        for _ in range(args.steps):
            dt, macs, used = oracle_sample(groups, cursor, rows, threads)
            cursor += rows
            samples.append(dt * 1e6 * macs_full / macs)
        desc = (f"each step: {rows} consecutive output rows (all N, all K) of the {sum(w['Ms'])} in one call, "
                f"cycling through the groups; time scaled by full/sampled multiply-adds")
        value = statistics.fmean(samples)
        print(json.dumps({
            "impl": "reference", "metric": "us per grouped call (NVFP4 block-scaled grouped GEMM, fp16 out)",
            "value": round(value, 1), "unit": "us", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(value / 1e3, 3), "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64 accumulate, fp16 out", "data": "synthetic",
            "config": {"workload": args.workload, "g": len(groups), "M": w["Ms"], "N": w["Ns"], "K": w["Ks"],
                       "seed": w["seed"]},
            "tflops": round(flops / (value * 1e-6) / 1e12, 6), "tbs": round(nbytes / (value * 1e-6) / 1e12, 6),
            "cpu_baseline": {"value": round(value, 1), "unit": "us", "cores": used, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 1), "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }))
        return 0

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if args.kernel != "auto":
        import block_scaled_fp4_persistent_gb300 as nv
        nv.nvfp4_set_option(nv.NVFP4_OPT_CTA_PAIR, KERNEL_CHOICE[args.kernel])
    if args.split == "replicas":
        # each rank draws its own replica of the workload (weak scaling)
        groups = gen.make_problem_set(w["seed"] + rank, w["Ms"], w["Ns"], w["Ks"])
    else:
        # every rank draws the same call and runs its share of it (strong scaling)
        groups = shard_inputs(gen.make_problem_set(w["seed"], w["Ms"], w["Ns"], w["Ks"]), world, rank, args.split)
    out = run_ours(args, groups, rank, world, local_rank)
    if world == 1 and args.workload == "moe_g8_n4096_k7168" and not args.no_other_workloads:
        # the other workloads, timed the same way (not part of the headline value)
        out["other_workloads"] = {}
        peaks, _ = load_peaks()
        for other in ("moe_g8_n7168_k2048", "g2_n3072_k4096", "g2_n4096_k1536", "tiny_g2"):
            other_groups = gen.make_workload(other)
            steps = min(args.steps, 2000)
            us, kern = time_flushed(other_groups, steps, args.warmup, local_rank)
            _, nb, _, t_fp4, t_hbm = roofline_terms(other_groups, peaks)
            out["other_workloads"][other] = {
                "value": round(us, 3), "unit": "us", "steps": steps,
                "roofline_fraction": round(max(t_fp4, t_hbm) / us, 4),
                "tbs": round(nb / (us * 1e-6) / 1e12, 4), "kernel": kern,
                "vs_baseline": round(us / PAGES_BEST_US[other], 4) if other in PAGES_BEST_US else None,
                "l2": "flushed before every timed call"}
    if rank == 0:
        if not args.no_cpu_baseline:
            threads = os.cpu_count() or 1
            us, desc, used = time_oracle(groups, args.cpu_seconds, threads)
            out["cpu_baseline"] = {"value": round(us, 1), "unit": "us", "cores": used, "kind": "oracle",
                                   "sample": desc}
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
