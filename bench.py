"""Benchmark of the tile-scheduled GEMM hot path on one GB300 (or N replicas).

One step = one pass of the whole hot path on the headline workload: a bf16
GEMM of 8192 x 8192 x 8192 (bf16 output, Cluster Launch Control scheduler,
2-CTA 256 x 256 tiles) followed by the grid-stride int16 copy of 2^28
elements.  Inputs are seeded synthetic data already resident in HBM; both
working sets are larger than L2 (256 MiB of GEMM operands, 1 GiB of copy
traffic), so no L2 flush is inserted between steps.

``value`` = GEMM TFLOP/s (2*M*N*K per launch / CUDA-event time of the GEMM
launches, summed over ranks).  The copy's HBM GB/s is reported beside it.
``e2e`` times the same GEMM through the public call with host buffers: the
host->device copy of A and B from pinned memory, the GEMM, and the
device->host read of D are all inside the timed region; its ``roofline`` sets
the host traffic of a step against the same copies timed alone, with no GEMM.

After the headline, the same line reports the other workloads, each timed in a
region of its own: ``gemm4096`` (4096^3 bf16-out, the automatic tile and the
128x256 tile, static persistent vs CLC, launches back to back over four
rotating buffer sets so that no launch finds its operands in L2),
``contended`` (the ragged 8191x6143x4096 fp32-out GEMM while a spin kernel
holds 32 SMs for half the solo time: >= 10 alternating static/CLC pairs, the
median times and each scheduler's launch tail from a traced run) and
``smallk`` (8192x8192x64 bf16-out, output-write bound, in HBM GB/s) and
``grouped`` (16 groups of 2048x2048 whose K ranges from 64 to 8192, the groups
scheduled longest K first, static persistent vs CLC).  Clocks
are sampled in process through read-only NVML queries every 1 ms during every
timed region.

``--impl reference`` times the CPU oracle (the plain fp64 triple loop) on the
host cores instead, on a bounded sample of the same workload (one row of D per
step); it is a deliberately slow baseline, not a competitor.

Multi-GPU (torchrun): every rank runs the same independent problem (weak
scaling, no data-path collective); a barrier brackets the timed region and the
slowest rank's time is used.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_PATH = os.path.join(ROOT, "profiles", "traffic.txt")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_SUSTAINED = 1700.0
KERNEL_SOURCES = {"gemm": ["gemm_kernel.cuh", "ptx.cuh", "gemm_params.h", "gemm_launch.cuh"],
                  "copy": ["copy.cu", "shift.cuh"], "rows": ["rows_copy.cu", "ptx.cuh", "gemm_params.h", "shift.cuh"]}


# ------------------------------------------------------------------ helpers
def _code_only(src: str) -> str:
    """C/C++ source without its comments and with whitespace runs collapsed (string and character
    literals kept as they are), so that a comment edit does not change a kernel's hash."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            i = src.find("\n", i)
            i = n if i < 0 else i
        elif src.startswith("/*", i):
            i = src.find("*/", i + 2)
            i = n if i < 0 else i + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(kernel: str) -> str:
    """Hash of a kernel's sources, code only: the key of the DRAM-traffic captures in profiles/."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "tile_scheduling_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def load_peaks():
    try:
        with open(PEAKS_PATH) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": FALLBACK_BF16_SUSTAINED, "source": "fallback"}


def load_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on the current kernel sources."""
    try:
        with open(TRAFFIC_PATH) as f:
            for line in f:
                if line.startswith("#") or not line.strip():
                    continue
                k, w, h, b = [x.strip() for x in line.split("|")[:4]]
                if k == kernel and w == workload and h == kernel_source_hash(kernel):
                    return float(b)
    except (OSError, ValueError):
        pass
    return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=5)
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts_, line in self.lines:
            if not (t0 <= ts_ <= t1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxes.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes), "reasons": sorted(reasons),
                "samples": len(sms)}


class NvmlLib:
    """Read-only NVML queries through the driver's libnvidia-ml (ctypes): SM clock, its maximum,
    power draw and the active clock-event reasons.  Nothing here changes a setting."""

    # nvmlClocksEventReasons bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}
    CLOCK_SM = 1

    def __init__(self, path: str = "libnvidia-ml.so.1"):
        import ctypes

        self.ct = ctypes
        self.lib = ctypes.CDLL(path)
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit_v2 failed")
        self._reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self._max = {}  # the maximum SM clock is fixed; its query takes ~1.5 ms, so it is asked once

    def handle(self, uuid: str | None, pci_bus_id: str | None, index: int):
        ct = self.ct
        h = ct.c_void_p()
        if uuid and self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ct.byref(h)) == 0:
            return h
        if pci_bus_id and self.lib.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ct.byref(h)) == 0:
            return h
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ct.c_uint(index), ct.byref(h)) == 0:
            return h
        raise OSError("no NVML handle for the device")

    def sample(self, h):
        """(sm_mhz, sm_max_mhz, power_w or None, reason bits)."""
        ct = self.ct
        clk, mw, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(h, self.CLOCK_SM, ct.byref(clk)) != 0:
            raise OSError("nvmlDeviceGetClockInfo failed")
        key = h.value
        if key not in self._max:
            mx = ct.c_uint()
            if self.lib.nvmlDeviceGetMaxClockInfo(h, self.CLOCK_SM, ct.byref(mx)) != 0:
                raise OSError("nvmlDeviceGetMaxClockInfo failed")
            self._max[key] = float(mx.value)
        power = float(mw.value) / 1e3 if self.lib.nvmlDeviceGetPowerUsage(h, ct.byref(mw)) == 0 else None
        bits = int(rs.value) if self._reasons(h, ct.byref(rs)) == 0 else 0
        return float(clk.value), self._max[key], power, bits


class NvmlClockSampler:
    """Samples the GPU's SM clock and clock-event reasons every `period_s` from a host thread, in
    process, through read-only NVML queries, so that even a timed region of a few milliseconds gets
    several samples.  `regions` collects (name, t0, t1) of the timed regions; `summary(name)` reduces
    the samples that fall inside one region (or all regions)."""

    def __init__(self, device: int = 0, period_s: float = 0.001, nvml=None):
        self.period = period_s
        self.samples = []  # (time, sm_mhz, sm_max_mhz, power_w, reason bits)
        self.regions = []
        self._stop = threading.Event()
        self._t = None
        self.error = None
        try:
            self.nvml = nvml if nvml is not None else NvmlLib()
            uuid = pci = None
            try:
                import torch

                prop = torch.cuda.get_device_properties(device)
                u = str(getattr(prop, "uuid", "") or "")
                uuid = (u if u.startswith("GPU-") else f"GPU-{u}") if u else None
                if hasattr(prop, "pci_bus_id"):
                    pci = f"{prop.pci_domain_id:08x}:{prop.pci_bus_id:02x}:{prop.pci_device_id:02x}.0"
            except Exception:  # noqa: BLE001 - a fake NVML needs no torch device
                pass
            self.h = self.nvml.handle(uuid, pci, device)
        except (OSError, AttributeError) as e:
            self.nvml = None
            self.error = str(e)

    def start(self):
        if self.nvml is None:
            return
        # the launching thread holds the interpreter for up to the switch interval
        # (5 ms by default) at a time: shorten it so the sampler keeps its period
        self._switch = sys.getswitchinterval()
        sys.setswitchinterval(min(self._switch, self.period / 4))
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()

    def _run(self):
        while not self._stop.is_set():
            try:
                self.samples.append((time.time(), *self.nvml.sample(self.h)))
            except OSError as e:
                self.error = str(e)
                return
            self._stop.wait(self.period)

    def stop(self):
        self._stop.set()
        if self._t:
            self._t.join(timeout=5)
            sys.setswitchinterval(self._switch)

    def region(self, name: str, t0: float, t1: float):
        self.regions.append((name, t0, t1))

    def summary(self, name: str | None = None):
        spans = [(a, b) for n, a, b in self.regions if name is None or n == name]
        sel = [s for s in self.samples if any(a <= s[0] <= b for a, b in spans)]
        out = {"source": "nvml, in process", "period_ms": round(self.period * 1e3, 2), "samples": len(sel)}
        if self.error:
            out["error"] = self.error
        if not sel:
            out.update(sm_mhz=None, sm_max_mhz=None, reasons=[])
            return out
        reasons = set()
        for s in sel:
            reasons.update(n for bit, n in NvmlLib.REASONS.items() if s[4] & bit)
        powers = [s[3] for s in sel if s[3] is not None]
        out.update(sm_mhz=statistics.median(s[1] for s in sel), sm_min_mhz=min(s[1] for s in sel),
                   sm_max_mhz=max(s[2] for s in sel), reasons=sorted(reasons),
                   power_w_max=round(max(powers), 1) if powers else None)
        return out


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_times(values, op: str):
    """Max (or sum) of per-rank floats over the default process group, or the values themselves alone."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return list(values)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor(values, dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return t.cpu().tolist()


# ------------------------------------------------------------ our GPU arm
def run_ours(args, ws, rank, local):
    import torch
    import torch.distributed as dist

    import tile_scheduling_gb300 as ts

    torch.cuda.set_device(local)
    w = synth.GEMM_8192
    M, N, K = w.M, w.N, w.K
    A_bits, B_bits = w.inputs()
    A = torch.from_numpy(A_bits.view(np.int16)).view(torch.bfloat16).cuda()
    B = torch.from_numpy(B_bits.view(np.int16)).view(torch.bfloat16).cuda()
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    n_copy = synth.COPY_N
    src = torch.from_numpy(synth.int16_uniform(synth.COPY_SEED, n_copy)).cuda()
    dst = torch.empty_like(src)
    stream = torch.cuda.current_stream()
    gemm_kw = dict(sched=args.sched, tile=args.tile)
    info = ts.ts_gemm_launch_info(M, N, K, ts.TS_OUT_BF16, args.sched, tile=args.tile)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        ts.ts_gemm_bf16_ex(A, B, D, stream=stream, **gemm_kw)
        if ev:
            ev[1].record(stream)
        ts.ts_copy_i16(src, dst, stream=stream)
        if ev:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ts.ts_sync_and_check()

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    outer0, outer1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = NvmlClockSampler(local)
    smi = None
    if sampler.nvml is None:  # no NVML in this process: fall back to nvidia-smi polling
        smi = ClockSampler(local)
        smi.start()
        time.sleep(0.3)
    sampler.start()
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    # a GPU sleep ahead of the region keeps the device busy while the host queues the
    # first steps, so the first GEMM's events do not count the host's submission time
    torch.cuda._sleep(4_000_000)
    outer0.record(stream)
    for i in range(args.steps):
        step(events[i])
    outer1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    sampler.region("headline", t0, t1)
    if ws > 1:
        dist.barrier()
    clocks = sampler.summary("headline") if smi is None else smi.stop(t0, t1)
    ts.ts_sync_and_check()

    gemm_ms = [e[0].elapsed_time(e[1]) for e in events]
    copy_ms = [e[1].elapsed_time(e[2]) for e in events]
    total_ms = outer0.elapsed_time(outer1)
    gemm_sum, copy_sum, total = reduce_times([sum(gemm_ms), sum(copy_ms), total_ms], "max")
    flops = 2.0 * M * N * K
    gemm_tflops = ws * flops * args.steps / (gemm_sum * 1e-3) / 1e12
    copy_bytes = 4.0 * n_copy
    copy_gbs = ws * copy_bytes * args.steps / (copy_sum * 1e-3) / 1e9

    # end-to-end through the public call with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, ts, A_bits, B_bits, M, N, K, ws)
    del A, B, D, src, dst
    torch.cuda.empty_cache()

    # the other GEMM workloads, each in its own timed region (rank 0 reports its own numbers)
    extra = {}
    if not args.no_configs:
        extra["gemm4096"] = measure_gemm4096(ts, sampler, reps=args.config_reps)
        extra["contended"] = measure_contended(ts, sampler, reps=max(10, args.reps), ctas=args.spin_ctas,
                                               tile=args.contended_tile, warmup=args.warmup)
        extra["smallk"] = measure_smallk(ts, sampler, samples=args.config_reps, warmup=args.warmup)
        extra["grouped"] = measure_grouped(ts, sampler, reps=args.config_reps)
    sampler.stop()
    if rank != 0:
        return None
    peaks = load_peaks()
    per_launch_s = gemm_sum * 1e-3 / args.steps
    achieved = flops / per_launch_s / 1e12
    workload = f"gemm_bf16 {M}x{N}x{K} bf16-out {args.tile} {args.sched} + copy_i16 n=2^28"
    # The burst figure is the peak for a GEMM timed in a short region; a region long enough to reach the
    # power cap (half a second or more, or the cap seen in the clock samples) takes the sustained one.
    capped = "sw_power_cap" in (clocks or {}).get("reasons", [])
    sustained = total / 1e3 >= 0.5 or capped
    peak = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
    kind = (f"{peaks['source']} bf16 sustained: the GEMM is timed in a region of {total / 1e3:.3f} s"
            + (" under the power cap" if capped else "") if sustained else
            f"{peaks['source']} bf16 burst: the GEMM is timed in a region of {total / 1e3:.3f} s, far shorter "
            "than the seconds-long loop of the sustained figure")
    roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak,
            "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
            "traffic": load_traffic("gemm", f"{M}x{N}x{K} {args.tile} {args.sched}"),
            "peak_kind": kind,
            "frac_of_burst": round(achieved / peaks["bf16_tflops"], 4), "peak_burst": peaks["bf16_tflops"],
            "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4),
            "peak_sustained": peaks["bf16_tflops_sustained"], "kernel": "gemm_ws_kernel",
            "algorithmic_flops_per_launch": flops}
    copy_roof = {"bound": "hbm", "achieved": round(copy_gbs / ws, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                 "frac": round(copy_gbs / ws / peaks["hbm_gbs"], 4), "traffic": load_traffic("copy", "n=2^28"),
                 "peak_kind": f"{peaks['source']} HBM copy", "kernel": "copy_i16_vec_kernel",
                 "algorithmic_bytes_per_launch": copy_bytes}
    line = {
        "metric": "bf16 GEMM TFLOP/s at 8192^3 (2-CTA 256x256, CLC); int16 copy HBM GB/s",
        "value": round(gemm_tflops, 2), "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload, "M": M, "N": N, "K": K, "out": "bf16", "tile": args.tile,
                   "sched": args.sched, "tiles": info["num_tiles"], "grid_ctas": info["grid_ctas"],
                   "stages": info["stages"], "epi_warps": info["epi_warps"], "copy_n": n_copy,
                   "l2": "inputs larger than L2 (256 MiB GEMM operands, 1 GiB copy traffic); no flush",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "seeds": {"A": hex(w.seed_a), "B": hex(w.seed_b), "copy": hex(synth.COPY_SEED)},
                   "gpu": torch.cuda.get_device_name(local), "sms": torch.cuda.get_device_properties(local).multi_processor_count},
        "gemm": {"tflops": round(gemm_tflops, 2), "ms_median": round(statistics.median(gemm_ms), 4),
                 "ms_min": round(min(gemm_ms), 4)},
        "copy": {"gbs": round(copy_gbs, 1), "ms_median": round(statistics.median(copy_ms), 4),
                 "roofline": copy_roof},
        "roofline": roof,
        "clocks": clocks,
        "gpu_launches": 2 * args.steps,
        "e2e": e2e,
        **extra,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args)
    return line


def _event_ms(fn, stream, sleep_cycles=500_000):
    """Device time of fn's launches on `stream` (CUDA events).

    A short GPU sleep queued ahead of the start event keeps the device busy
    while the host runs fn's Python and C setup, so that host overhead does not
    fall inside the timed region (otherwise an idle GPU records the start event
    at once and the gap until the launch is counted)."""
    import torch

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if sleep_cycles:
        torch.cuda._sleep(sleep_cycles)
    e0.record(stream)
    fn()
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1)


def _dev_bf16(bits):
    import torch

    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def _batched_ms(fns, reps, batch, stream, sampler=None, region=None, sleep_cycles=2_000_000):
    """Per-launch device time of each fn(i) in `fns`: `reps` samples, each `batch` calls queued back to
    back (i = 0, 1, ...) between two CUDA events on `stream`, behind a GPU sleep that covers the host's
    submission work; the configurations alternate so that clock drift reaches all of them alike.
    Returns {name: [ms per launch, one per sample]}."""
    import torch

    out = {k: [] for k in fns}
    for _ in range(reps):
        for k, f in fns.items():
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(sleep_cycles)
            e0.record(stream)
            t0 = time.time()
            for i in range(batch):
                f(i)
            e1.record(stream)
            e1.synchronize()
            if sampler is not None:
                sampler.region(region or k, t0, time.time())
            out[k].append(e0.elapsed_time(e1) / batch)
    return out


def measure_grouped(ts, sampler, reps=7, batch=5):
    """The grouped GEMM whose 16 groups of 2048 x 2048 differ in K (64 .. 8192, skewed), the groups
    scheduled longest K first, under the static persistent and the CLC scheduler (samples alternated).
    Each launch reads 624 MB of A and B, more than L2 holds, so no launch finds its operands there."""
    import torch

    w = synth.GROUPED
    off = w.k_offsets()
    A_bits, B_bits = w.inputs()
    A, B = _dev_bf16(A_bits), _dev_bf16(B_bits)
    D = torch.empty((w.groups, w.M, w.N), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    fns = {sched: (lambda i, sc=sched: ts.ts_gemm_bf16_grouped(A, B, D, off, sched=sc)) for sched in ("static", "clc")}
    for f in fns.values():
        for i in range(3):
            f(i)
    ms = _batched_ms(fns, reps, batch, stream, sampler, "grouped")
    ts.ts_sync_and_check()
    flops = 2.0 * w.M * w.N * off[-1]
    peak = load_peaks()["bf16_tflops"]
    runs = {}
    for sched, v in ms.items():
        med = statistics.median(v)
        runs[sched] = {"us_median": round(med * 1e3, 2), "us_min": round(min(v) * 1e3, 2),
                       "tflops": round(flops / (med * 1e-3) / 1e12, 1),
                       "frac_of_burst": round(flops / (med * 1e-3) / 1e12 / peak, 4)}
    del A, B, D
    torch.cuda.empty_cache()
    return {"metric": "grouped bf16 GEMM TFLOP/s, 16 groups of 2048x2048, K per group 64..8192 (skewed)",
            "unit": "TFLOP/s", "value": max(r["tflops"] for r in runs.values()), "runs": runs,
            "clc_speedup_over_static": round(runs["static"]["us_median"] / runs["clc"]["us_median"], 3),
            "order": "groups longest K first (ts_gemm_grouped_order)", "k_offsets": off,
            "samples": f"{reps} x {batch} back-to-back launches per scheduler, alternated"}


def measure_gemm4096(ts, sampler, reps=5, batch=20, nset=4):
    """4096^3 bf16-out GEMM, uniform [-1, 1] inputs: the automatic tile choice and the 128x256 tile, each
    under the static persistent and the CLC scheduler.  The launches of a sample run back to back over
    `nset` input/output buffer sets used in turn (4 x 96 MiB, larger than L2), so no launch finds its
    operands in L2 from the launch before."""
    import torch

    w = synth.GEMM_4096
    A_bits, B_bits = w.inputs()
    As = [_dev_bf16(A_bits) for _ in range(nset)]
    Bs = [_dev_bf16(B_bits) for _ in range(nset)]
    Ds = [torch.empty((w.M, w.N), dtype=torch.bfloat16, device="cuda") for _ in range(nset)]
    stream = torch.cuda.current_stream()
    runs = {}
    for ready in (0, 1):
        for tile in ("auto", "128x256"):
            for sched in ("static", "clc"):
                runs[f"{tile} {sched}" + (" inputs_ready" if ready else "")] = (
                    lambda i, tile=tile, sched=sched, ready=ready:
                    ts.ts_gemm_bf16_ex(As[i % nset], Bs[i % nset], Ds[i % nset], sched=sched, tile=tile,
                                       inputs_ready=ready))
    # the non-persistent shape: one cluster per work unit, each computing its unit and exiting
    runs["auto nonpersistent"] = (lambda i: ts.ts_gemm_bf16_ex(As[i % nset], Bs[i % nset], Ds[i % nset],
                                                               sched="nonpersistent", tile="auto"))
    for f in runs.values():
        for i in range(2 * nset):
            f(i)
    torch.cuda.synchronize()
    ts.ts_sync_and_check()
    times = _batched_ms(runs, reps, batch, stream, sampler, "gemm4096")
    ts.ts_sync_and_check()
    peaks = load_peaks()
    flops = 2.0 * w.M * w.N * w.K
    res = {}
    for k, v in times.items():
        tile, sched = k.split()[:2]
        ready = k.endswith("inputs_ready")
        med = statistics.median(v)
        info = ts.ts_gemm_launch_info(w.M, w.N, w.K, ts.TS_OUT_BF16, sched, tile=tile)
        tf = flops / (med * 1e-3) / 1e12
        res[k] = {"tile": f"{info['tile_m']}x{info['tile_n']}" + (" 2-CTA" if info["cluster"] == 2 else ""),
                  "sched": sched, "inputs_ready": int(ready), "us_median": round(med * 1e3, 2),
                  "us_min": round(min(v) * 1e3, 2), "tflops": round(tf, 1),
                  "frac_of_burst": round(tf / peaks["bf16_tflops"], 4),
                  "split_tail": f"{info['split_tiles']} tiles x {info['split_parts']} parts",
                  "stages": info["stages"], "epi_warps": info["epi_warps"],
                  # DRAM bytes of one launch: the captures ran the default mode, whose work is the same
                  "traffic": load_traffic("gemm", f"{w.M}x{w.N}x{w.K} {tile} {sched}")}
    autos = [k for k in res if k.startswith("auto")]
    best_auto = max(autos, key=lambda k: res[k]["tflops"])
    best_default = max(("auto static", "auto clc"), key=lambda k: res[k]["tflops"])
    return {"metric": "bf16 GEMM TFLOP/s, 4096^3 bf16-out, static vs CLC (and non-persistent), automatic tile and 128x256",
            "unit": "TFLOP/s", "value": res[best_auto]["tflops"], "frac_of_burst": res[best_auto]["frac_of_burst"],
            "reported": best_auto,
            "value_default_mode": res[best_default]["tflops"],
            "frac_of_burst_default_mode": res[best_default]["frac_of_burst"],
            "reported_default_mode": best_default,
            "inputs_ready": "runs marked inputs_ready pass that option (A and B were final before the previous "
                            "launch began, which holds here: nothing writes them), so their loads overlap the "
                            "previous launch's tail; the other runs wait for the previous launch first",
            "runs": res, "peak": peaks["bf16_tflops"],
            "peak_kind": f"{peaks['source']} bf16 burst", "samples": reps, "launches_per_sample": batch,
            "gpu_launches": reps * batch * len(runs),
            "clocks": sampler.summary("gemm4096") if sampler is not None else None,
            "config": {"workload": w.name, "l2": f"{nset} buffer sets of A, B, D used in turn ({nset} x 96 MiB, "
                                                  "larger than L2); launches back to back"}}


def run_gemm4096(args, ws, rank, local):
    """4096^3 bf16-out GEMM, static persistent vs CLC, automatic tile and 128x256."""
    import torch

    import tile_scheduling_gb300 as ts

    torch.cuda.set_device(local)
    sampler = NvmlClockSampler(local)
    sampler.start()
    line = measure_gemm4096(ts, sampler, reps=args.steps)
    sampler.stop()
    if rank != 0:
        return None
    return {**line, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "dtype": "bf16", "data": "synthetic"}


def run_grouped(args, ws, rank, local):
    """Grouped GEMM whose 16 groups differ in K (64..8192, skewed): static persistent vs CLC."""
    import torch

    import tile_scheduling_gb300 as ts

    torch.cuda.set_device(local)
    w = synth.GROUPED
    off = w.k_offsets()
    A_bits, B_bits = w.inputs()
    A = torch.from_numpy(A_bits.view(np.int16)).view(torch.bfloat16).cuda()
    B = torch.from_numpy(B_bits.view(np.int16)).view(torch.bfloat16).cuda()
    D = torch.empty((w.groups, w.M, w.N), dtype=torch.bfloat16, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    flops = 2.0 * w.M * w.N * off[-1]
    res = {}
    times = {"static": [], "clc": []}
    for sched in times:
        for _ in range(args.warmup):
            ts.ts_gemm_bf16_grouped(A, B, D, off, sched=sched, tile=args.tile)
    for _ in range(args.steps):  # alternate so clock drift hits both alike
        for sched in times:
            flush.zero_()
            times[sched].append(_event_ms(lambda: ts.ts_gemm_bf16_grouped(A, B, D, off, sched=sched, tile=args.tile),
                                          stream))
    ts.ts_sync_and_check()
    for sched, v in times.items():
        med = statistics.median(v)
        res[sched] = {"ms_median": round(med, 4), "ms_min": round(min(v), 4),
                      "tflops": round(flops / (med * 1e-3) / 1e12, 1)}
    if rank != 0:
        return None
    return {"metric": "grouped bf16 GEMM TFLOP/s, 16 groups of 2048x2048, K per group 64..8192 (skewed)",
            "unit": "TFLOP/s", "value": res["clc"]["tflops"], "static": res["static"], "clc": res["clc"],
            "clc_speedup_over_static": round(res["static"]["ms_median"] / res["clc"]["ms_median"], 3),
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "dtype": "bf16",
            "data": "synthetic", "config": {"workload": w.name, "k_offsets": off, "tile": args.tile,
                                            "l2": "256 MiB buffer written between launches"}}


def run_causal(args, ws, rank, local):
    """8192^3 bf16 GEMM with every output tile strictly above the diagonal skipped (a causal,
    block-sparse output): static persistent vs CLC, counting only the computed tiles' flops."""
    import torch

    import tile_scheduling_gb300 as ts

    torch.cuda.set_device(local)
    w = synth.GEMM_8192
    A_bits, B_bits = w.inputs()
    A = torch.from_numpy(A_bits.view(np.int16)).view(torch.bfloat16).cuda()
    B = torch.from_numpy(B_bits.view(np.int16)).view(torch.bfloat16).cuda()
    D = torch.zeros((w.M, w.N), dtype=torch.bfloat16, device="cuda")
    info = ts.ts_gemm_launch_info(w.M, w.N, w.K, ts.TS_OUT_BF16, "static", tile=args.tile, workspace=None)
    tm, tn, TM, TN = info["tile_m"], info["tile_n"], info["tiles_m"], info["tiles_n"]
    mb = np.arange(TM)[:, None]
    nb = np.arange(TN)[None, :]
    mask_np = (nb * tn > mb * tm + tm - 1).astype(np.uint8)
    mask = torch.from_numpy(mask_np.reshape(-1)).cuda()
    computed = int((mask_np == 0).sum())
    flops = 2.0 * tm * tn * w.K * computed
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    times = {"static": [], "clc": []}
    kw = dict(tile=args.tile, workspace=None, skip_tiles=mask)
    for sched in times:
        for _ in range(args.warmup):
            ts.ts_gemm_bf16_ex(A, B, D, sched=sched, **kw)
    for _ in range(args.steps):
        for sched in times:
            flush.zero_()
            times[sched].append(_event_ms(lambda: ts.ts_gemm_bf16_ex(A, B, D, sched=sched, **kw), stream))
    ts.ts_sync_and_check()
    res = {}
    for sched, v in times.items():
        med = statistics.median(v)
        res[sched] = {"ms_median": round(med, 4), "ms_min": round(min(v), 4),
                      "tflops": round(flops / (med * 1e-3) / 1e12, 1)}
    if rank != 0:
        return None
    return {"metric": "causal 8192^3 bf16 GEMM TFLOP/s (tiles above the diagonal skipped; computed tiles only)",
            "unit": "TFLOP/s", "value": res["clc"]["tflops"], "static": res["static"], "clc": res["clc"],
            "clc_speedup_over_static": round(res["static"]["ms_median"] / res["clc"]["ms_median"], 3),
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "dtype": "bf16",
            "data": "synthetic", "config": {"workload": "causal " + w.name, "tile": args.tile,
                                            "tiles_computed": computed, "tiles_skipped": int(mask_np.sum()),
                                            "l2": "256 MiB buffer written between launches"}}


def run_fork(args, ws, rank, local):
    """8192^3 bf16 GEMM with the Fork's second consumer (row sums of A) vs without, 1-CTA 128x256 tiles."""
    import torch

    import tile_scheduling_gb300 as ts

    torch.cuda.set_device(local)
    w = synth.GEMM_8192
    A_bits, B_bits = w.inputs()
    A = torch.from_numpy(A_bits.view(np.int16)).view(torch.bfloat16).cuda()
    B = torch.from_numpy(B_bits.view(np.int16)).view(torch.bfloat16).cuda()
    D = torch.empty((w.M, w.N), dtype=torch.bfloat16, device="cuda")
    R = torch.empty((w.M,), dtype=torch.float32, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    kw = dict(sched=args.sched, tile="128x256", workspace=None)
    fns = {"plain": lambda: ts.ts_gemm_bf16_ex(A, B, D, **kw),
           "fork_row_sums": lambda: ts.ts_gemm_bf16_ex(A, B, D, row_sums=R, **kw)}
    for f in fns.values():
        for _ in range(args.warmup):
            f()
    times = {k: [] for k in fns}
    for _ in range(args.steps):
        for k, f in fns.items():
            flush.zero_()
            times[k].append(_event_ms(f, stream))
    ts.ts_sync_and_check()
    flops = 2.0 * w.M * w.N * w.K
    res = {k: {"ms_median": round(statistics.median(v), 4),
               "tflops": round(flops / (statistics.median(v) * 1e-3) / 1e12, 1)} for k, v in times.items()}
    if rank != 0:
        return None
    return {"metric": "8192^3 bf16 GEMM TFLOP/s with the Fork row-sum consumer vs without (128x256)",
            "unit": "TFLOP/s", "value": res["fork_row_sums"]["tflops"], **res,
            "fork_overhead": round(res["fork_row_sums"]["ms_median"] / res["plain"]["ms_median"] - 1, 4),
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "dtype": "bf16",
            "data": "synthetic", "config": {"workload": w.name + " (128x256, " + args.sched + ")",
                                            "l2": "256 MiB buffer written between launches"}}


def run_rows(args, ws, rank, local):
    """Jagged int16 copy, 8192 rows of 64..262144 elements (log-uniform): the static grid-stride work
    queue vs the CLC one, plus an oversubscribed CLC launch (twice as many tiles as rows, the extra
    half skipped).  Inputs (0.5 GiB each way) are larger than L2."""
    import torch

    import tile_scheduling_gb300 as ts

    torch.cuda.set_device(local)
    w = synth.ROWS
    src_h, off_h = w.inputs()
    src = torch.from_numpy(src_h).cuda()
    dst = torch.empty_like(src)
    off = torch.from_numpy(off_h).cuda()
    stream = torch.cuda.current_stream()
    nbytes = 4.0 * src.numel()  # 2 bytes read + 2 written per element
    runs = {"static": dict(sched="static"), "clc": dict(sched="clc"), "nonpersistent": dict(sched="nonpersistent"),
            "clc_oversubscribed_2x": dict(sched="clc", tiles=2 * w.rows)}
    # chunked mode: rows cut into work tiles of at most `chunk` elements (a planning kernel maps tiles to
    # rows); packed mode: the rows laid end to end, every tile `chunk` of their elements
    for sched in ("clc", "static"):
        for pack in (0, 1):
            for chunk in (16384, 32768, 65536):
                need = ts.ts_copy_rows_launch_info(src.numel(), w.rows, sched, chunk=chunk,
                                                   pack=pack)["workspace_bytes"]
                runs[f"{sched}_{'packed' if pack else 'chunk'}_{chunk // 1024}k"] = dict(
                    sched=sched, chunk=chunk, pack=pack, workspace=torch.empty(need, dtype=torch.uint8, device="cuda"))
    need = ts.ts_copy_rows_launch_info(src.numel(), w.rows, "nonpersistent", chunk=32768)["workspace_bytes"]
    runs["nonpersistent_chunk_32k"] = dict(sched="nonpersistent", chunk=32768,
                                           workspace=torch.empty(need, dtype=torch.uint8, device="cuda"))
    times = {k: [] for k in runs}
    for k, kw in runs.items():
        for _ in range(args.warmup):
            ts.ts_copy_i16_rows(src, dst, off, **kw)
    for _ in range(args.steps):  # alternate so clock drift hits every variant alike
        for k, kw in runs.items():
            times[k].append(_event_ms(lambda: ts.ts_copy_i16_rows(src, dst, off, **kw), stream))
    ts.ts_sync_and_check()
    if not torch.equal(dst, src):
        raise RuntimeError("jagged copy result differs from its input")
    if rank != 0:
        return None
    peaks = load_peaks()
    res = {}
    for k, v in times.items():
        med = statistics.median(v)
        res[k] = {"ms_median": round(med, 4), "ms_min": round(min(v), 4),
                  "gbs": round(nbytes / (med * 1e-3) / 1e9, 1)}
    head = max(res, key=lambda k: res[k]["gbs"])  # the fastest configuration, named in config
    best = res[head]["gbs"]
    chunk = runs[head].get("chunk", 0)
    pack = runs[head].get("pack", 0)
    return {"metric": "jagged int16 row copy HBM GB/s (8192 rows, log-uniform lengths), static vs CLC work queue "
                      "(and non-persistent)",
            "unit": "GB/s", "value": best, **res,
            "clc_speedup_over_static": round(res["static"]["ms_median"] / res["clc"]["ms_median"], 3),
            "roofline": {"bound": "hbm", "achieved": best, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(best / peaks["hbm_gbs"], 4),
                         "traffic": load_traffic("rows", f"8192 rows log-uniform {runs[head]['sched']} "
                                                         f"{'packed' if pack else 'chunk'} {chunk}"),
                         "peak_kind": f"{peaks['source']} HBM copy", "kernel": "rows_copy_kernel"},
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "dtype": "int16",
            "data": "synthetic", "config": {"workload": w.name, "elements": int(src.numel()), "rows": w.rows,
                                            "reported": head, "sched": runs[head]["sched"], "chunk": chunk,
                                            "pack": pack,
                                            "l2": "inputs larger than L2 (0.5 GiB each way); no flush"}}


def measure_smallk(ts, sampler, samples=20, warmup=5, batch=25):
    """8192x8192x64 bf16-out GEMM: one k-block per tile, so the 134 MB output write bounds it (HBM GB/s).
    Both schedulers on the 2-CTA 256x256 tile and on the 1-CTA 128x256 tile, samples alternated; a
    sample is `batch` launches back to back (a launch takes ~25 us, close to the event timer's grain)."""
    import torch

    w = synth.GEMM_SMALLK
    A_bits, B_bits = w.inputs()
    A, B = _dev_bf16(A_bits), _dev_bf16(B_bits)
    D = torch.empty((w.M, w.N), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    nbytes = 2.0 * (w.M * w.K + w.N * w.K) + 2.0 * w.M * w.N  # A and B read once, D written once
    runs = {f"{sched} {tile}" + (" inputs_ready" if ready else ""):
            (lambda i, sched=sched, tile=tile, ready=ready:
             ts.ts_gemm_bf16_ex(A, B, D, sched=sched, tile=tile, inputs_ready=ready))
            for ready in (0, 1) for tile in ("256x256", "128x256") for sched in ("clc", "static")}
    runs["nonpersistent 128x256"] = lambda i: ts.ts_gemm_bf16_ex(A, B, D, sched="nonpersistent", tile="128x256")
    for f in runs.values():
        for i in range(warmup):
            f(i)
    torch.cuda.synchronize()
    times = _batched_ms(runs, samples, batch, stream, sampler, "smallk", sleep_cycles=4_000_000)
    ts.ts_sync_and_check()
    peaks = load_peaks()
    res = {}
    for k, v in times.items():
        med = statistics.median(v)
        res[k] = {"inputs_ready": int(k.endswith("inputs_ready")), "us_median": round(med * 1e3, 2),
                  "us_min": round(min(v) * 1e3, 2), "gbs": round(nbytes / (med * 1e-3) / 1e9, 1),
                  "frac_of_hbm": round(nbytes / (med * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                  "tflops": round(2.0 * w.M * w.N * w.K / (med * 1e-3) / 1e12, 1)}
    head = max(res, key=lambda k: res[k]["gbs"])  # the fastest configuration, named in config
    h_sched, h_tile = head.split()[:2]
    best = res[head]["gbs"]
    head_default = max((k for k in res if not res[k]["inputs_ready"]), key=lambda k: res[k]["gbs"])
    return {"metric": "small-K bf16 GEMM HBM GB/s (8192x8192x64, bf16 out)", "unit": "GB/s", "value": best,
            "frac_of_hbm": round(best / peaks["hbm_gbs"], 4), "reported": head,
            "value_default_mode": res[head_default]["gbs"], "frac_of_hbm_default_mode": res[head_default]["frac_of_hbm"],
            "reported_default_mode": head_default,
            "inputs_ready": "runs marked inputs_ready pass that option (A and B were final before the previous "
                            "launch began, which holds here: nothing writes them), so their loads and MMAs "
                            "overlap the previous launch's tail; the other runs wait for the previous launch first",
            "runs": res,
            "roofline": {"bound": "hbm", "achieved": best, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(best / peaks["hbm_gbs"], 4),
                         "traffic": load_traffic("gemm", f"{w.M}x{w.N}x{w.K} {h_tile} {h_sched}"),
                         "peak_kind": f"{peaks['source']} HBM copy", "kernel": "gemm_ws_kernel",
                         "algorithmic_bytes_per_launch": int(nbytes)},
            "samples": samples, "launches_per_sample": batch, "gpu_launches": samples * batch * len(runs),
            "clocks": sampler.summary("smallk") if sampler is not None else None,
            "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "tile": h_tile, "sched": h_sched,
                       "inputs_ready": res[head]["inputs_ready"],
                       "epi_warps": ts.ts_gemm_launch_info(w.M, w.N, w.K, ts.TS_OUT_BF16, h_sched,
                                                           tile=h_tile)["epi_warps"],
                       "l2": "output (134 MB) larger than L2; A and B (1 MiB each) stay resident; no flush"}}


def run_ingress(args, ws, rank, local):
    """How fast one SM takes in operands: the 8192^3 GEMM under the static scheduler with a cap on the
    persistent workers, 1-CTA 128x256 and 2-CTA 256x256 tiles, no split tiles.  From the kernel's
    per-unit trace, each worker's tile period (the median gap between the ends of its consecutive
    tiles) gives the tensor rate per SM; the clock samples of each run are reported beside it.  If
    the rate of the 1-CTA tile were bound by something the SMs share (L2, the crossbar), it would
    rise as fewer SMs run; if it is bound per SM, it rises only as much as the clock does."""
    import torch

    import tile_scheduling_gb300 as ts

    torch.cuda.set_device(local)
    sampler = NvmlClockSampler(local)
    sampler.start()
    w = synth.GEMM_8192
    A_bits, B_bits = w.inputs()
    A, B = _dev_bf16(A_bits), _dev_bf16(B_bits)
    D = torch.empty((w.M, w.N), dtype=torch.bfloat16, device="cuda")
    sms = ts.ts_num_sms()
    runs = {}
    for tile, cg, counts in (("128x256", 1, (sms, 3 * sms // 4, sms // 2, sms // 4, sms // 8)),
                             ("256x256", 2, (sms // 2, 3 * sms // 8, sms // 4, sms // 8))):
        for workers in counts:
            kw = dict(sched="static", tile=tile, max_workers=workers, workspace=None)
            info = ts.ts_gemm_launch_info(w.M, w.N, w.K, ts.TS_OUT_BF16, **kw)
            trace = torch.zeros(4 * info["num_units"], dtype=torch.int64, device="cuda")
            for _ in range(max(1, args.warmup // 3)):
                ts.ts_gemm_bf16_ex(A, B, D, **kw)
            torch.cuda.synchronize()
            t0 = time.time()
            ts.ts_gemm_bf16_ex(A, B, D, trace=trace, **kw)
            torch.cuda.synchronize()
            sampler.region(f"{tile} {workers}", t0, time.time())
            ts.ts_sync_and_check()
            tr = trace.view(-1, 4).cpu().numpy()
            ends = {}
            for u in range(info["num_units"]):
                ends.setdefault(int(tr[u, 1]), []).append(int(tr[u, 3]))
            gaps = [g for e in ends.values() for g in np.diff(np.sort(np.array(e))).tolist()]
            period_us = statistics.median(gaps) / 1e3
            tile_flops = 2.0 * info["tile_m"] * info["tile_n"] * w.K
            clk = sampler.summary(f"{tile} {workers}")
            runs[f"{tile} x{workers}"] = {
                "tile": tile, "workers": workers, "sms": workers * cg, "tile_period_us": round(period_us, 2),
                "tflops_per_sm": round(tile_flops / cg / (period_us * 1e-6) / 1e12, 2),
                "sm_mhz": clk.get("sm_mhz"), "reasons": clk.get("reasons")}
    sampler.stop()
    if rank != 0:
        return None
    return {"metric": "operand ingress per SM: tensor TFLOP/s per SM of the 8192^3 GEMM vs the SMs in use",
            "unit": "TFLOP/s per SM", "value": runs[f"128x256 x{sms}"]["tflops_per_sm"], "runs": runs,
            "n_gpus": ws, "steps": 1, "warmup": args.warmup, "higher_is_better": True, "dtype": "bf16",
            "data": "synthetic", "config": {"workload": w.name + " static, capped workers, no split tiles",
                                            "flop_per_sm_cycle": 8192}}


def run_smallk(args, ws, rank, local):
    """8192x8192x64 bf16-out GEMM in HBM GB/s."""
    import torch

    import tile_scheduling_gb300 as ts

    torch.cuda.set_device(local)
    sampler = NvmlClockSampler(local)
    sampler.start()
    line = measure_smallk(ts, sampler, samples=args.steps, warmup=args.warmup)
    sampler.stop()
    if rank != 0:
        return None
    return {**line, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "dtype": "bf16", "data": "synthetic"}


def measure_contended(ts, sampler, reps=10, ctas=32, tile="256x256", warmup=5):
    """Ragged 8191x6143x4096 fp32-out GEMM while a spin kernel on a second stream holds `ctas` SMs for
    half the solo static GEMM time.  Static persistent vs CLC in `reps` alternating pairs (a fresh spin
    per run); a traced run per scheduler gives the tail (the last worker's finish minus the median
    worker's finish)."""
    import torch

    w = synth.GEMM_RAGGED
    A_bits, B_bits = w.inputs()
    A, B = _dev_bf16(A_bits), _dev_bf16(B_bits)
    Dbuf = torch.empty((w.M, 6144), dtype=torch.float32, device="cuda")
    D = Dbuf[:, :w.N]  # 6144-element pitch: TMA stores, masked at N = 6143
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    started = torch.zeros(1, dtype=torch.int32).pin_memory()

    def gemm(sched, trace=None):
        ts.ts_gemm_bf16_ex(A, B, D, sched=sched, tile=tile, trace=trace)

    solo = {}
    for sched in ("static", "clc"):
        for _ in range(warmup):
            gemm(sched)
        solo[sched] = statistics.median([_event_ms(lambda: gemm(sched), stream) for _ in range(reps)])
    # half the solo time from the GEMM's start, plus the ~30 us of sleep queued ahead of it
    spin_ns = int(0.5 * solo["static"] * 1e6) + 30_000

    def contended(sched, trace=None):
        started.zero_()
        torch.cuda.synchronize()
        ts.ts_spin(ctas, spin_ns, started, stream=side)
        ts.ts_spin_wait_started(started, ctas, 5.0)
        # a short sleep only (~30 us): it hides the host's launch work, and the GEMM
        # still starts while the spin holds its SMs for most of its time
        t0 = time.time()
        ms = _event_ms(lambda: gemm(sched, trace), stream, sleep_cycles=60_000)
        if sampler is not None:
            sampler.region("contended", t0, time.time())
        torch.cuda.synchronize()
        return ms

    times = {"static": [], "clc": []}
    for _ in range(reps):
        for sched in ("static", "clc"):
            times[sched].append(contended(sched))
    tails = {}
    for sched in ("static", "clc"):
        info = ts.ts_gemm_launch_info(w.M, w.N, w.K, ts.TS_OUT_F32, sched, tile=tile, ldd=6144)
        trace = torch.zeros(4 * info["num_units"], dtype=torch.int64, device="cuda")
        contended(sched, trace)
        tr = trace.view(-1, 4).cpu().numpy()
        t0 = tr[:, 2].min()
        fin = {}
        for t in range(tr.shape[0]):
            fin[int(tr[t, 1])] = max(fin.get(int(tr[t, 1]), 0), int(tr[t, 3]))
        f = np.array(sorted(fin.values()), dtype=np.float64)
        tails[sched] = {"workers_ran": len(fin), "tail_us": round((f.max() - np.median(f)) / 1e3, 1),
                        "span_us": round((f.max() - t0) / 1e3, 1), "visits_ok": bool(np.all(tr[:, 0] == 1))}
    ts.ts_sync_and_check()
    flops = 2.0 * w.M * w.N * w.K
    out = {}
    for sched in ("static", "clc"):
        med = statistics.median(times[sched])
        out[sched] = {"ms_median": round(med, 4), "ms_min": round(min(times[sched]), 4),
                      "tflops": round(flops / (med * 1e-3) / 1e12, 1), "solo_ms": round(solo[sched], 4),
                      "solo_tflops": round(flops / (solo[sched] * 1e-3) / 1e12, 1), **tails[sched]}
    return {"metric": "ragged 8191x6143x4096 fp32-out GEMM TFLOP/s with 32 SMs held for half the solo time",
            "unit": "TFLOP/s", "value": out["clc"]["tflops"], "static": out["static"], "clc": out["clc"],
            "clc_speedup_over_static": round(out["static"]["ms_median"] / out["clc"]["ms_median"], 3),
            "clc_tail_shorter": bool(out["clc"]["tail_us"] < out["static"]["tail_us"]),
            "pairs": reps, "gpu_launches": 2 * reps + 2,
            "clocks": sampler.summary("contended") if sampler is not None else None,
            "config": {"workload": w.name, "tile": tile, "spin_ctas": ctas, "spin_ns": spin_ns, "ldd": 6144,
                       "l2": "inputs larger than L2 (A 67 MB, B 50 MB, D 201 MB); one launch per timed region"}}


def run_contended(args, ws, rank, local):
    """Ragged 8191x6143x4096 fp32-out GEMM with 32 SMs held: static persistent vs CLC."""
    import torch

    import tile_scheduling_gb300 as ts

    torch.cuda.set_device(local)
    sampler = NvmlClockSampler(local)
    sampler.start()
    line = measure_contended(ts, sampler, reps=args.reps, ctas=args.spin_ctas, tile=args.tile, warmup=args.warmup)
    sampler.stop()
    if rank != 0:
        return None
    return {**line, "n_gpus": ws, "higher_is_better": True, "dtype": "bf16", "data": "synthetic"}


def run_e2e(args, ts, A_bits, B_bits, M, N, K, ws):
    """The GEMM through the public call on host buffers, copies inside the timed region.

    Every step is one ts_gemm_bf16_host call: it copies A and B from pinned host memory into
    device buffers, runs the GEMM and copies D back to pinned host memory, all on one stream.
    Consecutive steps go round-robin to three streams, each with its own device buffers, so one
    step's copies overlap the others' GEMMs and copies."""
    import torch

    nbuf = 3
    A_h = torch.from_numpy(A_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    B_h = torch.from_numpy(B_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    D_h = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(nbuf)]
    A = [torch.empty((M, K), dtype=torch.bfloat16, device="cuda") for _ in range(nbuf)]
    B = [torch.empty((N, K), dtype=torch.bfloat16, device="cuda") for _ in range(nbuf)]
    D = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(nbuf)]
    streams = [torch.cuda.Stream() for _ in range(nbuf)]
    # calls on different streams overlap, so each stream gets its own split-tile workspace (zeroed)
    need = ts.ts_gemm_launch_info(M, N, K, ts.TS_OUT_BF16, args.sched, tile=args.tile,
                                  workspace=None)["workspace_bytes"]
    wsp = [torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda") for _ in range(nbuf)]

    def step(i):
        b = i % nbuf
        ts.ts_gemm_bf16_host(A_h, B_h, D_h[b], A[b], B[b], D[b], sched=args.sched, tile=args.tile,
                             workspace=wsp[b], stream=streams[b])

    for i in range(nbuf):
        step(i)
    torch.cuda.synchronize()
    steps = max(3, min(args.steps, args.e2e_steps))
    # three timed regions of `steps` steps each; the median region is reported (the host submits
    # every step, so a region also shows any stall of the host that drives it)
    regions = []
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(streams[0])
        for st in streams[1:]:
            st.wait_event(e0)
        for i in range(steps):
            step(i)
        for st in streams[1:]:
            streams[0].wait_stream(st)
        e1.record(streams[0])
        torch.cuda.synchronize()
        regions.append(e0.elapsed_time(e1))
    ms = reduce_times([statistics.median(regions)], "max")[0]
    ts.ts_sync_and_check()
    flops = 2.0 * M * N * K
    h2d = int(A_h.numel() * 2 + B_h.numel() * 2)
    d2h = int(D_h[0].numel() * 2)
    link = measure_host_link(A_h, B_h, D_h[0], A[0], B[0], D[0], streams[0], streams[1])
    host_gbs = (h2d + d2h) * steps / (ms * 1e-3) / 1e9
    return {"value": round(ws * flops * steps / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps, "ms_per_step": round(ms / steps, 4), "call": "ts_gemm_bf16_host",
            "regions_ms": [round(r, 3) for r in regions], "reported": "the median of the three regions",
            "pipelining": f"one call per step (copy in, GEMM, copy out on one stream); steps round-robin over "
                          f"{nbuf} streams and buffer sets",
            "roofline": {"bound": "host link", "achieved": round(host_gbs, 1), "peak": link["both_gbs"],
                         "unit": "GB/s", "frac": round(host_gbs / link["both_gbs"], 4),
                         "peak_kind": "measured here: the step's copies alone (A and B in on one stream, D out on "
                                      "another, at once), no GEMM",
                         "link": link}}


def measure_host_link(A_h, B_h, D_h, A, B, D, s_in, s_out, reps=5):
    """Host link rates on this machine for the end-to-end step's own copies, with no GEMM running:
    A and B in, D out, and both directions at once on two streams (median of `reps`)."""
    import torch

    h2d = (A_h.numel() + B_h.numel()) * A_h.element_size()
    d2h = D_h.numel() * D_h.element_size()

    def copy_in():
        with torch.cuda.stream(s_in):
            A.copy_(A_h, non_blocking=True)
            B.copy_(B_h, non_blocking=True)

    def copy_out():
        with torch.cuda.stream(s_out):
            D_h.copy_(D, non_blocking=True)

    def timed(*fns):
        out = []
        for _ in range(reps + 1):
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s_in)
            s_out.wait_event(e0)
            for fn in fns:
                fn()
            s_in.wait_stream(s_out)
            e1.record(s_in)
            torch.cuda.synchronize()
            out.append(e0.elapsed_time(e1))
        return statistics.median(out[1:])

    t_in, t_out, t_both = timed(copy_in), timed(copy_out), timed(copy_in, copy_out)
    return {"h2d_gbs": round(h2d / t_in / 1e6, 1), "d2h_gbs": round(d2h / t_out / 1e6, 1),
            "both_gbs": round((h2d + d2h) / t_both / 1e6, 1), "ms_step_copies_alone": round(t_both, 4)}


# -------------------------------------------------------- CPU oracle arm
def _oracle_sample_rate(rows: int, threads: int):
    """Time the oracle's triple loop on `rows` full rows of the 8192^3 workload."""
    import oracle

    w = synth.GEMM_8192
    rng = np.random.default_rng(0)
    A = synth.normal_bf16(w.seed_a, (rows, w.K), 1.0 / np.sqrt(w.K))  # same distribution, first rows' shape
    B_bits = _B_cache()
    ii = np.repeat(np.arange(rows), w.N)
    jj = np.tile(np.arange(w.N), rows)
    del rng
    t0 = time.perf_counter()
    oracle.gemm_entries_f64(A, B_bits, ii, jj, threads=threads)
    dt = time.perf_counter() - t0
    return 2.0 * rows * w.N * w.K / dt, dt


_BCACHE = {}


def _B_cache():
    if "B" not in _BCACHE:
        w = synth.GEMM_8192
        _BCACHE["B"] = synth.normal_bf16(w.seed_b, (w.N, w.K), 1.0 / np.sqrt(w.K))
    return _BCACHE["B"]


def cpu_baseline(args):
    """The oracle as it stands, timed on the host cores on a bounded sample (~args.cpu_seconds of work)."""
    import oracle

    threads = oracle.default_threads()
    w = synth.GEMM_8192
    probe_rate, _ = _oracle_sample_rate(2, threads)
    rows = int(max(2, min(4096, args.cpu_seconds * probe_rate / (2.0 * w.N * w.K))))
    rate, dt = _oracle_sample_rate(rows, threads)
    return {"value": round(rate / 1e12, 8), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{rows} full rows of D ({rows * w.N} entries, K={w.K}) of the {w.M}x{w.N}x{w.K} workload, "
                      f"fp64 triple loop over {threads} OpenMP threads, {dt:.1f} s"}


def run_reference(args, ws, rank):
    """The oracle as it stands on the host cores; rank 0 only."""
    if rank != 0:
        return None
    import oracle

    threads = oracle.default_threads()
    w = synth.GEMM_8192
    B_bits = _B_cache()
    A_rows = synth.normal_bf16(w.seed_a, (1, w.K), 1.0 / np.sqrt(w.K))
    ii = np.zeros(w.N, dtype=np.int64)
    jj = np.arange(w.N, dtype=np.int64)
    for _ in range(args.warmup):
        oracle.gemm_entries_f64(A_rows, B_bits, ii, jj, threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.gemm_entries_f64(A_rows, B_bits, ii, jj, threads=threads)
    dt = time.perf_counter() - t0
    flops = 2.0 * w.N * w.K * args.steps
    value = flops / dt / 1e12
    sample = f"one row of D per step (8192 entries, K=8192) of the 8192^3 workload, fp64 triple loop"
    return {"impl": "reference", "metric": "bf16 GEMM TFLOP/s at 8192^3 (2-CTA 256x256, CLC); int16 copy HBM GB/s",
            "value": round(value, 8), "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3 / args.steps, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"gemm_bf16 {w.M}x{w.N}x{w.K} (oracle sample)", "M": w.M, "N": w.N, "K": w.K},
            "cpu_baseline": {"value": round(value, 8), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 8), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--tile", default="256x256", choices=["128x128", "128x256", "256x256", "auto"])
    ap.add_argument("--sched", default="clc", choices=["static", "clc"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--workload", default="headline", choices=["headline", "gemm4096", "contended", "grouped", "causal", "fork",
                                                                   "rows", "smallk", "ingress"])
    ap.add_argument("--reps", type=int, default=10, help="static/CLC pairs of the contended workload (>= 10)")
    ap.add_argument("--spin-ctas", type=int, default=32)
    ap.add_argument("--no-configs", action="store_true",
                    help="headline only: skip the 4096^3, contended and small-K measurements")
    ap.add_argument("--config-reps", type=int, default=7,
                    help="samples per configuration of the 4096^3 and small-K measurements")
    ap.add_argument("--contended-tile", default="256x256", choices=["128x128", "128x256", "256x256", "auto"])
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    ws, rank, local = dist_env()
    if args.gpus != ws and ws > 1:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={ws}")

    if args.impl == "reference":
        line = run_reference(args, ws, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0

    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    try:
        if args.workload == "gemm4096":
            line = run_gemm4096(args, ws, rank, local)
        elif args.workload == "contended":
            line = run_contended(args, ws, rank, local)
        elif args.workload == "grouped":
            line = run_grouped(args, ws, rank, local)
        elif args.workload == "causal":
            line = run_causal(args, ws, rank, local)
        elif args.workload == "rows":
            line = run_rows(args, ws, rank, local)
        elif args.workload == "fork":
            line = run_fork(args, ws, rank, local)
        elif args.workload == "smallk":
            line = run_smallk(args, ws, rank, local)
        elif args.workload == "ingress":
            line = run_ingress(args, ws, rank, local)
        else:
            line = run_ours(args, ws, rank, local)
    finally:
        if ws > 1:
            import torch.distributed as dist

            dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
