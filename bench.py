"""Throughput of C = A x B^T (bf16 8192^3 by default) on one GB300 through the C ABI.

    python bench.py [--steps K] [--warmup W] [--workload NAME] [--repeats R] [--impl reference]

One step = one gemm_tn call over the workload's operands, already resident in
HBM. Prints ONE JSON line: TFLOP/s = 2*M*N*K / device time, where the device
time follows the pages' protocol ("0. A Minimal Hopper Matmul", sections
"Running the Kernel" and "Performance"): CUDA events around every call, the
median call of each process, and the median over R fresh processes. The line
also carries the roofline fraction of the kernel (its mean event-timed launch
against the measured peak), the modelled tile traffic beside the ncu-measured
DRAM bytes, the other GEMM workloads (each with its own roofline), an
end-to-end figure through gemm_tn_host (pinned host buffers, copies inside the
timed region, with the link rates and the process's NUMA placement), the fp64
CPU oracle timed on this host's cores as a reported baseline, and the SM
clocks sampled through NVML during the timed region.

The path runs on one GPU. Launched on several (WORLD_SIZE > 1 or --gpus > 1)
the native arm loads no library and prints one line saying so: the product has
no multi-GPU path, and its cluster-multicast kernel is kept to single-GPU
processes.

--impl reference times the CPU oracle (the only reference implementation of
this path) on bounded samples of the same workload; under torchrun rank 0
alone runs it and prints the line.

--workload attn_* measures the attention forward pass (flash_attn_fwd) on one
of the seeded [batch, seq, heads, dim] workloads instead, with the same line:
TFLOP/s = 4 * batch * heads * (visible query-key pairs) * dim / device time.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

METRIC = "TFLOP/s (2MNK/t) for C=A·Bᵀ bf16 8192³ on 1 GB300; % of dense tensor peak"
ATTN_METRIC = ("TFLOP/s (4·B·H·visible pairs·D / t) for the attention forward pass "
               "softmax(scale·QKᵀ, mask)·V on 1 GB300; % of dense tensor peak")
SINGLE_GPU_ONLY = ("single-GPU path: the product has no multi-GPU form (replicas only) and its "
                   "cluster-multicast kernel runs only in single-GPU processes, so no library is loaded here")
L2_BYTES = 126 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
#: GB300's nominal dense bf16/fp16 tensor peak (no sparsity), TFLOP/s
NOMINAL_BF16_TFLOPS = 2250.0
#: dense bf16/fp16 tcgen05 work of one SM per clock: with the SM count and a
#: sampled SM clock it gives the tensor peak at the clock the kernel ran at
DENSE_FLOP_PER_SM_CLOCK = 8192
CSRC = ROOT / "dense_tiled_gemm_03_gb300" / "csrc"

# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one
# ncu capture of the kernel on the workload, with the digest of the library's
# CUDA sources at capture time: the figure is reported only while the sources
# are unchanged (a changed kernel makes it stale). Keyed by (workload, kernel
# configuration) or, for the fused kernels, (workload, configuration, epilogue).
NCU_TRAFFIC: dict[tuple, dict] = {
    ("bf16_8192x8192x8192", "2cta_n256"): {  # 546.8 us
        "bytes": 1082566400 + 136527872, "when": "2026-12-02", "source": "c6c6d69fc4ea",
        "kernel": "gemm_tn_sm103_kernel<GemmConfig<2, 256, 6, 1, 1, 0, 0, 0, 0>>"},
    ("fp16_4096x4096x4096", "2cta_n256_mc"): {  # 81.9 us
        "bytes": 106305536 + 33761792, "when": "2026-12-02", "source": "c6c6d69fc4ea",
        "kernel": "gemm_tn_sm103_kernel<GemmConfig<2, 256, 6, 0, 2, 0, 0, 0, 0>>"},
    ("fp16_3001x5003x4097", "2cta_n256_mc"): {  # 83.9 us
        "bytes": 96957440 + 27212800, "when": "2026-12-02", "source": "c6c6d69fc4ea",
        "kernel": "gemm_tn_sm103_kernel<GemmConfig<2, 256, 6, 0, 2, 0, 0, 0, 0>>"},
    ("bf16_128x16384x16384", "1cta_n128"): {  # 92.0 us
        "bytes": 542159872 + 3272960, "when": "2026-12-02", "source": "c6c6d69fc4ea",
        "kernel": "gemm_tn_sm103_kernel<GemmConfig<1, 128, 6, 1, 1, 0, 0, 0, 0>>"},
    ("fp16_256x256x256", "1cta_n64"): {  # 6.8 us
        "bytes": 305920 + 0, "when": "2026-12-02", "source": "c6c6d69fc4ea",
        "kernel": "gemm_tn_sm103_kernel<GemmConfig<1, 64, 4, 0, 1, 0, 0, 0, 1>>"},
    ("bf16_8x4096x4096", "1cta_decode_splitk"): {  # 11.9 us
        "bytes": 33637632 + 0, "when": "2026-12-02", "source": "c6c6d69fc4ea",
        "kernel": "gemm_tn_decode_kernel<4, 16, 1, 2>"},
    ("bf16_8192x8192x8192", "2cta_n256", "bias_gelu"): {  # 555.5 us
        "bytes": 1072375040 + 135900416, "when": "2026-12-02", "source": "c6c6d69fc4ea",
        "kernel": "gemm_tn_sm103_kernel<GemmConfig<2, 256, 6, 1, 1, 0, 1, 0, 0>>"},
}
# the same for the attention kernel, keyed by workload
NCU_TRAFFIC_ATTN: dict[str, dict] = {
    "attn_bf16_b2_s8192_h32_d128_causal": {  # 754.8 us
        "bytes": 454553088 + 117239552, "when": "2026-12-02", "source": "b1f83bdde46d",
        "kernel": "flash_attn_fwd_kernel<Cfg<128, 1>>"},
}

# fused epilogues the benchmark can time: (alpha, bias?, activation, output dtype name or None for A's)
EPILOGUES = {
    "none": None,
    "bias": (1.0, True, "none", None),
    "bias_gelu": (1.0, True, "gelu", None),
    "fp32": (1.0, False, "none", "float32"),
    "e4m3": (1.0 / 16, False, "none", "float8_e4m3fn"),   # alpha as the quantisation scale
}

# output tile of each kernel configuration for the traffic model: rows of A
# and rows of B one tile reads over K (a multicast cluster shares its A rows
# over 512 columns; the decode kernel reads every row of A for 128 rows of B)
TILE_OF_CONFIG = {
    "1cta_n256": (128, 256), "1cta_n128": (128, 128), "2cta_n256": (256, 256), "2cta_n128": (256, 128),
    "2cta_n256_mc": (256, 512), "1cta_n128_splitk": (128, 128), "1cta_decode_splitk": (None, 128),
    "1cta_n64": (128, 64),
}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="bf16_8192x8192x8192")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--repeats", type=int, default=3,
                    help="fresh processes whose median call times give the headline (the first is this one)")
    ap.add_argument("--workloads", default="all", choices=["all", "none"],
                    help="also time every other GEMM workload, each with its own roofline (GEMM workloads, "
                         "plain epilogue)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the oracle CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--config", default=None, help="force a kernel configuration (GEMM_TN_FORCE_CONFIG)")
    ap.add_argument("--epilogue", default="none", choices=sorted(EPILOGUES),
                    help="time gemm_tn_fused with this epilogue instead of the plain gemm_tn (GEMM workloads; "
                         "no end-to-end figure: the host-buffer entry point has no fused form)")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="budget of the whole --impl reference run (oracle work)")
    ap.add_argument("--cublas-context", action="store_true",
                    help="also time torch.matmul(a, b.T) (cuBLAS) on the same operands, the same way, and add it "
                         "to the line as context (not part of the product)")
    ap.add_argument("--oracle-table", action="store_true",
                    help="instead of the benchmark line: time the CPU oracle on every GEMM workload, with all "
                         "host threads and with one thread (one JSON line per workload and thread count)")
    ap.add_argument("--sustained", type=float, default=0.0,
                    help="also run the step back to back for this many seconds (power-capped steady state) and "
                         "report its TFLOP/s, median SM clock and TFLOP/s per GHz")
    ap.add_argument("--child-median", action="store_true", help=argparse.SUPPRESS)
    return ap.parse_args(argv)


def load_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# CUDA sources each kernel family is built from: the attention kernel's own
# translation unit, the PTX helpers and the host side that encodes its maps;
# the GEMM kernels are built from every other file but the repack kernel's
ATTN_SOURCES = ("sm103_flash_attn.cu", "sm103_ptx.cuh", "gemm_tn_internal.h", "gemm_tn_api.cu")
NOT_GEMM_SOURCES = ("sm103_flash_attn.cu", "repack.cu")


def source_digest(kind: str = "gemm") -> str:
    """Digest of the CUDA sources of one kernel family, in name order: "gemm"
    every file under csrc/ but NOT_GEMM_SOURCES, "attn" ATTN_SOURCES."""
    h = hashlib.sha256()
    for p in sorted(CSRC.iterdir()):
        if not (p.is_file() and p.suffix in (".cu", ".cuh", ".h")):
            continue
        if kind == "attn" and p.name not in ATTN_SOURCES:
            continue
        if kind == "gemm" and p.name in NOT_GEMM_SOURCES:
            continue
        h.update(p.name.encode())
        h.update(p.read_bytes())
    return h.hexdigest()[:12]


def stored_traffic(entry: dict | None, digest: str) -> tuple[int | None, str]:
    """(bytes, provenance) of a stored ncu capture: the bytes only while the
    CUDA sources still match the capture's digest."""
    if entry is None:
        return None, "no ncu capture of this kernel and workload"
    what = f"ncu capture of {entry['kernel']} on {entry['when']} (sources {entry['source']})"
    if entry["source"] != digest:
        return None, f"stale: the CUDA sources ({digest}) changed since the {what}"
    return int(entry["bytes"]), what


def modelled_traffic_bytes(m: int, n: int, k: int, tile_m: int, tile_n: int, elem_bytes: int = 2,
                           out_bytes: int = 2) -> int:
    """HBM bytes of a tiled product with no reuse between tiles ("Tiling a
    matmul", section "Counting traffic", for a rectangular tile_m x tile_n
    output tile): each tile reads its tile_m rows of A and tile_n rows of B
    over all of K, so A is read ceil(N / tile_n) times and B ceil(M / tile_m)
    times, and C is written once."""
    return elem_bytes * (m * k * math.ceil(n / tile_n) + n * k * math.ceil(m / tile_m)) + out_bytes * m * n


def tile_of(cfg_name: str, m: int) -> tuple[int, int]:
    tm, tn = TILE_OF_CONFIG[cfg_name]
    return (m if tm is None else tm), tn


# ------------------------------------------------------------------ clocks

class NvmlSampler:
    """SM clock, power and clock-event reasons of one GPU, read through NVML
    (read-only queries) every `period_s` while running. Falls back to an
    nvidia-smi subprocess when NVML cannot be loaded."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}
    SMI_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str, period_s: float = 0.002):
        self.uuid = uuid
        self.period = period_s
        self.nvml = None
        self.handle = None
        self.samples: list[tuple[float, float, int]] = []
        self.max_mhz = None
        self.thread = None
        self.proc = None
        self.stop_flag = threading.Event()
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() == 0:
                h = ctypes.c_void_p()
                if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) == 0:
                    self.nvml, self.handle = lib, h
                    mx = ctypes.c_uint()
                    if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:   # NVML_CLOCK_SM
                        self.max_mhz = float(mx.value)
        except OSError:
            self.nvml = None

    def _poll(self):
        lib, h = self.nvml, self.handle
        mhz, mw, reasons = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop_flag.is_set():
            ok = lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0
            pw = lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw)) == 0
            rs = lib.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(reasons)) == 0
            if ok:
                self.samples.append((float(mhz.value), mw.value / 1000.0 if pw else float("nan"),
                                     int(reasons.value) if rs else 0))
            time.sleep(self.period)

    def start(self):
        self.samples = []
        self.stop_flag.clear()
        if self.nvml is not None:
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            time.sleep(0.01)   # a first sample before the timed region
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.uuid}", f"--query-gpu={self.SMI_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self) -> dict:
        if self.thread is not None:
            self.stop_flag.set()
            self.thread.join()
            self.thread = None
            sm = [s[0] for s in self.samples]
            power = [s[1] for s in self.samples if s[1] == s[1]]
            reasons = sorted({name for s in self.samples for bit, name in self.REASONS.items() if s[2] & bit})
            return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                    "reasons": reasons, "samples": len(sm), "sm_mhz_min": min(sm) if sm else None,
                    "power_w_max": max(power) if power else None,
                    "source": f"NVML every {self.period * 1e3:.0f} ms"}
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.proc = None
        sm, smax, power, reasons = [], None, [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
                power.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None, "source": "nvidia-smi every 100 ms"}


def gpu_uuid(dev) -> str:
    import torch
    text = str(torch.cuda.get_device_properties(dev).uuid)
    return text if text.startswith("GPU-") else f"GPU-{text}"


# ------------------------------------------------------------------ NUMA placement

def parse_cpulist(text: str) -> set[int]:
    cpus: set[int] = set()
    for part in text.strip().split(","):
        if not part:
            continue
        lo, _, hi = part.partition("-")
        cpus.update(range(int(lo), int(hi or lo) + 1))
    return cpus


def format_cpulist(cpus) -> str:
    out, run = [], []
    for c in sorted(cpus):
        if run and c == run[-1] + 1:
            run.append(c)
            continue
        if run:
            out.append(f"{run[0]}-{run[-1]}" if len(run) > 1 else str(run[0]))
        run = [c]
    if run:
        out.append(f"{run[0]}-{run[-1]}" if len(run) > 1 else str(run[0]))
    return ",".join(out)


def gpu_placement(dev) -> dict:
    """The GPU's PCI address, its NUMA node and local CPUs (sysfs), this
    process's CPU affinity, and the CPUs to pin to while allocating and using
    pinned host buffers: the allowed CPUs local to the GPU, when that is a
    proper, non-empty subset."""
    import torch
    p = torch.cuda.get_device_properties(dev)
    bdf = f"{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
    base = Path("/sys/bus/pci/devices") / bdf

    def read(name):
        try:
            return (base / name).read_text().strip()
        except OSError:
            return None

    numa, local = read("numa_node"), read("local_cpulist")
    allowed = os.sched_getaffinity(0)
    use = allowed & parse_cpulist(local) if local else set()
    return {"pci": bdf, "numa_node": None if numa is None else int(numa), "local_cpulist": local,
            "affinity": format_cpulist(allowed),
            "pin_to": format_cpulist(use) if use and use != allowed else None}


# ------------------------------------------------------------------ timing

def time_calls(step, steps: int, warmup: int, stream, flush=None, sampler=None, count=None) -> dict:
    """Run `step` warmup times, then time `steps` calls with CUDA events on
    `stream` around each call (after an L2 flush when `flush` is given, outside
    the events). Returns per-call statistics in ms, the event-timed region
    around all calls, the library's launches inside it and the sampled clocks."""
    import torch
    for _ in range(warmup):
        if flush is not None:
            flush()
        step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if sampler is not None:
        sampler.start()
    torch.cuda.synchronize()
    launches0 = count() if count else 0
    r0.record(stream)
    for i in range(steps):
        if flush is not None:
            flush()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    r1.record(stream)
    launches = (count() - launches0) if count else None
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler is not None else None
    times = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return {"median_ms": statistics.median(times), "min_ms": min(times), "mean_ms": sum(times) / len(times),
            "region_ms": r0.elapsed_time(r1), "launches": launches, "clocks": clocks}


def sustained_run(step, seconds: float, stream, flops: float, sampler) -> dict:
    """The step back to back for about `seconds` (no events between calls):
    TFLOP/s over the whole region, with the SM clock sampled meanwhile and the
    rate per GHz of median clock, so that runs at different clocks compare."""
    import torch
    step()
    torch.cuda.synchronize()
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    r0.record(stream)
    for _ in range(3):
        step()
    r1.record(stream)
    torch.cuda.synchronize()
    per_call = r0.elapsed_time(r1) / 3 / 1e3
    calls = max(3, int(seconds / max(per_call, 1e-6)))
    sampler.start()
    torch.cuda.synchronize()
    r0.record(stream)
    for _ in range(calls):
        step()
    r1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    s = r0.elapsed_time(r1) / 1e3
    tflops = calls * flops / s / 1e12
    mhz = clocks.get("sm_mhz")
    return {"tflops": round(tflops, 1), "seconds": round(s, 3), "calls": calls, "clocks": clocks,
            "tflops_per_ghz": round(tflops / (mhz / 1e3), 1) if mhz else None}


def child_median(args) -> dict:
    """One fresh process's median call time of the workload (the --repeats
    children): the same operands, warm-up and timing as the headline."""
    import torch
    import dense_tiled_gemm_03_gb300 as gt
    from dense_tiled_gemm_03_gb300.workloads import WORKLOADS, workload_operands
    w = WORKLOADS[args.workload]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    a_cpu, b_cpu = workload_operands(w)
    a, b = a_cpu.to(dev), b_cpu.to(dev)
    c = torch.empty((w.m, w.n), dtype=a.dtype, device=dev)
    flush = l2_flusher(dev, (w.m * w.k + w.n * w.k) * 2)
    t = time_calls(lambda: gt.mm_tn(a, b, out=c), args.steps, args.warmup, torch.cuda.current_stream(dev), flush)
    return {"median_ms": t["median_ms"], "min_ms": t["min_ms"], "mean_ms": t["mean_ms"]}


def l2_flusher(dev, input_bytes: int):
    """A callable that writes a buffer of twice the L2 size when the inputs are
    smaller than that (so each timed call starts with them out of L2), else None."""
    import torch
    if input_bytes >= 2 * L2_BYTES:
        return None
    scratch = torch.empty(L2_BYTES * 2 // 4, dtype=torch.int32, device=dev)
    return lambda: scratch.fill_(1)


# ------------------------------------------------------------------ oracle baseline

def cpu_oracle_rate(a, b, seconds: float):
    """Time the fp64 oracle on a bounded row sample of the workload; returns
    (TFLOP/s, cores, description)."""
    import oracle
    m, k = a.shape
    n = b.shape[0]
    cores = oracle.host_threads()
    rows = max(1, min(m, cores))
    t0 = time.perf_counter()
    oracle.gemm_tn_reference(a[:rows], b)
    dt = time.perf_counter() - t0
    target_rows = int(min(m, max(rows, rows * seconds / max(dt, 1e-6))))
    if target_rows > rows:
        t0 = time.perf_counter()
        oracle.gemm_tn_reference(a[:target_rows], b)
        dt = time.perf_counter() - t0
        rows = target_rows
    flops = 2.0 * rows * n * k
    return flops / dt / 1e12, cores, f"first {rows} of {m} rows of C (all {n} columns, K={k}), {dt:.1f} s"


def oracle_table():
    """The CPU baseline per GEMM workload on this host: the fp64 oracle with
    every host thread on a row sample of about 10 s, and with one thread on the
    whole product for the two smallest workloads or on a 256-row slice (the
    rate extrapolated to the whole product, labelled as such) for the others."""
    import platform
    import oracle
    from dense_tiled_gemm_03_gb300.workloads import WORKLOADS, workload_operands
    cpu = platform.processor() or platform.machine()
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        cpu = next((ln.split(":", 1)[1].strip() for ln in out.splitlines() if ln.startswith("Model name")), cpu)
    except (OSError, subprocess.SubprocessError):
        pass
    for name, w in WORKLOADS.items():
        a, b = workload_operands(w)
        for threads in (oracle.host_threads(), 1):
            if threads == 1 and w.m * w.n * w.k <= 4096 ** 3:
                rows, how = w.m, "whole product"
            elif threads == 1:
                rows, how = min(w.m, 256), f"first {min(w.m, 256)} rows, rate extrapolated to the whole product"
            else:
                rows = max(1, min(w.m, threads))
                t0 = time.perf_counter()
                oracle.gemm_tn_reference(a[:rows], b, nthreads=threads)
                per_row = (time.perf_counter() - t0) / rows
                rows = int(min(w.m, max(rows, 10.0 / max(per_row, 1e-9))))
                how = "whole product" if rows == w.m else f"first {rows} rows, rate extrapolated to the whole product"
            t0 = time.perf_counter()
            oracle.gemm_tn_reference(a[:rows], b, nthreads=threads)
            dt = time.perf_counter() - t0
            flops = 2.0 * rows * w.n * w.k
            print(json.dumps({"oracle_table": name, "threads": threads, "cpu": cpu, "sample": how,
                              "seconds": round(dt, 3), "gflops": round(flops / dt / 1e9, 3),
                              "seconds_whole_product": round(dt * w.m / rows, 2)}), flush=True)


# ------------------------------------------------------------------ native arm

def gemm_roofline(w, cfg_name: str, t: dict, peaks, peak_src, digest: str, c_elem: int = 2,
                  traffic_key=None, kernel_name=None) -> dict:
    """Roofline of one GEMM kernel from its mean event-timed launch: tensor-
    bound against the bf16 peak, or HBM-bound (ideal intensity under the
    ridge) against the copy bandwidth, with the compulsory and the modelled
    tile traffic and the stored ncu DRAM bytes."""
    tensor_peak = float(peaks["bf16_tflops"])
    hbm_peak = float(peaks["hbm_gbs"])
    mean_s = t["mean_ms"] * 1e-3
    compulsory = (w.m * w.k + w.n * w.k) * 2 + w.m * w.n * c_elem
    hbm_bound = hbm_peak * 1e9 * (w.flops / compulsory) < tensor_peak * 1e12
    if hbm_bound:
        achieved = compulsory / mean_s / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4),
                "tflops": round(w.flops / mean_s / 1e12, 2)}
    else:
        achieved = w.flops / mean_s / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": tensor_peak, "unit": "TFLOP/s",
                "frac": round(achieved / tensor_peak, 4),
                "frac_of_sustained": round(achieved / float(peaks.get("bf16_tflops_sustained", tensor_peak)), 4)}
    traffic, provenance = stored_traffic(NCU_TRAFFIC.get(traffic_key or (w.name, cfg_name)), digest)
    tm, tn = tile_of(cfg_name, w.m)
    modelled = modelled_traffic_bytes(w.m, w.n, w.k, tm, tn, 2, c_elem)
    roof.update({
        "traffic": traffic, "traffic_source": provenance, "algorithmic_bytes": compulsory,
        "modelled_traffic": modelled, "modelled_tile": [tm, tn],
        "modelled_traffic_note": "tile traffic with no reuse between tiles; the measured bytes fall below it by "
                                 "what L2 reuse saves",
        "peak_source": f"{peak_src} ({'hbm_gbs' if hbm_bound else 'bf16_tflops'} burst; kernel timed alone)",
        "kernel": kernel_name or kernel_label(cfg_name),
        "launch_ms_mean": round(t["mean_ms"], 5),
    })
    return roof


def kernel_label(cfg_name: str, fused: bool = False) -> str:
    if cfg_name == "1cta_decode_splitk":
        return "gemm_tn_decode_kernel"
    if cfg_name.endswith("splitk"):
        return "gemm_tn_splitk_kernel"
    return f"gemm_tn_sm103_kernel<{cfg_name}{', fused' if fused else ''}>"


def time_workload(gt, torch, dev, w, steps, warmup, peaks, peak_src, digest) -> dict:
    """One of the other GEMM workloads: median / min call time, TFLOP/s and
    its own roofline."""
    from dense_tiled_gemm_03_gb300.workloads import workload_operands
    a_cpu, b_cpu = workload_operands(w)
    a, b = a_cpu.to(dev), b_cpu.to(dev)
    c = torch.empty((w.m, w.n), dtype=a.dtype, device=dev)
    op_bytes = (w.m * w.k + w.n * w.k) * 2
    flush = l2_flusher(dev, op_bytes)
    t = time_calls(lambda: gt.mm_tn(a, b, out=c), steps, warmup, torch.cuda.current_stream(dev), flush,
                   count=gt.gemm_tn_launch_count)
    cfg_name = gt.gemm_tn_config_name(gt.gemm_tn_last_config())
    return {
        "value": round(w.flops / (t["median_ms"] * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
        "ms_per_step": round(t["median_ms"], 5), "min_ms": round(t["min_ms"], 5),
        "dtype": w.dtype, "m": w.m, "n": w.n, "k": w.k, "seed": w.seed, "kernel_config": cfg_name,
        "gpu_launches": t["launches"],
        "l2": "L2 flushed between calls" if flush else "inputs larger than L2",
        "roofline": gemm_roofline(w, cfg_name, t, peaks, peak_src, digest),
    }


def e2e_leg(gt, torch, dev, w, a_cpu, b_cpu, steps: int, device_ms: float, placement: dict) -> dict:
    """End to end through gemm_tn_host: pinned host A and B in, C back to
    pinned host memory, every step, timed on the host clock. The pinned
    buffers are allocated (and first touched) with this thread pinned to the
    GPU's local CPUs when those are known. Also measures the plain host link
    rates for the step's bytes and the GEMM's share of the step."""
    before = os.sched_getaffinity(0)
    if placement.get("pin_to"):
        os.sched_setaffinity(0, parse_cpulist(placement["pin_to"]))
    try:
        pin_a, pin_b = a_cpu.pin_memory(), b_cpu.pin_memory()
        pin_c = torch.empty((w.m, w.n), dtype=a_cpu.dtype).pin_memory()
        # plain copy rates of the step's bytes (best of three, CUDA events)
        da, db = torch.empty_like(pin_a, device=dev), torch.empty_like(pin_b, device=dev)
        dc = torch.empty((w.m, w.n), dtype=a_cpu.dtype, device=dev)
        stream = torch.cuda.current_stream(dev)
        h2d, d2h = [], []
        for _ in range(3):
            e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            e0.record(stream)
            da.copy_(pin_a, non_blocking=True)
            db.copy_(pin_b, non_blocking=True)
            e1.record(stream)
            pin_c.copy_(dc, non_blocking=True)
            e2.record(stream)
            torch.cuda.synchronize(dev)
            h2d.append(e0.elapsed_time(e1))
            d2h.append(e1.elapsed_time(e2))
        del da, db, dc
        in_bytes, out_bytes = pin_a.numel() * 2 + pin_b.numel() * 2, w.m * w.n * 2
        gt.mm_tn_host(pin_a, pin_b, out=pin_c, device=dev)   # warm: staging pool, copy streams
        times = []
        for _ in range(steps):
            t0 = time.perf_counter()
            gt.mm_tn_host(pin_a, pin_b, out=pin_c, device=dev)
            times.append(time.perf_counter() - t0)
    finally:
        os.sched_setaffinity(0, before)
    e2e_s = statistics.median(times)
    return {"value": round(w.flops / e2e_s / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out_bytes + 4,
            "steps": steps, "ms_per_step": round(e2e_s * 1e3, 3), "ms_min": round(min(times) * 1e3, 3),
            "statistic": "median call on the host clock",
            "entry_point": "gemm_tn_host (pinned host buffers)",
            "h2d_gbs": round(in_bytes / (min(h2d) * 1e-3) / 1e9, 1),
            "d2h_gbs": round(out_bytes / (min(d2h) * 1e-3) / 1e9, 1),
            "serial_copy_ms": round(min(h2d) + min(d2h), 3),
            "gemm_share": round(device_ms / (e2e_s * 1e3), 4),
            "placement": placement}


def run_native(args, peaks, peak_src):
    import torch
    import dense_tiled_gemm_03_gb300 as gt
    from dense_tiled_gemm_03_gb300 import build as native_build
    from dense_tiled_gemm_03_gb300.workloads import WORKLOADS, workload_operands

    native_build.build()
    digest = source_digest()
    w = WORKLOADS[args.workload]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    placement = gpu_placement(dev)
    a_cpu, b_cpu = workload_operands(w)
    a, b = a_cpu.to(dev), b_cpu.to(dev)
    c = torch.empty((w.m, w.n), dtype=a.dtype, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    op_bytes = (w.m * w.k + w.n * w.k) * 2
    flush = l2_flusher(dev, op_bytes)
    fused = EPILOGUES[args.epilogue]
    c_elem = 2
    if fused is None:
        def step():
            gt.mm_tn(a, b, out=c, status=status)
    else:
        alpha, with_bias, act, out_name = fused
        out_dtype = getattr(torch, out_name) if out_name else a.dtype
        c = torch.empty((w.m, w.n), dtype=out_dtype, device=dev)
        c_elem = c.element_size()
        bias = torch.linspace(-1.0, 1.0, w.n, dtype=torch.float32, device=dev) if with_bias else None

        def step():
            gt.mm_tn_fused(a, b, out=c, alpha=alpha, bias=bias, activation=act, out_dtype=out_dtype, status=status)

    sampler = NvmlSampler(gpu_uuid(dev))
    t = time_calls(step, args.steps, args.warmup, stream, flush, sampler, gt.gemm_tn_launch_count)
    if int(status.item()) != 0:
        raise RuntimeError(f"device watchdog fired: {gt.gemm_tn_status_string(int(status.item()))}")
    cfg_name = gt.gemm_tn_config_name(gt.gemm_tn_last_config())
    clocks = t["clocks"]

    # the other GEMM workloads, each with its own roofline (plain epilogue)
    workloads = None
    if args.workloads == "all" and fused is None and args.config is None:
        workloads = {}
        for name, other in WORKLOADS.items():
            if name != w.name:
                workloads[name] = time_workload(gt, torch, dev, other, args.steps, args.warmup, peaks, peak_src,
                                                digest)

    sustained = None
    if args.sustained > 0:
        sustained = sustained_run(step, args.sustained, stream, w.flops, NvmlSampler(gpu_uuid(dev), 0.02))

    e2e = None
    if fused is None and not args.no_e2e:
        e2e = e2e_leg(gt, torch, dev, w, a_cpu, b_cpu, args.e2e_steps, t["median_ms"], placement)

    # the pages' protocol: the median call of R fresh processes (this one first)
    per_process = [{"median_ms": t["median_ms"], "min_ms": t["min_ms"], "mean_ms": t["mean_ms"]}]
    if fused is None and args.config is None:
        for _ in range(max(0, args.repeats - 1)):
            per_process.append(run_child(args))
    med = statistics.median(p["median_ms"] for p in per_process)
    value = w.flops / (med * 1e-3) / 1e12

    roofline = gemm_roofline(w, cfg_name, t, peaks, peak_src, digest, c_elem,
                             traffic_key=None if fused is None else (w.name, cfg_name, args.epilogue),
                             kernel_name=kernel_label(cfg_name, fused is not None))
    sm_clock = clocks.get("sm_mhz") if clocks else None
    if sm_clock:
        # the tensor peak at the sampled clock: frac above 1 would mean the
        # measured peak is not a ceiling for this kernel
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        at_clock = sms * DENSE_FLOP_PER_SM_CLOCK * sm_clock * 1e6 / 1e12
        roofline["peak_at_sampled_clock"] = round(at_clock, 1)
        roofline["frac_of_peak_at_sampled_clock"] = round(w.flops / (t["mean_ms"] * 1e-3) / 1e12 / at_clock, 4)
    roofline["frac_above_one"] = roofline["frac"] > 1.0

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(med, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic",
        "config": {"workload": w.name, "m": w.m, "n": w.n, "k": w.k, "dist": w.dist, "seed": w.seed,
                   "kernel_config": cfg_name, "parallelism": "single GPU",
                   "l2": "L2 flushed between calls" if flush else
                   f"inputs larger than L2 ({op_bytes / 1e6:.0f} MB of operands vs {L2_BYTES / 1e6:.0f} MB)",
                   "accumulate": "fp32", "epilogue": args.epilogue},
        "timing": {"protocol": "CUDA events around each call on the launching stream; the median call of each "
                               "process; value = the median over the fresh processes",
                   "repeats": len(per_process),
                   "per_process": [{k: round(v, 5) for k, v in p.items()} for p in per_process],
                   "median_ms": round(med, 5), "min_ms": round(min(p["min_ms"] for p in per_process), 5),
                   "region_ms_per_step": round(t["region_ms"] / args.steps, 5)},
        "pct_of_peak": round(100 * w.flops / (med * 1e-3) / 1e12 / float(peaks["bf16_tflops"]), 2),
        "pct_of_nominal_peak": round(100 * w.flops / (med * 1e-3) / 1e12 / NOMINAL_BF16_TFLOPS, 2),
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": t["launches"],
        "clocks": clocks,
        "workloads": workloads,
    }
    if sustained is not None:
        line["sustained"] = sustained
    if args.cublas_context:
        # the same operands through torch.matmul (cuBLAS), timed the same way
        ref_c = torch.empty((w.m, w.n), dtype=a.dtype, device=dev)
        tc = time_calls(lambda: torch.matmul(a, b.t(), out=ref_c), args.steps, args.warmup, stream, flush)
        cublas_tflops = w.flops / (tc["median_ms"] * 1e-3) / 1e12
        line["context"] = {"cublas_tflops": round(cublas_tflops, 2),
                           "ratio_to_cublas": round(w.flops / (t["median_ms"] * 1e-3) / 1e12 / cublas_tflops, 4),
                           "what": "torch.matmul(a, b.T) on the same operands, timed the same way (median call)"}
    if not args.no_cpu_baseline:
        v, cores, sample = cpu_oracle_rate(a_cpu, b_cpu, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(v, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                "sample": sample}
    return line


def run_child(args) -> dict:
    cmd = [sys.executable, str(Path(__file__).resolve()), "--child-median", "--workload", args.workload,
           "--steps", str(args.steps), "--warmup", str(args.warmup)]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600)
    if res.returncode != 0:
        raise RuntimeError(f"repeat process failed ({res.returncode}): {res.stderr[-2000:]}")
    return json.loads(res.stdout.strip().splitlines()[-1])


# ------------------------------------------------------------------ attention

def attn_sample_rows(w, budget_flops: float) -> list[int]:
    """Query rows spread over the sequence whose oracle work (all batches and
    heads) stays near budget_flops."""
    per_row = 4.0 * w.batch * w.heads * w.dim * ((w.seq + 1) / 2 if w.causal else w.seq)
    n = int(max(1, min(w.seq, budget_flops / per_row)))
    step = w.seq / n
    return sorted({min(w.seq - 1, int(i * step + step / 2)) for i in range(n)})


def attn_rows_flops(w, rows) -> float:
    return sum(4.0 * w.batch * w.heads * w.dim * ((r + 1) if w.causal else w.seq) for r in rows)


def cpu_oracle_attn_rate(w, q, k, v, seconds: float):
    """Time the fp64 attention oracle on a bounded sample of query rows;
    returns (TFLOP/s, cores, description)."""
    import oracle
    cores = oracle.host_threads()
    probe = attn_sample_rows(w, 2e9)
    t0 = time.perf_counter()
    oracle.attention_reference(q, k, v, causal=w.causal, rows=probe)
    dt = time.perf_counter() - t0
    rate = attn_rows_flops(w, probe) / max(dt, 1e-6)
    rows = attn_sample_rows(w, rate * seconds)
    t0 = time.perf_counter()
    oracle.attention_reference(q, k, v, causal=w.causal, rows=rows)
    dt = time.perf_counter() - t0
    flops = attn_rows_flops(w, rows)
    return flops / dt / 1e12, cores, (f"{len(rows)} of {w.seq} query rows spread over the sequence, every batch "
                                      f"and head, {dt:.1f} s")


def run_native_attn(args, peaks, peak_src):
    import torch
    import dense_tiled_gemm_03_gb300 as gt
    from dense_tiled_gemm_03_gb300 import build as native_build
    from dense_tiled_gemm_03_gb300.workloads import ATTN_WORKLOADS, make_qkv

    native_build.build()
    digest = source_digest("attn")
    w = ATTN_WORKLOADS[args.workload]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    placement = gpu_placement(dev)
    q_cpu, k_cpu, v_cpu = make_qkv(w.batch, w.seq, w.heads, w.dim, w.dtype, seed=w.seed)
    q, k, v = q_cpu.to(dev), k_cpu.to(dev), v_cpu.to(dev)
    o = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    tensor_bytes = q.numel() * 2
    io_bytes = 4 * tensor_bytes   # Q, K, V read once, O written once
    flush = l2_flusher(dev, io_bytes)
    sampler = NvmlSampler(gpu_uuid(dev))
    t = time_calls(lambda: gt.flash_attn(q, k, v, causal=w.causal, out=o, status=status), args.steps, args.warmup,
                   stream, flush, sampler, gt.gemm_tn_launch_count)
    if int(status.item()) != 0:
        raise RuntimeError(f"device watchdog fired: {gt.gemm_tn_status_string(int(status.item()))}")
    med = t["median_ms"]
    value = w.flops / (med * 1e-3) / 1e12
    tensor_peak = float(peaks["bf16_tflops"])
    achieved = w.flops / (t["mean_ms"] * 1e-3) / 1e12
    traffic, provenance = stored_traffic(NCU_TRAFFIC_ATTN.get(w.name), digest)
    roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": tensor_peak, "unit": "TFLOP/s",
                "frac": round(achieved / tensor_peak, 4),
                "frac_of_sustained": round(achieved / float(peaks.get("bf16_tflops_sustained", tensor_peak)), 4),
                "traffic": traffic, "traffic_source": provenance, "algorithmic_bytes": io_bytes,
                "peak_source": f"{peak_src} (bf16_tflops burst; kernel timed alone)",
                "kernel": f"flash_attn_fwd_kernel<dim {w.dim}, {w.dtype}>", "launch_ms_mean": round(t["mean_ms"], 5)}

    # end to end: pinned host Q, K, V in, O back to pinned host memory, each step
    before = os.sched_getaffinity(0)
    if placement.get("pin_to"):
        os.sched_setaffinity(0, parse_cpulist(placement["pin_to"]))
    try:
        pins = [x.pin_memory() for x in (q_cpu, k_cpu, v_cpu)]
        pin_o = torch.empty_like(q_cpu).pin_memory()
        dq, dk, dv, do = (torch.empty_like(q) for _ in range(4))

        def e2e_step():
            for dst, src in zip((dq, dk, dv), pins):
                dst.copy_(src, non_blocking=True)
            gt.flash_attn(dq, dk, dv, causal=w.causal, out=do, status=status)
            pin_o.copy_(do, non_blocking=True)
            torch.cuda.current_stream(dev).synchronize()

        e2e_step()
        times = []
        for _ in range(args.e2e_steps):
            t0 = time.perf_counter()
            e2e_step()
            times.append(time.perf_counter() - t0)
    finally:
        os.sched_setaffinity(0, before)
    e2e_s = statistics.median(times)
    e2e = {"value": round(w.flops / e2e_s / 1e12, 2), "unit": "TFLOP/s",
           "h2d_bytes_per_step": 3 * tensor_bytes, "d2h_bytes_per_step": tensor_bytes, "steps": args.e2e_steps,
           "ms_per_step": round(e2e_s * 1e3, 3), "statistic": "median call on the host clock",
           "entry_point": "flash_attn_fwd with pinned host copies on the same stream",
           "gemm_share": round(med / (e2e_s * 1e3), 4), "placement": placement}
    line = {
        "metric": ATTN_METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(med, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "seq": w.seq, "heads": w.heads, "dim": w.dim,
                   "causal": w.causal, "seed": w.seed, "parallelism": "single GPU",
                   "l2": "L2 flushed between calls" if flush else
                   f"inputs larger than L2 ({io_bytes / 1e6:.0f} MB of Q, K, V and O vs {L2_BYTES / 1e6:.0f} MB)",
                   "accumulate": "fp32"},
        "timing": {"protocol": "CUDA events around each call on the launching stream; median call",
                   "median_ms": round(med, 5), "min_ms": round(t["min_ms"], 5), "mean_ms": round(t["mean_ms"], 5),
                   "region_ms_per_step": round(t["region_ms"] / args.steps, 5)},
        "pct_of_peak": round(100 * value / tensor_peak, 2),
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": t["launches"],
        "clocks": t["clocks"],
    }
    if not args.no_cpu_baseline:
        rate, cores, sample = cpu_oracle_attn_rate(w, q_cpu, k_cpu, v_cpu, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(rate, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                "sample": sample}
    return line


def run_reference_attn(args, world: int):
    """The attention oracle as it stands, on bounded row samples per step."""
    from dense_tiled_gemm_03_gb300.workloads import ATTN_WORKLOADS, make_qkv
    import oracle

    w = ATTN_WORKLOADS[args.workload]
    q, k, v = make_qkv(w.batch, w.seq, w.heads, w.dim, w.dtype, seed=w.seed)
    cores = oracle.host_threads()
    total = args.steps + args.warmup
    probe = attn_sample_rows(w, 2e9)
    t0 = time.perf_counter()
    oracle.attention_reference(q, k, v, causal=w.causal, rows=probe)
    rate = attn_rows_flops(w, probe) / max(time.perf_counter() - t0, 1e-6)
    rows = attn_sample_rows(w, rate * args.ref_seconds / total)
    for _ in range(args.warmup):
        oracle.attention_reference(q, k, v, causal=w.causal, rows=rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.attention_reference(q, k, v, causal=w.causal, rows=rows)
    dt = time.perf_counter() - t0
    value = args.steps * attn_rows_flops(w, rows) / dt / 1e12
    sample = f"{len(rows)} of {w.seq} query rows per step (every batch and head) of {w.name}"
    return {
        "impl": "reference", "metric": ATTN_METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "seq": w.seq, "heads": w.heads, "dim": w.dim,
                   "causal": w.causal, "seed": w.seed},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------------ reference arm

def run_reference(args, world: int):
    """The CPU oracle, timed as it stands on this host's cores: each step is a
    bounded row sample of the workload, sized so the whole run takes about
    --ref-seconds (two minutes by default)."""
    from dense_tiled_gemm_03_gb300.workloads import WORKLOADS, workload_operands
    import oracle

    w = WORKLOADS[args.workload]
    a_cpu, b_cpu = workload_operands(w)
    cores = oracle.host_threads()
    total = args.steps + args.warmup
    # calibrate rows per step against the budget for the whole run
    probe = max(1, min(w.m, cores))
    t0 = time.perf_counter()
    oracle.gemm_tn_reference(a_cpu[:probe], b_cpu)
    per_row = (time.perf_counter() - t0) / probe
    rows = int(max(1, min(w.m, args.ref_seconds / total / max(per_row, 1e-9))))
    for i in range(args.warmup):
        r0 = (i * rows) % w.m
        oracle.gemm_tn_reference(a_cpu[r0:r0 + rows], b_cpu)
    t0 = time.perf_counter()
    done = 0
    for i in range(args.steps):
        r0 = (i * rows) % w.m
        oracle.gemm_tn_reference(a_cpu[r0:r0 + rows], b_cpu)
        done += min(rows, w.m - r0)
    dt = time.perf_counter() - t0
    value = 2.0 * done * w.n * w.k / dt / 1e12
    sample = f"{rows} rows of C per step (all {w.n} columns, K={w.k}) of {w.name}"
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "m": w.m, "n": w.n, "k": w.k, "seed": w.seed},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse_args(argv)
    if args.config:
        os.environ["GEMM_TN_FORCE_CONFIG"] = args.config
    if args.gpus < 1:
        raise SystemExit("--gpus must be >= 1")
    if args.epilogue != "none" and (args.workload.startswith("attn_") or args.impl == "reference"):
        raise SystemExit("--epilogue applies to the native GEMM workloads only")
    if args.oracle_table:
        oracle_table()
        return
    if args.child_median:
        print(json.dumps(child_median(args)), flush=True)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    attn = args.workload.startswith("attn_")
    if args.impl == "reference":
        # the oracle runs on the host: rank 0 alone, the other ranks exit
        if rank == 0:
            line = run_reference_attn(args, world) if attn else run_reference(args, world)
            print(json.dumps(line), flush=True)
        return
    if world > 1 or args.gpus > 1:
        if rank == 0:
            print(json.dumps({"metric": ATTN_METRIC if attn else METRIC, "n_gpus": max(world, args.gpus),
                              "unavailable": SINGLE_GPU_ONLY}), flush=True)
        return
    peaks, src = load_peaks()
    line = run_native_attn(args, peaks, src) if attn else run_native(args, peaks, src)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
