"""Throughput of C = A x B^T (bf16 8192^3 by default) on GB300 through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step = one gemm_tn call over the workload's operands, already resident in
HBM. Prints ONE JSON line (rank 0): TFLOP/s = 2*M*N*K / device time, its
roofline fraction (live CUDA-event launch durations against the measured peak),
an end-to-end figure through gemm_tn_host (host buffers, copies inside the
timed region), the fp64 CPU oracle timed on this host's cores as a reported
baseline, and SM clocks sampled during the timed region.

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the product needs no exchange between GPUs); `value` is the sum over ranks of
the work divided by the slowest rank's time.

--impl reference times the CPU oracle (the only reference implementation of
this path) on bounded samples of the same workload.

--workload attn_* measures the attention forward pass (flash_attn_fwd) on one
of the seeded [batch, seq, heads, dim] workloads instead, with the same line:
TFLOP/s = 4 * batch * heads * (visible query-key pairs) * dim / device time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

METRIC = "TFLOP/s (2MNK/t) for C=A·Bᵀ bf16 8192³ on 1 GB300; % of dense tensor peak"
ATTN_METRIC = ("TFLOP/s (4·B·H·visible pairs·D / t) for the attention forward pass "
               "softmax(scale·QKᵀ, mask)·V on 1 GB300; % of dense tensor peak")
L2_BYTES = 126 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Algorithmic DRAM traffic per launch measured by ncu for the default workload
# (dram__bytes_read.sum + dram__bytes_write.sum); see profiles/. None until a
# capture of the current kernel exists.
NCU_TRAFFIC_BYTES = {
    # dram__bytes_read.sum + dram__bytes_write.sum of one launch of the current
    # kernels (profiles/gemm_tn_*.md)
    ("bf16_8192x8192x8192", "2cta_n256"): 1_074_012_416 + 125_360_896,
    ("fp16_4096x4096x4096", "2cta_n256_mc"): 81_974_528 + 15_100_928,
    ("bf16_128x16384x16384", "1cta_n128"): 542_159_872 + 2_915_584,
    ("fp16_3001x5003x4097", "2cta_n256_mc"): 82_883_328 + 14_531_328,
    ("bf16_8x4096x4096", "1cta_decode_splitk"): 33_638_144 + 0,
}
# the same for the fused kernels, keyed by (workload, configuration, epilogue)
NCU_TRAFFIC_FUSED_BYTES: dict[tuple[str, str, str], int] = {
    ("bf16_8192x8192x8192", "2cta_n256", "e4m3"): 1_053_888_512 + 63_751_680,
}

# the same for the attention kernel, keyed by workload
NCU_TRAFFIC_ATTN_BYTES: dict[str, int] = {
    "attn_bf16_b2_s8192_h32_d128_causal": 453_134_336 + 116_694_016,
}


# fused epilogues the benchmark can time: (alpha, bias?, activation, output dtype name or None for A's)
EPILOGUES = {
    "none": None,
    "bias": (1.0, True, "none", None),
    "bias_gelu": (1.0, True, "gelu", None),
    "fp32": (1.0, False, "none", "float32"),
    "e4m3": (1.0 / 16, False, "none", "float8_e4m3fn"),   # alpha as the quantisation scale
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="bf16_8192x8192x8192")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=10)
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
    return ap.parse_args()


def load_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ distributed

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group("gloo")
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ------------------------------------------------------------------ clocks

def gpu_smi_id(dev) -> str:
    """nvidia-smi --id for a torch device: its UUID (robust to CUDA_VISIBLE_DEVICES)."""
    import torch
    uuid = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    if uuid is not None:
        text = str(uuid)
        return text if text.startswith("GPU-") else f"GPU-{text}"
    return str(dev.index)


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)  # let the first sample land before the timed region
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
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
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


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

def run_native(args, dist: Dist, peaks, peak_src):
    import torch
    import dense_tiled_gemm_03_gb300 as gt
    from dense_tiled_gemm_03_gb300 import build as native_build
    from dense_tiled_gemm_03_gb300.workloads import WORKLOADS, workload_operands

    if dist.rank == 0 or not native_build.LIBRARY.exists():
        native_build.build()
    dist.barrier()
    w = WORKLOADS[args.workload]
    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    a_cpu, b_cpu = workload_operands(w)
    a, b = a_cpu.to(dev), b_cpu.to(dev)
    c = torch.empty((w.m, w.n), dtype=a.dtype, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    cfg_name = gt.gemm_tn_config_name(gt.gemm_tn_select_config(int(w.dtype == "bf16"), w.m, w.n, w.k))
    op_bytes = (w.m * w.k + w.n * w.k) * 2
    flush = op_bytes < 2 * L2_BYTES
    scratch = torch.empty(L2_BYTES * 2 // 4, dtype=torch.int32, device=dev) if flush else None
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
        # the fused kernels: single-CTA 128 x 128 tiles where the plain choice is those, else pairs
        cfg_name = cfg_name if cfg_name == "1cta_n128" else ("1cta_n128" if w.m <= 128 else "2cta_n256")

        def step():
            gt.mm_tn_fused(a, b, out=c, alpha=alpha, bias=bias, activation=act, out_dtype=out_dtype, status=status)

    for _ in range(args.warmup):
        if flush:
            scratch.fill_(1)
        step()
    torch.cuda.synchronize(dev)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    region0 = torch.cuda.Event(enable_timing=True)
    region1 = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(gpu_smi_id(dev))
    if dist.rank == 0:
        sampler.start()
    dist.barrier()
    torch.cuda.synchronize(dev)
    launches0 = gt.gemm_tn_launch_count()
    region0.record(stream)
    for i in range(args.steps):
        if flush:
            scratch.fill_(1)   # write a buffer larger than L2 between timed launches
            starts[i].record(stream)
        step()
        if flush:
            ends[i].record(stream)
    region1.record(stream)
    launches = gt.gemm_tn_launch_count() - launches0   # this library's kernels in the timed region
    torch.cuda.synchronize(dev)
    dist.barrier()
    clocks = sampler.stop() if dist.rank == 0 else None
    if int(status.item()) != 0:
        raise RuntimeError(f"device watchdog fired: {gt.gemm_tn_status_string(int(status.item()))}")

    region_ms = region0.elapsed_time(region1)
    # With an L2 flush between launches the region includes the flushes: the
    # step time comes from events around each launch. Otherwise the launches
    # run back to back between the region's two events (events between
    # launches would add their own gaps).
    avg_launch_ms = (sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / args.steps if flush
                     else region_ms / args.steps)
    step_ms = avg_launch_ms
    step_ms = dist.max(step_ms)
    avg_launch_ms = dist.max(avg_launch_ms)
    value = dist.world * w.flops / (step_ms * 1e-3) / 1e12

    # roofline of the dominant (only) kernel of the step
    tensor_peak = float(peaks["bf16_tflops"])
    hbm_peak = float(peaks["hbm_gbs"])
    # algorithmic bytes: each operand read once, C written once (in its own element size)
    compulsory = (w.m * w.k + w.n * w.k) * 2 + w.m * w.n * c_elem
    hbm_bound = hbm_peak * 1e9 * (w.flops / compulsory) < tensor_peak * 1e12
    if hbm_bound:
        achieved = compulsory / (avg_launch_ms * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                    "frac": round(achieved / hbm_peak, 4)}
    else:
        achieved = w.flops / (avg_launch_ms * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": tensor_peak, "unit": "TFLOP/s",
                    "frac": round(achieved / tensor_peak, 4),
                    "frac_of_sustained": round(achieved / float(peaks.get("bf16_tflops_sustained", tensor_peak)), 4)}
    roofline["traffic"] = (NCU_TRAFFIC_BYTES.get((w.name, cfg_name)) if fused is None
                           else NCU_TRAFFIC_FUSED_BYTES.get((w.name, cfg_name, args.epilogue)))
    roofline["algorithmic_bytes"] = compulsory
    roofline["peak_source"] = f"{peak_src} ({'hbm_gbs' if hbm_bound else 'bf16_tflops'} burst; kernel timed alone)"
    roofline["kernel"] = ("gemm_tn_decode_kernel" if cfg_name == "1cta_decode_splitk"
                          else "gemm_tn_splitk_kernel" if cfg_name.endswith("splitk")
                          else f"gemm_tn_sm103_kernel<{cfg_name}>" if fused is None
                          else f"gemm_tn_sm103_kernel<{cfg_name}, fused>")

    # end to end through the host-buffer entry point (the plain GEMM only)
    e2e = None
    if fused is None:
        pin_a, pin_b = a_cpu.pin_memory(), b_cpu.pin_memory()
        pin_c = torch.empty((w.m, w.n), dtype=a_cpu.dtype).pin_memory()
        gt.mm_tn_host(pin_a, pin_b, out=pin_c, device=dev)   # warm
        dist.barrier()
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            gt.mm_tn_host(pin_a, pin_b, out=pin_c, device=dev)
        e2e_s = dist.max((time.perf_counter() - t0) / max(args.e2e_steps, 1))
        e2e = {"value": round(dist.world * w.flops / e2e_s / 1e12, 2), "unit": "TFLOP/s",
               "h2d_bytes_per_step": op_bytes, "d2h_bytes_per_step": w.m * w.n * 2 + 4,
               "steps": args.e2e_steps, "entry_point": "gemm_tn_host (pinned host buffers)"}

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": dist.world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic",
        "config": {"workload": w.name, "m": w.m, "n": w.n, "k": w.k, "dist": w.dist, "seed": w.seed,
                   "kernel_config": cfg_name, "parallelism": f"replicas x{dist.world}" if dist.world > 1 else "single GPU",
                   "l2": "L2 flushed between launches" if flush else
                   f"inputs larger than L2 ({op_bytes / 1e6:.0f} MB of operands vs {L2_BYTES / 1e6:.0f} MB)",
                   "accumulate": "fp32", "epilogue": args.epilogue},
        "pct_of_peak": round(100 * w.flops / (avg_launch_ms * 1e-3) / 1e12 / tensor_peak, 2),
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if args.cublas_context:
        # the same operands through torch.matmul (cuBLAS), timed the same way
        ref_c = torch.empty((w.m, w.n), dtype=a.dtype, device=dev)
        for _ in range(args.warmup):
            if flush:
                scratch.fill_(1)
            torch.matmul(a, b.t(), out=ref_c)
        torch.cuda.synchronize(dev)
        times = []
        r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        r0.record(stream)
        for _ in range(args.steps):
            if flush:
                scratch.fill_(1)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
            torch.matmul(a, b.t(), out=ref_c)
            if flush:
                e1.record(stream)
                times.append((e0, e1))
        r1.record(stream)
        torch.cuda.synchronize(dev)
        ms = (sum(x.elapsed_time(y) for x, y in times) / len(times) if flush
              else r0.elapsed_time(r1) / args.steps)
        cublas_tflops = w.flops / (ms * 1e-3) / 1e12
        line["context"] = {"cublas_tflops": round(cublas_tflops, 2),
                           "ratio_to_cublas": round(w.flops / (avg_launch_ms * 1e-3) / 1e12 / cublas_tflops, 4),
                           "what": "torch.matmul(a, b.T) on the same operands, timed the same way"}
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        v, cores, sample = cpu_oracle_rate(a_cpu, b_cpu, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(v, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                "sample": sample}
    return line


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


def run_native_attn(args, dist: Dist, peaks, peak_src):
    import torch
    import dense_tiled_gemm_03_gb300 as gt
    from dense_tiled_gemm_03_gb300 import build as native_build
    from dense_tiled_gemm_03_gb300.workloads import ATTN_WORKLOADS, make_qkv

    if dist.rank == 0 or not native_build.LIBRARY.exists():
        native_build.build()
    dist.barrier()
    w = ATTN_WORKLOADS[args.workload]
    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    q_cpu, k_cpu, v_cpu = make_qkv(w.batch, w.seq, w.heads, w.dim, w.dtype, seed=w.seed)
    q, k, v = q_cpu.to(dev), k_cpu.to(dev), v_cpu.to(dev)
    o = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    tensor_bytes = q.numel() * 2
    io_bytes = 4 * tensor_bytes   # Q, K, V read once, O written once
    flush = io_bytes < 2 * L2_BYTES
    scratch = torch.empty(L2_BYTES * 2 // 4, dtype=torch.int32, device=dev) if flush else None

    def step():
        gt.flash_attn(q, k, v, causal=w.causal, out=o, status=status)

    for _ in range(args.warmup):
        if flush:
            scratch.fill_(1)
        step()
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    region0 = torch.cuda.Event(enable_timing=True)
    region1 = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(gpu_smi_id(dev))
    if dist.rank == 0:
        sampler.start()
    dist.barrier()
    torch.cuda.synchronize(dev)
    launches0 = gt.gemm_tn_launch_count()
    region0.record(stream)
    for i in range(args.steps):
        if flush:
            scratch.fill_(1)
            starts[i].record(stream)
        step()
        if flush:
            ends[i].record(stream)
    region1.record(stream)
    launches = gt.gemm_tn_launch_count() - launches0   # this library's kernels in the timed region
    torch.cuda.synchronize(dev)
    dist.barrier()
    clocks = sampler.stop() if dist.rank == 0 else None
    if int(status.item()) != 0:
        raise RuntimeError(f"device watchdog fired: {gt.gemm_tn_status_string(int(status.item()))}")
    avg_launch_ms = (sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / args.steps if flush
                     else region0.elapsed_time(region1) / args.steps)
    step_ms = avg_launch_ms
    step_ms = dist.max(step_ms)
    avg_launch_ms = dist.max(avg_launch_ms)
    value = dist.world * w.flops / (step_ms * 1e-3) / 1e12
    tensor_peak = float(peaks["bf16_tflops"])
    achieved = w.flops / (avg_launch_ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": tensor_peak, "unit": "TFLOP/s",
                "frac": round(achieved / tensor_peak, 4),
                "frac_of_sustained": round(achieved / float(peaks.get("bf16_tflops_sustained", tensor_peak)), 4),
                "traffic": NCU_TRAFFIC_ATTN_BYTES.get(w.name), "algorithmic_bytes": io_bytes,
                "peak_source": f"{peak_src} (bf16_tflops burst; kernel timed alone)",
                "kernel": f"flash_attn_fwd_kernel<dim {w.dim}, {w.dtype}>"}

    # end to end: pinned host Q, K, V in, O back to pinned host memory, each step
    pins = [t.pin_memory() for t in (q_cpu, k_cpu, v_cpu)]
    pin_o = torch.empty_like(q_cpu).pin_memory()
    dq, dk, dv, do = (torch.empty_like(q) for _ in range(4))

    def e2e_step():
        for dst, src in zip((dq, dk, dv), pins):
            dst.copy_(src, non_blocking=True)
        gt.flash_attn(dq, dk, dv, causal=w.causal, out=do, status=status)
        pin_o.copy_(do, non_blocking=True)
        torch.cuda.current_stream(dev).synchronize()

    e2e_step()
    dist.barrier()
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        e2e_step()
    e2e_s = dist.max((time.perf_counter() - t0) / args.e2e_steps)
    e2e = {"value": round(dist.world * w.flops / e2e_s / 1e12, 2), "unit": "TFLOP/s",
           "h2d_bytes_per_step": 3 * tensor_bytes, "d2h_bytes_per_step": tensor_bytes, "steps": args.e2e_steps,
           "entry_point": "flash_attn_fwd with pinned host copies on the same stream"}
    line = {
        "metric": ATTN_METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": dist.world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "seq": w.seq, "heads": w.heads, "dim": w.dim,
                   "causal": w.causal, "seed": w.seed,
                   "parallelism": f"replicas x{dist.world}" if dist.world > 1 else "single GPU",
                   "l2": "L2 flushed between launches" if flush else
                   f"inputs larger than L2 ({io_bytes / 1e6:.0f} MB of Q, K, V and O vs {L2_BYTES / 1e6:.0f} MB)",
                   "accumulate": "fp32"},
        "pct_of_peak": round(100 * achieved / tensor_peak, 2),
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        rate, cores, sample = cpu_oracle_attn_rate(w, q_cpu, k_cpu, v_cpu, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(rate, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                "sample": sample}
    return line


def run_reference_attn(args, dist: Dist):
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
        "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "seq": w.seq, "heads": w.heads, "dim": w.dim,
                   "causal": w.causal, "seed": w.seed},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------------ reference arm

def run_reference(args, dist: Dist):
    """The CPU oracle, timed as it stands on this host's cores: each step is a
    bounded row sample of the workload, sized so the whole run takes about
    --ref-seconds (two minutes by default)."""
    from dense_tiled_gemm_03_gb300.workloads import WORKLOADS, workload_operands
    import oracle

    w = WORKLOADS[args.workload]
    a_cpu, b_cpu = workload_operands(w)
    cores = oracle.host_threads()
    total = args.steps + args.warmup
    # calibrate rows per step against a ~120 s budget for the whole run
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
        "n_gpus": dist.world,
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


def main():
    args = parse_args()
    if args.config:
        os.environ["GEMM_TN_FORCE_CONFIG"] = args.config
    if args.gpus < 1:
        raise SystemExit("--gpus must be >= 1")
    if args.epilogue != "none" and (args.workload.startswith("attn_") or args.impl == "reference"):
        raise SystemExit("--epilogue applies to the native GEMM workloads only")
    if args.oracle_table:
        oracle_table()
        return
    dist = Dist()
    try:
        attn = args.workload.startswith("attn_")
        if args.impl == "reference":
            if dist.rank == 0:
                line = run_reference_attn(args, dist) if attn else run_reference(args, dist)
                print(json.dumps(line), flush=True)
            return
        peaks, src = load_peaks()
        line = run_native_attn(args, dist, peaks, src) if attn else run_native(args, dist, peaks, src)
        if dist.rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
