"""Host-side logic of bench.py on CPU: rank aggregation over world size 2
(gloo), the reference arm under torchrun (rank 0 alone prints), and the JSON
line's contract keys."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys
from pathlib import Path

import pytest
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parents[1]


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _dist_worker(rank: int, world: int, port: int, out_dir: str):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, str(ROOT))
    import bench
    d = bench.Dist()
    d.barrier()
    got = d.max(10.0 + rank)
    d.barrier()
    d.close()
    Path(out_dir, f"rank{rank}.txt").write_text(repr(got))


def test_dist_max_over_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.start_processes(_dist_worker, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn")
    assert [float((tmp_path / f"rank{r}.txt").read_text()) for r in range(2)] == [11.0, 11.0]


def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), str(ROOT / "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "1",
           "--workload", "fp16_256x256x256", "--ref-seconds", "2"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-3000:]
    lines = [json.loads(l) for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    for key in ("metric", "value", "unit", "steps", "warmup", "ms_per_step", "higher_is_better", "config",
                "cpu_baseline", "e2e"):
        assert key in line
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["value"] > 0 and line["unit"] == "TFLOP/s"


def test_reference_arm_single_process():
    cmd = [sys.executable, str(ROOT / "bench.py"), "--impl", "reference", "--steps", "2", "--warmup", "1",
           "--workload", "fp16_256x256x256", "--ref-seconds", "1"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-3000:]
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 1
    assert line["config"]["workload"] == "fp16_256x256x256"


def test_reference_arm_attention_workload():
    """--workload attn_* times the attention oracle on a bounded row sample and
    prints the same line with the attention metric."""
    cmd = [sys.executable, str(ROOT / "bench.py"), "--impl", "reference", "--steps", "2", "--warmup", "1",
           "--workload", "attn_fp16_b1_s1024_h8_d64_causal", "--ref-seconds", "2"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-3000:]
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["config"]["workload"] == "attn_fp16_b1_s1024_h8_d64_causal" and line["config"]["causal"] is True
    assert "attention" in line["metric"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_attention_row_sample_and_flop_count():
    """The oracle samples' FLOP count is the visible-pair count of the rows."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", ROOT / "bench.py")
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    from dense_tiled_gemm_03_gb300.workloads import ATTN_WORKLOADS
    w = ATTN_WORKLOADS["attn_fp16_b1_s1024_h8_d64_causal"]
    rows = bench.attn_sample_rows(w, 1e18)
    assert rows == list(range(w.seq))
    assert bench.attn_rows_flops(w, rows) == w.flops
    few = bench.attn_sample_rows(w, w.flops / 10)
    assert 0 < len(few) < w.seq and few == sorted(set(few))


def test_epilogue_option_scope():
    """--epilogue names the fused paths the benchmark can time; it is refused
    for attention workloads and the reference arm before any device work."""
    sys.path.insert(0, str(ROOT))
    import bench
    assert set(bench.EPILOGUES) == {"none", "bias", "bias_gelu", "fp32", "e4m3"}
    assert bench.EPILOGUES["none"] is None
    alpha, with_bias, act, out = bench.EPILOGUES["e4m3"]
    assert out == "float8_e4m3fn" and 0.0 < alpha < 1.0 and act == "none"
    for extra in (["--workload", "attn_bf16_b2_s8192_h32_d128_causal"], ["--impl", "reference"]):
        r = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--epilogue", "e4m3", *extra],
                           capture_output=True, text=True, timeout=120)
        assert r.returncode != 0 and "native GEMM workloads only" in r.stderr
