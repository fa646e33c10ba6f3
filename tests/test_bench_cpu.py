"""Host-side logic of bench.py on CPU: the native arm's refusal of several
GPUs, the reference arm under torchrun (rank 0 alone prints), the JSON line's
contract keys, the tile-traffic model and the provenance of stored ncu
figures."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_native_arm_refuses_several_gpus_without_loading_the_library():
    """The product runs on one GPU: launched for 2 GPUs (by flag, or as a rank
    of a 2-process job) the native arm prints one line saying so and exits 0
    without loading the CUDA library, so its cluster-multicast kernel never
    runs in a multi-GPU process."""
    probe = ("import json, sys; sys.path.insert(0, {root!r}); import bench; bench.main({argv!r}); "
             "maps = open('/proc/self/maps').read(); "
             "print(json.dumps({{'loaded': 'libgemm_tn' in maps, "
             "'binding': 'dense_tiled_gemm_03_gb300._native' in sys.modules}}))")
    for argv, env in ((["--gpus", "2"], {}), ([], {"WORLD_SIZE": "2", "RANK": "0"}),
                      (["--gpus", "2"], {"WORLD_SIZE": "2", "RANK": "1"})):
        res = subprocess.run([sys.executable, "-c", probe.format(root=str(ROOT), argv=argv)],
                             capture_output=True, text=True, timeout=300, cwd=ROOT, env={**os.environ, **env})
        assert res.returncode == 0, res.stderr[-3000:]
        lines = [json.loads(l) for l in res.stdout.splitlines() if l.startswith("{")]
        probe_out = lines[-1]
        assert probe_out == {"loaded": False, "binding": False}
        printed = lines[:-1]
        if env.get("RANK") == "1":
            assert printed == []          # only rank 0 prints
        else:
            assert len(printed) == 1 and "unavailable" in printed[0] and printed[0]["n_gpus"] == 2


def test_modelled_traffic_matches_the_oracle_model():
    """The benchmark's tile-traffic model is the oracle's rectangular model
    (written twice, independently) for the tiles of every configuration."""
    import bench
    from oracle import tiling_model
    for (m, n, k) in [(8192, 8192, 8192), (4096, 4096, 4096), (3001, 5003, 4097), (128, 16384, 16384),
                      (256, 256, 256), (8, 4096, 4096)]:
        for cfg in bench.TILE_OF_CONFIG:
            tm, tn = bench.tile_of(cfg, m)
            assert bench.modelled_traffic_bytes(m, n, k, tm, tn) == tiling_model.rect_traffic_bytes(m, n, k, tm, tn)
    # the headline on CTA-pair tiles: A and B each read 32 times, C written once
    assert bench.modelled_traffic_bytes(8192, 8192, 8192, 256, 256) == 2 * (2 * 8192 * 8192 * 32) + 2 * 8192 ** 2


def test_stored_traffic_goes_stale_with_the_sources():
    import bench
    digest = bench.source_digest()
    assert len(digest) == 12 and digest == bench.source_digest()
    entry = {"bytes": 123, "kernel": "k", "when": "d", "source": digest}
    assert bench.stored_traffic(entry, digest)[0] == 123
    got, why = bench.stored_traffic(dict(entry, source="000000000000"), digest)
    assert got is None and why.startswith("stale")
    assert bench.stored_traffic(None, digest)[0] is None
    for e in list(bench.NCU_TRAFFIC.values()) + list(bench.NCU_TRAFFIC_ATTN.values()):
        assert set(e) >= {"bytes", "kernel", "when", "source"}


def test_cpulist_round_trip():
    import bench
    assert bench.parse_cpulist("0-3,8,10-11\n") == {0, 1, 2, 3, 8, 10, 11}
    assert bench.format_cpulist({0, 1, 2, 3, 8, 10, 11}) == "0-3,8,10-11"
    assert bench.format_cpulist(set()) == ""


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
