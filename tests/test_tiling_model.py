"""Pins for the oracle's tiling model against the pages' printed numbers.

"Tiling a matmul", sections "Counting traffic", "Code" (the printed output of
the 32 x 32 check and the N = 8192 table), "Shared memory sets the ceiling" and
"Try it"; "TileLang: a tile language one level below Triton", section
"Exercises" (answers 1 and 2).
"""
from __future__ import annotations

import json
import random
import sys
from math import ceil
from pathlib import Path

import pytest

from oracle import tiling_model as tm

GOLDEN = Path(__file__).resolve().parent / "golden"
P2 = json.loads((GOLDEN / "tiling_a_matmul_printed_output.json").read_text())
P3 = json.loads((GOLDEN / "tilelang_exercises_smem.json").read_text())


def _n32_inputs():
    case = P2["check_n32"]
    rng = random.Random(case["seed"])
    n = case["n"]
    a = [[rng.random() for _ in range(n)] for _ in range(n)]
    b = [[rng.random() for _ in range(n)] for _ in range(n)]
    return n, a, b


@pytest.mark.parametrize("row", P2["check_n32"]["rows"], ids=lambda r: f"t{r['tile']}")
def test_tiled_equals_naive_32(row):
    n, a, b = _n32_inputs()
    ref = tm.naive_matmul(a, b, n)
    c, loads = tm.tiled_matmul_counted(a, b, n, row["tile"])
    err = max(abs(c[i][j] - ref[i][j]) for i in range(n) for j in range(n))
    assert loads == row["element_loads"] == 2 * n ** 3 // row["tile"]
    assert err <= 1e-14
    if sys.version_info >= (3, 12):
        # built-in float sum is compensated from 3.12 on, as on the page's run
        assert f"{err:.1e}" == row["max_error"]


@pytest.mark.parametrize("tile", [1, 4, 16])
def test_tiled_equals_naive_transposed_b(tile):
    n, a, b = _n32_inputs()
    bt = [[b[k][j] for k in range(n)] for j in range(n)]  # B^T stored [N, K]
    ref = tm.naive_matmul(a, bt, n, b_transposed=True)
    c, loads = tm.tiled_matmul_counted(a, bt, n, tile, b_transposed=True)
    c0, loads0 = tm.tiled_matmul_counted(a, b, n, tile)
    assert loads == loads0
    assert c == c0  # same terms in the same order
    assert max(abs(c[i][j] - ref[i][j]) for i in range(n) for j in range(n)) <= 1e-14


def test_traffic_table_n8192():
    t = P2["traffic_n8192"]
    n = t["n"]
    assert f"{tm.matmul_flops(n, n, n) / 1e12:.1f}" == t["total_tflop"]
    for row in t["rows"]:
        got = tm.traffic_table_row(n, row["tile"], t["hbm_bytes_per_s"], t["flops_per_s"], t["elem_bytes"])
        assert f"{got['traffic_gb']:.1f}" == row["traffic_gb"]
        assert f"{got['flop_per_byte']:.1f}" == row["flop_per_byte"]
        assert f"{got['hbm_ms']:.2f}" == row["hbm_ms"]
        assert f"{got['compute_ms']:.2f}" == row["compute_ms"]


# Tiles named by the workloads: the page's table tiles plus the tile shapes this
# library runs (128 x 128, 128 x 256 and the 256 x 256 pair tile).
@pytest.mark.parametrize("n", [256, 4096, 8192])
@pytest.mark.parametrize("tile", [1, 16, 32, 64, 128, 256])
def test_closed_form_2n3_over_t_plus_n2(n, tile):
    assert tm.square_traffic_elements(n, tile) == 2 * n ** 3 // tile + n * n
    assert tm.square_traffic_bytes(n, tile) == 2 * (2 * n ** 3 // tile + n * n)


def _count_rect_by_tiles(m, n, k, tile_m, tile_n):
    """Brute-force count: visit every output tile and add the strips it reads."""
    total = 0
    for i0 in range(0, m, tile_m):
        for j0 in range(0, n, tile_n):
            rows_a = min(tile_m, m - i0)
            rows_b = min(tile_n, n - j0)
            total += (rows_a + rows_b) * k
    return total + m * n


@pytest.mark.parametrize("shape", [(64, 64, 64, 16, 16), (100, 37, 9, 16, 32), (3001, 5003, 4097, 128, 256),
                                   (128, 16384, 16384, 128, 128), (8192, 8192, 8192, 256, 256)])
def test_rect_traffic_matches_tile_count(shape):
    m, n, k, tmm, tnn = shape
    assert tm.rect_traffic_elements(m, n, k, tmm, tnn) == _count_rect_by_tiles(m, n, k, tmm, tnn)


@pytest.mark.parametrize("n,tile", [(8192, 128), (8192, 256), (4096, 64)])
def test_rect_reduces_to_square(n, tile):
    assert tm.rect_traffic_bytes(n, n, n, tile, tile) == tm.square_traffic_bytes(n, tile)


def test_rect_exercise_128x256_vs_181x181():
    n = 8192
    r1 = tm.rect_traffic_elements(n, n, n, 128, 256)
    r2 = tm.rect_traffic_elements(n, n, n, 181, 181)
    # both tiles have about the same area: 128 x 256 re-reads the operands
    # 32 + 64 = 96 times, 181 x 181 (46 ragged tiles a side) 46 + 46 = 92 times
    assert r1 == n * n * ceil(n / 256) + n * n * ceil(n / 128) + n * n
    assert r2 == 2 * n * n * ceil(n / 181) + n * n
    assert (r1 - n * n) // (n * n) == 96 and (r2 - n * n) // (n * n) == 92


def test_intensity_is_about_t_over_2():
    # "Counting traffic": intensity ~ T/2 FLOP per byte in BF16, ignoring writes
    n = 8192
    for t in (64, 128, 256):
        reads_bytes = 2 * tm.square_read_elements(n, t)
        assert tm.matmul_flops(n, n, n) / reads_bytes == pytest.approx(t / 2)


def test_smem_per_tile_pair():
    for row in P2["smem_tile_pair_kib"]:
        assert tm.smem_tile_pair_bytes(row["tile"]) // 1024 == row["kib"]
    c = P2["smem_ceiling"]
    assert tm.smem_tile_pair_bytes(c["tile"]) // 1024 == c["pair_kb"]
    assert c["stages"] * tm.smem_tile_pair_bytes(c["tile"]) // 1024 == c["stages_kb"] < c["h100_smem_kb"]


def test_tilelang_exercise_smem():
    bm, bn, bk, e = P3["block_m"], P3["block_n"], P3["block_k"], P3["elem_bytes"]
    assert bm * bk * e // 1024 == P3["per_operand_stage_kb"]
    assert tm.smem_pipeline_bytes(bm, bn, bk, 1, e) // 1024 == P3["per_stage_kb"]
    s3 = tm.smem_pipeline_bytes(bm, bn, bk, 3, e)
    assert s3 // 1024 == P3["stages_3_kb"]
    assert tm.smem_b_offset(bm, bk, 3, e) == P3["b_shared_offset_bytes"]
    assert tm.blocks_per_sm(s3, P3["h100_smem_per_sm_kb"] * 1024) == P3["blocks_per_sm_at_3_stages"]
    assert tm.smem_pipeline_bytes(bm, bn, bk, 2, e) // 1024 == P3["stages_2_kb"]
    assert tm.smem_pipeline_bytes(bm, bn, bk, 4, e) // 1024 == P3["stages_4_kb"]


def test_roofline_helpers():
    # compulsory traffic and the roofline of the 8192^3 shape
    n = 8192
    assert tm.compulsory_bytes(n, n, n) == 3 * n * n * 2
    assert tm.ideal_intensity(n, n, n) == pytest.approx(2 * n ** 3 / (6 * n * n))
    assert tm.roofline_flops(n, n, n, 2e15, 8e12) == 2e15
    assert tm.roofline_flops(128, 16384, 16384, 2e15, 8e12) == pytest.approx(
        8e12 * tm.ideal_intensity(128, 16384, 16384))
