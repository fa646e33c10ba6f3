"""Traffic, intensity and shared-memory model of a tiled matmul, plus the counted
tiled loop -- TEST INFRASTRUCTURE ONLY (part of the oracle).

Every function states the passage it restates. All arithmetic is exact integer
arithmetic except the derived ratios and times.

Pages:
  * "Tiling a matmul" (Hritesh Sonawane), sections "Counting traffic",
    "Shared memory sets the ceiling", "Code" (the traffic table and the 32 x 32
    naive-vs-tiled check) and "Try it" (rectangular tiles).
  * "TileLang: a tile language one level below Triton", section "Exercises"
    (shared memory of a 3-stage 128 x 128 x 64 fp16 pipeline).
"""
from __future__ import annotations

from math import ceil

#: bytes per element of bf16 / fp16 ("Tiling a matmul", section "Code").
ELEM_BYTES_16BIT = 2


# --------------------------------------------------------------------------
# Square N x N model, square T x T tiles ("Tiling a matmul", "Counting traffic")
# --------------------------------------------------------------------------

def square_read_elements(n: int, tile: int) -> int:
    """Global-memory element reads of a T-tiled N x N matmul.

    There are (N // T)^2 output tiles; each streams a T x N strip of one operand
    and an N x T strip of the other, 2*T*N elements, so the reads total
    2 * N^2 * (N // T) elements (= 2N^3 / T when T divides N)."""
    return 2 * n * n * (n // tile)


def square_write_elements(n: int) -> int:
    """The output is written once: N^2 elements."""
    return n * n


def square_traffic_elements(n: int, tile: int) -> int:
    """Closed form 2N^3/T + N^2 elements of HBM traffic with no cache reuse."""
    return square_read_elements(n, tile) + square_write_elements(n)


def square_traffic_bytes(n: int, tile: int, elem_bytes: int = ELEM_BYTES_16BIT) -> int:
    """Bytes moved, reads plus the single write of C ("Tiling a matmul", "Code")."""
    return square_traffic_elements(n, tile) * elem_bytes


def matmul_flops(m: int, n: int, k: int) -> int:
    """2*M*N*K: one multiply and one add per (i, j, k)."""
    return 2 * m * n * k


def traffic_table_row(n: int, tile: int, hbm_bytes_per_s: float, flops_per_s: float,
                      elem_bytes: int = ELEM_BYTES_16BIT) -> dict:
    """One row of the page's N = 8192 table: traffic in GB, intensity in FLOP per
    byte (writes included, as the printed figures are), and the times the
    traffic and the arithmetic would take at the given rates."""
    tb = square_traffic_bytes(n, tile, elem_bytes)
    flops = matmul_flops(n, n, n)
    return {
        "tile": tile,
        "traffic_gb": tb / 1e9,
        "flop_per_byte": flops / tb,
        "hbm_ms": tb / hbm_bytes_per_s * 1e3,
        "compute_ms": flops / flops_per_s * 1e3,
    }


# --------------------------------------------------------------------------
# Rectangular generalisation ("Tiling a matmul", "Try it": rectangular tiles)
# --------------------------------------------------------------------------

def rect_traffic_elements(m: int, n: int, k: int, tile_m: int, tile_n: int) -> int:
    """HBM element traffic of C[M,N] = A[M,K] x B[N,K]^T tiled tile_m x tile_n,
    with no cache reuse: every output tile reads the K-long strips of the rows
    of A and of B it covers (a ragged edge tile reads only the rows that exist),
    and C is written once. A is re-read once per tile column, B once per tile
    row: M*K*ceil(N/tile_n) + N*K*ceil(M/tile_m) + M*N."""
    return m * k * ceil(n / tile_n) + n * k * ceil(m / tile_m) + m * n


def rect_traffic_bytes(m: int, n: int, k: int, tile_m: int, tile_n: int,
                       elem_bytes: int = ELEM_BYTES_16BIT) -> int:
    return rect_traffic_elements(m, n, k, tile_m, tile_n) * elem_bytes


def compulsory_bytes(m: int, n: int, k: int, elem_bytes: int = ELEM_BYTES_16BIT) -> int:
    """Each operand read once and C written once: (M*K + N*K + M*N) elements."""
    return (m * k + n * k + m * n) * elem_bytes


def ideal_intensity(m: int, n: int, k: int, elem_bytes: int = ELEM_BYTES_16BIT) -> float:
    """FLOP per compulsory byte."""
    return matmul_flops(m, n, k) / compulsory_bytes(m, n, k, elem_bytes)


def roofline_flops(m: int, n: int, k: int, tensor_flops_per_s: float, hbm_bytes_per_s: float,
                   elem_bytes: int = ELEM_BYTES_16BIT) -> float:
    """min(dense tensor peak, HBM bandwidth x ideal intensity)."""
    return min(tensor_flops_per_s, hbm_bytes_per_s * ideal_intensity(m, n, k, elem_bytes))


# --------------------------------------------------------------------------
# Shared memory ("Tiling a matmul", "Shared memory sets the ceiling";
# TileLang page, "Exercises")
# --------------------------------------------------------------------------

def smem_tile_pair_bytes(tile: int, elem_bytes: int = ELEM_BYTES_16BIT) -> int:
    """A T x T tile of A plus a T x T tile of B."""
    return 2 * tile * tile * elem_bytes


def smem_pipeline_bytes(block_m: int, block_n: int, block_k: int, stages: int,
                        elem_bytes: int = ELEM_BYTES_16BIT) -> int:
    """Stages x (A tile block_m x block_k + B tile block_k x block_n)."""
    return stages * (block_m * block_k + block_k * block_n) * elem_bytes


def smem_b_offset(block_m: int, block_k: int, stages: int, elem_bytes: int = ELEM_BYTES_16BIT) -> int:
    """Offset of the first B buffer when all A stages are laid out first."""
    return stages * block_m * block_k * elem_bytes


def blocks_per_sm(smem_per_block: int, smem_per_sm: int) -> int:
    return smem_per_sm // smem_per_block


# --------------------------------------------------------------------------
# Naive and counted tiled loops ("Tiling a matmul", "Code": the 32 x 32 check)
# --------------------------------------------------------------------------

def naive_matmul(a, b, n: int, b_transposed: bool = False):
    """Plain N x N product from Python lists; each output is one dot product
    taken with Python's built-in float ``sum`` (compensated summation on
    Python >= 3.12, which is what reproduces the page's printed errors).
    With b_transposed, b is indexed [j][k] (C = A x B^T)."""
    if b_transposed:
        return [[sum(a[i][k] * b[j][k] for k in range(n)) for j in range(n)] for i in range(n)]
    return [[sum(a[i][k] * b[k][j] for k in range(n)) for j in range(n)] for i in range(n)]


def tiled_matmul_counted(a, b, n: int, tile: int, b_transposed: bool = False):
    """The same product computed tile by tile, counting element loads.

    Output tiles (bi, bj) of side T are visited in order; for each, the K axis is
    walked in T-wide steps. Each step stands for one shared-memory tile pair and
    loads 2*T*T elements; every output of the tile adds that step's partial dot
    product (a built-in ``sum`` over the step's T terms) to its running value
    with a plain floating-point add. Returns (c, loads). With b_transposed, b is
    indexed [j][k] (C = A x B^T); the counts do not depend on that choice."""
    c = [[0.0] * n for _ in range(n)]
    loads = 0
    for bi in range(0, n, tile):
        for bj in range(0, n, tile):
            for bk in range(0, n, tile):
                loads += 2 * tile * tile
                ks = range(bk, bk + tile)
                for i in range(bi, bi + tile):
                    for j in range(bj, bj + tile):
                        if b_transposed:
                            part = sum(a[i][k] * b[j][k] for k in ks)
                        else:
                            part = sum(a[i][k] * b[k][j] for k in ks)
                        c[i][j] += part
    return c, loads
