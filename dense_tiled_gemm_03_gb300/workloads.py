"""Seeded synthetic operands for C = A x B^T.

This module only draws inputs; it holds none of the product's arithmetic, and
both the CUDA path's tests/benchmark and the oracle read the same arrays from it.

Recipe (every workload): a numpy ``Generator(PCG64(seed))`` draws A [M, K] first
and then B [N, K] in row-major order, in fp32; the fp32 values are rounded to
nearest-even into the storage dtype (fp16 or bf16) by torch on the CPU.
``uniform`` draws from [-1, 1); ``normal_over_sqrt_k`` draws a standard normal
and divides it by sqrt(K) in fp32.

The five workloads are the shapes the pages measure or model: square fp16
matmuls ("0. A Minimal Hopper Matmul", sections "Running the Kernel" and
"Performance"), the N = 8192 BF16 matmul of "Tiling a matmul" (section "Code"),
a ragged shape whose M, N, K divide no tile ("Tiling a matmul", "Where it
breaks": edge tiles) and a skinny low-reuse shape (same section: small M).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str            # "fp16" or "bf16": storage dtype of A, B and C
    m: int
    n: int
    k: int
    dist: str             # "uniform" or "normal_over_sqrt_k"
    seed: int

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    @property
    def flops(self) -> int:
        return 2 * self.m * self.n * self.k


WORKLOADS = {
    w.name: w for w in [
        Workload("fp16_256x256x256", "fp16", 256, 256, 256, "uniform", 1001),
        Workload("fp16_4096x4096x4096", "fp16", 4096, 4096, 4096, "normal_over_sqrt_k", 1002),
        Workload("bf16_8192x8192x8192", "bf16", 8192, 8192, 8192, "uniform", 1003),
        Workload("fp16_3001x5003x4097", "fp16", 3001, 5003, 4097, "uniform", 1004),
        Workload("bf16_128x16384x16384", "bf16", 128, 16384, 16384, "normal_over_sqrt_k", 1005),
        # decode-like: a few rows against a square weight (few output tiles, long K)
        Workload("bf16_8x4096x4096", "bf16", 8, 4096, 4096, "normal_over_sqrt_k", 1006),
    ]
}

#: The headline shape: C = A x B^T, bf16, M = N = K = 8192.
HEADLINE = "bf16_8192x8192x8192"


def _draw(gen: np.random.Generator, rows: int, cols: int, dist: str, k: int) -> np.ndarray:
    if dist == "uniform":
        return gen.uniform(-1.0, 1.0, size=(rows, cols)).astype(np.float32)
    if dist == "normal_over_sqrt_k":
        x = gen.standard_normal(size=(rows, cols), dtype=np.float32)
        return x / np.float32(np.sqrt(np.float32(k)))
    if dist == "int_small":
        return gen.integers(-2, 3, size=(rows, cols)).astype(np.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def make_operands(m: int, n: int, k: int, dtype: str | torch.dtype, dist: str = "uniform",
                  seed: int = 0) -> tuple[torch.Tensor, torch.Tensor]:
    """A [m, k] and B [n, k] on the CPU, contiguous, in the storage dtype."""
    tdt = DTYPES[dtype] if isinstance(dtype, str) else dtype
    gen = np.random.Generator(np.random.PCG64(seed))
    a = torch.from_numpy(_draw(gen, m, k, dist, k)).to(tdt)
    b = torch.from_numpy(_draw(gen, n, k, dist, k)).to(tdt)
    return a, b


def workload_operands(w: Workload | str) -> tuple[torch.Tensor, torch.Tensor]:
    w = WORKLOADS[w] if isinstance(w, str) else w
    return make_operands(w.m, w.n, w.k, w.dtype, w.dist, w.seed)


# ---------------------------------------------------------------- attention

@dataclass(frozen=True)
class AttnWorkload:
    """Q, K, V and O of shape [batch, seq, heads, dim] ("TileLang: a tile
    language one level below Triton", section "FlashAttention: online softmax
    as tile code": its kernel's tensors are (batch, seq, heads, dim))."""
    name: str
    dtype: str            # storage dtype of Q, K, V and O
    batch: int
    seq: int
    heads: int
    dim: int
    causal: bool
    seed: int

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    @property
    def shape(self) -> tuple[int, int, int, int]:
        return (self.batch, self.seq, self.heads, self.dim)

    @property
    def flops(self) -> int:
        """Multiply-adds of the two products counted as 2 FLOP each: 4 * S^2 * D
        per batch and head, over the visible (query, key) pairs only when
        causal: S (S + 1) / 2 of the S^2."""
        pairs = self.seq * (self.seq + 1) // 2 if self.causal else self.seq * self.seq
        return 4 * self.batch * self.heads * pairs * self.dim


ATTN_WORKLOADS = {
    w.name: w for w in [
        # the section's own call: flash_attn(batch 1, heads 8, seq 1024, dim 64), fp16, causal
        AttnWorkload("attn_fp16_b1_s1024_h8_d64_causal", "fp16", 1, 1024, 8, 64, True, 2001),
        AttnWorkload("attn_fp16_b4_s4096_h16_d64_causal", "fp16", 4, 4096, 16, 64, True, 2002),
        AttnWorkload("attn_bf16_b2_s8192_h32_d128_causal", "bf16", 2, 8192, 32, 128, True, 2003),
        AttnWorkload("attn_bf16_b2_s4096_h16_d128", "bf16", 2, 4096, 16, 128, False, 2004),
    ]
}


def make_qkv(batch: int, seq: int, heads: int, dim: int, dtype: str | torch.dtype,
             seed: int = 0) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Q, K, V [batch, seq, heads, dim] on the CPU, contiguous, in the storage
    dtype: a numpy Generator(PCG64(seed)) draws Q, then K, then V as standard
    normals in fp32, rounded to nearest-even by torch."""
    tdt = DTYPES[dtype] if isinstance(dtype, str) else dtype
    gen = np.random.Generator(np.random.PCG64(seed))
    shape = (batch, seq, heads, dim)
    return tuple(torch.from_numpy(gen.standard_normal(size=shape, dtype=np.float32)).to(tdt)
                 for _ in range(3))
