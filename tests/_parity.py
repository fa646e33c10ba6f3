"""Helpers shared by the GPU parity tests: run C = A x B^T through the C ABI
and compare with the fp64 oracle element by element (or on sampled rows and
columns for the full-size workloads)."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
import dense_tiled_gemm_03_gb300 as gt


def require_gpu():
    import pytest
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    major, minor = torch.cuda.get_device_capability(0)
    assert (major, minor) == (10, 3), f"expected a GB300 (sm_103), got sm_{major}{minor}"


class env_var:
    """Context manager: set (or, with None, unset) one environment variable."""

    def __init__(self, key: str, value: str | None):
        self.key, self.value, self.old = key, value, None

    def __enter__(self):
        self.old = os.environ.get(self.key)
        if self.value is None:
            os.environ.pop(self.key, None)
        else:
            os.environ[self.key] = self.value
        return self

    def __exit__(self, *exc):
        if self.old is None:
            os.environ.pop(self.key, None)
        else:
            os.environ[self.key] = self.old


def forced_config(name: str | None):
    """Run the library with GEMM_TN_FORCE_CONFIG set to a configuration name."""
    return env_var("GEMM_TN_FORCE_CONFIG", name)


def epilogue_mode(mode: str):
    """"auto": TMA-store epilogue whenever C allows it; "direct": force the
    predicated element-store epilogue."""
    return env_var("GEMM_TN_EPILOGUE", "direct" if mode == "direct" else None)


def gpu_gemm(a_cpu: torch.Tensor, b_cpu: torch.Tensor, config: str | None = None, out_fill=float("nan"),
             epilogue: str = "auto"):
    """Copy A, B to cuda:0, run mm_tn (C pre-filled with NaN so every element
    must be written), return C on the CPU and the device status word."""
    dev = torch.device("cuda", 0)
    a = a_cpu.to(dev)
    b = b_cpu.to(dev)
    out = torch.full((a.shape[0], b.shape[0]), out_fill, dtype=a.dtype, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    with forced_config(config), epilogue_mode(epilogue):
        gt.mm_tn(a, b, out=out, status=status)
    torch.cuda.synchronize()
    return out.cpu(), int(status.item())


def assert_parity(c: torch.Tensor, a_cpu: torch.Tensor, b_cpu: torch.Tensor, label: str = ""):
    ref, bound = oracle.gemm_tn_reference(a_cpu, b_cpu)
    rep = oracle.parity_report(c, ref, bound)
    assert rep.ok, f"{label}: {rep}"
    return rep


def assert_sampled_parity(c: torch.Tensor, a_cpu: torch.Tensor, b_cpu: torch.Tensor, rows, cols, label=""):
    """Full-size check on a sample the oracle computes one by one: every column
    of the sampled rows, and every row of the sampled columns."""
    rows = torch.as_tensor(sorted(set(int(r) for r in rows)), dtype=torch.long)
    cols = torch.as_tensor(sorted(set(int(x) for x in cols)), dtype=torch.long)
    ref_r, bound_r = oracle.gemm_tn_reference(a_cpu.index_select(0, rows), b_cpu)
    rep_r = oracle.parity_report(c.index_select(0, rows), ref_r, bound_r)
    assert rep_r.ok, f"{label} sampled rows: {rep_r}"
    ref_c, bound_c = oracle.gemm_tn_reference(a_cpu, b_cpu.index_select(0, cols))
    rep_c = oracle.parity_report(c.index_select(1, cols), ref_c, bound_c)
    assert rep_c.ok, f"{label} sampled cols: {rep_c}"
    return rep_r, rep_c


def edge_indices(extent: int, tile: int, rng: np.random.Generator, extra: int) -> list[int]:
    """First/last index of every tile boundary region plus random picks."""
    picks = {0, extent - 1}
    for t in range(0, extent, tile):
        picks.update({t, min(t + tile - 1, extent - 1)})
    picks.update(int(x) for x in rng.integers(0, extent, size=extra))
    return sorted(p for p in picks if 0 <= p < extent)
