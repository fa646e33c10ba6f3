"""gemm_tn_ex_noalloc: the entry point for callers that cannot allocate device
memory (a framework that has reserved the GPU's memory for its own pool, or a
code path that must not block or fail on an allocation). It must give the
results gemm_tn_ex gives, taking the repack scratch from the library's static
device array instead of cudaMallocAsync, and reject problems that would need
more scratch than that array holds.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import dense_tiled_gemm_03_gb300 as gt
import oracle
from dense_tiled_gemm_03_gb300.workloads import make_operands

from _parity import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    from dense_tiled_gemm_03_gb300 import build as native_build
    native_build.build()


def _padded(t: torch.Tensor, pad: int, dev) -> torch.Tensor:
    """A device view of t whose row pitch is t's width + pad elements."""
    rows, cols = t.shape
    big = torch.zeros((rows, cols + pad), dtype=t.dtype)
    big[:, :cols] = t
    return big.to(dev)[:, :cols]


def _call(fn, a, b, c, status):
    dtype = gt.GEMM_TN_BF16 if a.dtype == torch.bfloat16 else gt.GEMM_TN_F16
    m, k = a.shape
    n = b.shape[0]
    return fn(dtype, m, n, k, a.data_ptr(), a.stride(0), b.data_ptr(), b.stride(0), c.data_ptr(), c.stride(0),
              status.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("dtype,mnk,pads", [
    ("fp16", (301, 503, 409), (0, 0, 0)),     # K = 409: both row pitches misaligned -> both repacked
    ("bf16", (257, 640, 1000), (3, 0, 5)),    # A padded to an odd pitch, B aligned, C odd pitch
    ("fp16", (512, 384, 256), (0, 0, 0)),     # aligned: no scratch used at all
])
def test_noalloc_matches_gemm_tn_ex_on_two_calls_in_a_row(dtype, mnk, pads):
    m, n, k = mnk
    dev = torch.device("cuda", 0)
    a_cpu, b_cpu = make_operands(m, n, k, dtype, "uniform", seed=m + n + k)
    a = _padded(a_cpu, pads[0], dev)
    b = _padded(b_cpu, pads[1], dev)
    c_ref = _padded(torch.full((m, n), float("nan"), dtype=a.dtype), pads[2], dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    assert _call(gt.gemm_tn_ex, a, b, c_ref, status) == gt.GEMM_TN_OK
    torch.cuda.synchronize()
    ref, bound = oracle.gemm_tn_reference(a_cpu, b_cpu)
    allowance = oracle.ALLOW_REL * bound + oracle.ALLOW_ABS
    expected = c_ref.cpu().double().numpy()
    for call in range(2):
        c = _padded(torch.full((m, n), float("nan"), dtype=a.dtype), pads[2], dev)
        rc = _call(gt.gemm_tn_ex_noalloc, a, b, c, status)
        assert rc == gt.GEMM_TN_OK, gt.gemm_tn_last_error_message()
        torch.cuda.synchronize()
        got = c.cpu().double().numpy()
        assert np.isfinite(got).all(), f"call {call}: unwritten output"
        assert (np.abs(got - expected) <= allowance).all(), f"call {call}: differs from gemm_tn_ex"
        assert oracle.parity_report(got, ref, bound).ok, f"call {call}: fails the oracle criterion"
    assert int(status.item()) == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    """Repacking A and B of 8192 x 4097 fp16 needs 2 * 8192 * 4104 * 2 bytes,
    more than the 64 MiB static scratch: rejected, nothing written."""
    m = n = 8192
    k = 4097
    dev = torch.device("cuda", 0)
    a = torch.zeros((m, k), dtype=torch.float16, device=dev)
    b = torch.zeros((n, k), dtype=torch.float16, device=dev)
    c = torch.full((m, n), 7.0, dtype=torch.float16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    rc = _call(gt.gemm_tn_ex_noalloc, a, b, c, status)
    assert rc == gt.GEMM_TN_ERR_INVALID_VALUE
    assert "static scratch" in gt.gemm_tn_last_error_message()
    torch.cuda.synchronize()
    assert (c == 7.0).all()
    assert gt.GEMM_TN_NOALLOC_SCRATCH_BYTES == 64 * 1024 * 1024


# CUmemPool_attribute values (cuda.h): bytes of the pool in use now, and the
# high-water mark of that since it was last reset (setting it to 0 resets it
# to the current use)
_POOL_USED_MEM_CURRENT = 7
_POOL_USED_MEM_HIGH = 8


def _current_pool(ordinal: int):
    """The memory pool cudaMallocAsync draws from on device `ordinal` (its
    current pool), through the driver API."""
    cuda = ctypes.CDLL("libcuda.so.1")
    assert cuda.cuInit(0) == 0
    dev = ctypes.c_int()
    assert cuda.cuDeviceGet(ctypes.byref(dev), ordinal) == 0
    pool = ctypes.c_void_p()
    assert cuda.cuDeviceGetMemPool(ctypes.byref(pool), dev) == 0
    return cuda, pool


def _pool_attr(cuda, pool, attr: int) -> int:
    v = ctypes.c_uint64()
    assert cuda.cuMemPoolGetAttribute(pool, attr, ctypes.byref(v)) == 0
    return v.value


def _reset_high(cuda, pool) -> None:
    zero = ctypes.c_uint64(0)
    assert cuda.cuMemPoolSetAttribute(pool, _POOL_USED_MEM_HIGH, ctypes.byref(zero)) == 0


def test_noalloc_allocates_nothing_where_gemm_tn_ex_does():
    """A problem whose operands both need the padded copy (K = 409: odd row
    pitches). gemm_tn_ex takes that copy from the library's workspace pool, so
    the pool's high-water mark rises by at least its size (the control);
    gemm_tn_ex_noalloc on the same problem leaves the high-water marks of that
    pool and of the device's current pool (the one cudaMallocAsync uses) where
    they were, and both calls give the same results."""
    m, n, k = 301, 503, 409
    dev = torch.device("cuda", 0)
    a_cpu, b_cpu = make_operands(m, n, k, "fp16", "uniform", seed=99)
    a, b = a_cpu.to(dev), b_cpu.to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    c_noalloc = torch.full((m, n), float("nan"), dtype=a.dtype, device=dev)
    c_ex = torch.full((m, n), float("nan"), dtype=a.dtype, device=dev)
    torch.cuda.synchronize()
    cuda, device_pool = _current_pool(0)
    lib_pool = ctypes.c_void_p(gt.gemm_tn_workspace_pool())
    assert lib_pool.value, "no workspace pool on the device"
    pools = {"device": device_pool, "library": lib_pool}
    used0 = {name: _pool_attr(cuda, p, _POOL_USED_MEM_CURRENT) for name, p in pools.items()}

    for p in pools.values():
        _reset_high(cuda, p)
    assert _call(gt.gemm_tn_ex_noalloc, a, b, c_noalloc, status) == gt.GEMM_TN_OK
    torch.cuda.synchronize()
    for name, p in pools.items():
        assert _pool_attr(cuda, p, _POOL_USED_MEM_HIGH) == used0[name], f"the no-alloc call allocated from the {name} pool"

    _reset_high(cuda, lib_pool)
    assert _call(gt.gemm_tn_ex, a, b, c_ex, status) == gt.GEMM_TN_OK
    torch.cuda.synchronize()
    # the padded copies: rows of round_up(409, 8) = 416 elements, each copy
    # rounded up to 256 bytes
    padded = (-(-m * 416 * 2 // 256) + -(-n * 416 * 2 // 256)) * 256
    assert _pool_attr(cuda, lib_pool, _POOL_USED_MEM_HIGH) >= used0["library"] + padded, \
        "control: gemm_tn_ex did not take its workspace from the pool"
    assert _pool_attr(cuda, lib_pool, _POOL_USED_MEM_CURRENT) == used0["library"], \
        "gemm_tn_ex did not give its workspace back"
    assert int(status.item()) == 0
    ref, bound = oracle.gemm_tn_reference(a_cpu, b_cpu)
    allowance = oracle.ALLOW_REL * bound + oracle.ALLOW_ABS
    got, expected = c_noalloc.cpu().double().numpy(), c_ex.cpu().double().numpy()
    assert np.isfinite(got).all() and (np.abs(got - expected) <= allowance).all()
