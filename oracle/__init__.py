"""The CPU oracle for C = A x B^T -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package. The product path (the CUDA
library and its Python binding) never imports it and shares no code with it.

Contents:
  * ``gemm_tn_reference``  -- the fp64 triple loop (C, ``gemm_oracle.c``): the
    plain product ref = A x B^T and the magnitude sum bound = sum |a*b|.
  * ``parity_report``      -- the element-wise pass criterion
        |c - ref| <= 1e-2 * bound + 1e-3
    with NaN/Inf anywhere in c counted as a failure.
  * ``tiling_model``       -- the traffic / shared-memory model and the counted
    tiled loop of "Tiling a matmul" (pure Python).
  * ``fused_reference``    -- the fused epilogue act(alpha * A x B^T + beta * C
    + bias) written out element by element on top of gemm_tn_reference, with
    ``fused_parity_report`` / ``fused_e4m3_parity_report`` carrying the
    criterion through it (the latter for the fp8 e4m3 output, ``fp8``).
  * ``attention_reference`` -- the attention forward pass that consumes the
    GEMM (C, ``attention_oracle.c``): O = softmax(scale * Q K^T, causal mask) V
    per batch and head, with bound = sum_j p_j |V_j|; checked with the same
    criterion by ``parity_report``.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``,
``tests/test_attention_oracle_pins.py`` and ``tests/test_tiling_model.py`` to values fixed by the pages or by mathematics
(exact rational brute force, identity/permutation/integer closed forms, the
pages' printed tables); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

from . import build as _build
from . import fp8

__all__ = ["attention_reference", "gemm_tn_reference", "gemm_nn_reference", "fused_reference", "fused_parity_report", "fused_e4m3_parity_report", "fp8", "parity_report", "ParityReport", "ALLOW_REL", "ALLOW_ABS",
           "host_threads", "load_library"]

#: The pass criterion's two constants: |c - ref| <= ALLOW_REL * bound + ALLOW_ABS.
ALLOW_REL = 1e-2
ALLOW_ABS = 1e-3

_LIBS: dict[tuple, ctypes.CDLL] = {}


def host_threads() -> int:
    """Threads the oracle uses: every core this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover - non-Linux
        return max(1, os.cpu_count() or 1)


def load_library(plant: int = 0, out_dir=None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle's C library."""
    key = (plant, str(out_dir))
    lib = _LIBS.get(key)
    if lib is not None:
        return lib
    path = _build.build(plant=plant, out_dir=out_dir)
    lib = ctypes.CDLL(str(path))
    fn = lib.oracle_gemm_tn_f64
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                   ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    fa = lib.oracle_attention_f64
    fa.restype = ctypes.c_int
    fa.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                   ctypes.c_int64, ctypes.c_int64, ctypes.c_double, ctypes.c_int, ctypes.c_void_p,
                   ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    _LIBS[key] = lib
    return lib


def _as_f64(x) -> np.ndarray:
    """Widen an fp16/bf16 (torch or numpy) matrix exactly to a C-contiguous fp64
    numpy array. Widening fp16 or bf16 to fp64 is exact."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu", torch.float64).contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def gemm_tn_reference(a, b, nthreads: int | None = None, lib: ctypes.CDLL | None = None):
    """ref, bound for C = A x B^T.

    a: [M, K], b: [N, K] (torch or numpy; fp16/bf16/fp32/fp64 values, read
    exactly as fp64). Returns two fp64 numpy arrays of shape [M, N]:
    ref[i, j] = sum_k a[i, k] * b[j, k] summed in increasing k, and
    bound[i, j] = sum_k |a[i, k] * b[j, k]|.
    "0. A Minimal Hopper Matmul", section "Block Tiling" (C = A x B^T, A (M, K),
    B (N, K)). ``lib`` selects another build of the C loop (the pinning tests
    pass deliberately wrong builds); by default the real one is used.
    """
    A = _as_f64(a)
    B = _as_f64(b)
    if A.ndim != 2 or B.ndim != 2 or A.shape[1] != B.shape[1]:
        raise ValueError(f"expected A [M,K] and B [N,K], got {A.shape} and {B.shape}")
    M, K = A.shape
    N = B.shape[0]
    ref = np.zeros((M, N), dtype=np.float64)
    bound = np.zeros((M, N), dtype=np.float64)
    if M and N:
        lib = lib or load_library()
        rc = lib.oracle_gemm_tn_f64(A.ctypes.data, B.ctypes.data, M, N, K,
                                    ref.ctypes.data, bound.ctypes.data,
                                    int(nthreads or host_threads()))
        if rc != 0:
            raise RuntimeError(f"oracle_gemm_tn_f64 failed with {rc}")
    return ref, bound


def gemm_nn_reference(a, b, nthreads: int | None = None):
    """ref, bound for C = A x B with B stored [K, N]: C[i][j] = sum_k a[i, k] *
    b[k, j]. The same plain product as gemm_tn_reference with B's rows and
    columns exchanged ("TileLang: a tile language one level below Triton",
    section "The first kernel: GEMM": B declared (K, N))."""
    B = _as_f64(b)
    return gemm_tn_reference(a, np.ascontiguousarray(B.T), nthreads=nthreads)


def attention_reference(q, k, v, causal: bool = True, scale: float | None = None, rows=None,
                        nthreads: int | None = None, lib: ctypes.CDLL | None = None):
    """out, bound of the attention forward pass ("TileLang: a tile language one
    level below Triton", section "FlashAttention: online softmax as tile code").

    q, k, v: [batch, seq, heads, dim] (torch or numpy, read exactly as fp64).
    For every batch b, head h and query position i in ``rows`` (all positions
    when None), with the visible keys j <= i (causal) or all j:
        s_j = scale * q[b, i, h] . k[b, j, h]      (scale default 1/sqrt(dim))
        p_j = exp(s_j - max s) / sum_j' exp(s_j' - max s)
        out[b, r, h, d] = sum_j p_j v[b, j, h, d]
        bound[b, r, h, d] = sum_j p_j |v[b, j, h, d]|
    Returns two fp64 arrays of shape [batch, len(rows), heads, dim]. ``lib``
    selects another build (the pinning tests pass deliberately wrong ones).
    """
    Q, K, V = _as_f64(q), _as_f64(k), _as_f64(v)
    if Q.ndim != 4 or Q.shape != K.shape or Q.shape != V.shape:
        raise ValueError(f"expected q, k, v of one shape [B, S, H, D], got {Q.shape}, {K.shape}, {V.shape}")
    B, S, H, D = Q.shape
    sc = float(scale) if scale is not None else (1.0 / np.sqrt(D) if D else 1.0)
    rows_arr = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
    R = S if rows_arr is None else rows_arr.size
    out = np.zeros((B, R, H, D), dtype=np.float64)
    bound = np.zeros((B, R, H, D), dtype=np.float64)
    if B and R and H and D:
        lib = lib or load_library()
        rc = lib.oracle_attention_f64(Q.ctypes.data, K.ctypes.data, V.ctypes.data, B, S, H, D, sc,
                                      1 if causal else 0,
                                      None if rows_arr is None else rows_arr.ctypes.data, R,
                                      out.ctypes.data, bound.ctypes.data, int(nthreads or host_threads()))
        if rc != 0:
            raise RuntimeError(f"oracle_attention_f64 failed with {rc}")
    return out, bound


#: activation codes of the fused epilogue (same numbering as the C ABI)
ACT_NONE, ACT_RELU, ACT_GELU = 0, 1, 2
#: largest slope of each activation (GELU's derivative peaks at ~1.129)
ACT_LIPSCHITZ = {ACT_NONE: 1.0, ACT_RELU: 1.0, ACT_GELU: 1.13}


def _activation(x: np.ndarray, act: int) -> np.ndarray:
    if act == ACT_NONE:
        return x
    if act == ACT_RELU:
        return np.maximum(x, 0.0)
    if act == ACT_GELU:  # x * Phi(x), Phi the standard normal CDF
        from scipy.special import erf
        return 0.5 * x * (1.0 + erf(x / np.sqrt(2.0)))
    raise ValueError(f"unknown activation {act}")


def fused_reference(a, b, alpha=1.0, beta=0.0, c_in=None, bias=None, activation=ACT_NONE, b_kn=False,
                    product=None):
    """D = act(alpha * (A x B^T) + beta * C_in + bias[j]) in fp64, with the
    magnitude bound of the pre-activation value:
        pre_bound[i][j] = |alpha| * sum_k |a_ik b_jk| + |beta * c_ij| + |bias_j|.
    The GEMM part is gemm_tn_reference (gemm_nn_reference with b_kn); the
    epilogue is the product's definition written out element by element
    (scale, add, add, activate). ``product``: the (ref, bound) pair that
    gemm_tn_reference returned for these a and b, when the caller has it
    already (a and b are then not read). Returns (d, pre_bound)."""
    if product is not None:
        ref, bound = product
    else:
        ref, bound = gemm_nn_reference(a, b) if b_kn else gemm_tn_reference(a, b)
    pre = float(alpha) * ref
    pre_bound = abs(float(alpha)) * bound
    if beta != 0.0 and c_in is not None:
        cin = _as_f64(c_in)
        pre = pre + float(beta) * cin
        pre_bound = pre_bound + np.abs(float(beta) * cin)
    if bias is not None:
        bb = _as_f64(bias).reshape(1, -1)
        pre = pre + bb
        pre_bound = pre_bound + np.abs(bb)
    return _activation(pre, activation), pre_bound


def fused_parity_report(d, d_ref: np.ndarray, pre_bound: np.ndarray, activation=ACT_NONE) -> "ParityReport":
    """The GEMM criterion carried through the epilogue: an error e in the
    pre-activation value moves the output by at most L*e (L the activation's
    largest slope), so |d - d_ref| <= L * (1e-2 * pre_bound + 1e-3)."""
    lip = ACT_LIPSCHITZ[activation]
    return parity_report(d, d_ref, lip * pre_bound + (lip - 1.0) * ALLOW_ABS / ALLOW_REL) if lip != 1.0 \
        else parity_report(d, d_ref, pre_bound)


def fused_e4m3_parity_report(codes, d_ref: np.ndarray, pre_bound: np.ndarray, activation=ACT_NONE) -> "ParityReport":
    """The fused criterion for an e4m3 output (``codes``: the stored bytes).
    Before its one rounding the kernel's fp32 value v is within
    E = L * (1e-2 * pre_bound + 1e-3) of d_ref (fused_parity_report), and
    clamping to [-448, 448] moves neither side apart. Rounding v to nearest
    e4m3 then moves it by at most half a step: 2^-4 * |v| for normal values
    (3 mantissa bits) and 2^-10 below 2^-6 (subnormal step 2^-9). So
        |decode(codes) - clamp(d_ref)| <= E + 2^-4 * (|clamp(d_ref)| + E) + 2^-10."""
    lip = ACT_LIPSCHITZ[activation]
    e = lip * (ALLOW_REL * pre_bound + ALLOW_ABS)
    target = np.clip(d_ref, -fp8.E4M3_MAX, fp8.E4M3_MAX)
    allow = e + 2.0 ** -4 * (np.abs(target) + e) + 2.0 ** -10
    return _report(fp8.e4m3_decode(codes), target, allow)


@dataclass
class ParityReport:
    ok: bool
    max_ratio: float          # max over elements of |c - ref| / allowance
    argmax: tuple             # (i, j) of that element
    n_bad: int                # elements over the allowance or not finite
    n_nonfinite: int
    max_abs_err: float

    def __str__(self) -> str:
        return (f"ok={self.ok} max_ratio={self.max_ratio:.3e} at {self.argmax} "
                f"bad={self.n_bad} nonfinite={self.n_nonfinite} max_abs_err={self.max_abs_err:.3e}")


def parity_report(c, ref: np.ndarray, bound: np.ndarray) -> ParityReport:
    """Apply the pass criterion |c - ref| <= 1e-2 * bound + 1e-3 element-wise.

    c is the result under test (any dtype, widened to fp64); NaN or Inf in c
    fails (the inputs of every workload are finite and in range).
    """
    return _report(_as_f64(c), ref, ALLOW_REL * bound + ALLOW_ABS)


def _report(C: np.ndarray, ref: np.ndarray, allow: np.ndarray) -> ParityReport:
    """|C - ref| <= allow element-wise; non-finite entries of C fail."""
    if C.shape != ref.shape:
        raise ValueError(f"shape mismatch {C.shape} vs {ref.shape}")
    if C.size == 0:
        return ParityReport(True, 0.0, (), 0, 0, 0.0)
    finite = np.isfinite(C)
    err = np.abs(C - ref)
    ratio = np.where(finite, err / allow, np.inf)
    flat = int(np.argmax(ratio))
    idx = tuple(int(v) for v in np.unravel_index(flat, ratio.shape))
    bad = ~(ratio <= 1.0)
    max_abs = float(np.max(np.where(finite, err, 0.0)))
    return ParityReport(bool(not bad.any()), float(ratio.flat[flat]), idx, int(bad.sum()),
                        int((~finite).sum()), max_abs)
