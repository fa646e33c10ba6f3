"""ctypes binding of ``libgemm_tn.so`` (the C ABI in ``include/gemm_tn.h`` and
``include/flash_attn.h``).

Argument marshalling only: every step of the product runs in the library's
CUDA kernels. The functions keep the C names and signatures; ``mm_tn`` and
``mm_tn_host`` are conveniences that take torch tensors, pass their pointers,
strides and the current CUDA stream, and raise ``GemmTnError`` on a non-zero
status. There is no fallback: if the library is missing or cannot be loaded,
every call raises.
"""
from __future__ import annotations

import ctypes
import threading
from pathlib import Path

PKG = Path(__file__).resolve().parent
LIBRARY_PATH = PKG / "libgemm_tn.so"

GEMM_TN_F16 = 0
GEMM_TN_BF16 = 1

GEMM_TN_OK = 0
GEMM_TN_ERR_INVALID_VALUE = 1
GEMM_TN_ERR_UNSUPPORTED_DTYPE = 2
GEMM_TN_ERR_MISALIGNED = 3
GEMM_TN_ERR_UNSUPPORTED_DEVICE = 4
GEMM_TN_ERR_CUDA = 5
GEMM_TN_ERR_TIMEOUT = 6

GEMM_TN_ACT_NONE, GEMM_TN_ACT_RELU, GEMM_TN_ACT_GELU = 0, 1, 2
GEMM_TN_OUT_INPUT, GEMM_TN_OUT_F32, GEMM_TN_OUT_E4M3 = 0, 1, 2


class GemmTnEpilogue(ctypes.Structure):
    """struct gemm_tn_epilogue of include/gemm_tn.h."""
    _fields_ = [("alpha", ctypes.c_float), ("beta", ctypes.c_float), ("bias", ctypes.c_void_p),
                ("activation", ctypes.c_int), ("out_dtype", ctypes.c_int)]


_lock = threading.Lock()
_lib: ctypes.CDLL | None = None

_i64 = ctypes.c_int64
_int = ctypes.c_int
_ptr = ctypes.c_void_p

_SIGNATURES = {
    "gemm_tn": (_int, [_int, _i64, _i64, _i64, _ptr, _ptr, _ptr, _ptr]),
    "gemm_tn_ex": (_int, [_int, _i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, _ptr, _ptr]),
    "gemm_tn_fused": (_int, [_int, _i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64,
                             ctypes.POINTER(GemmTnEpilogue), _ptr, _ptr]),
    "gemm_nn": (_int, [_int, _i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, _ptr, _ptr]),
    "gemm_tn_ex_noalloc": (_int, [_int, _i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, _ptr, _ptr]),
    "gemm_tn_host": (_int, [_int, _i64, _i64, _i64, _ptr, _ptr, _ptr, _ptr]),
    "gemm_tn_select_config": (_int, [_int, _i64, _i64, _i64]),
    "gemm_tn_select_splits": (_int, [_int, _i64, _i64, _i64]),
    "gemm_tn_last_config": (_int, []),
    "gemm_tn_workspace_pool": (_ptr, []),
    "gemm_tn_trim_workspace": (_int, []),
    "gemm_tn_multicast_allowed": (_int, [_ptr, _ptr]),
    "gemm_tn_num_configs": (_int, []),
    "gemm_tn_config_name": (ctypes.c_char_p, [_int]),
    "gemm_tn_status_string": (ctypes.c_char_p, [_int]),
    "gemm_tn_last_cuda_error": (_int, []),
    "gemm_tn_last_error_message": (ctypes.c_char_p, []),
    "gemm_tn_version": (_int, []),
    "gemm_tn_launch_count": (ctypes.c_uint64, []),
    "flash_attn_fwd": (_int, [_int, _i64, _i64, _i64, _i64, _ptr, _ptr, _ptr, _ptr, ctypes.c_float, _int, _ptr,
                              _ptr]),
}


class GemmTnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        lib = library()
        msg = lib.gemm_tn_last_error_message().decode()
        super().__init__(f"{where}: {lib.gemm_tn_status_string(status).decode()} ({msg})")


def library() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not LIBRARY_PATH.exists():
                raise RuntimeError(
                    f"{LIBRARY_PATH} is missing: build it with `python -m dense_tiled_gemm_03_gb300.build` "
                    "(there is no CPU fallback)")
            lib = ctypes.CDLL(str(LIBRARY_PATH))
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


# ---------------------------------------------------------------- C-named calls

def gemm_tn(dtype, m, n, k, a, b, c, stream=None) -> int:
    return library().gemm_tn(dtype, m, n, k, a, b, c, stream)


def gemm_tn_ex(dtype, m, n, k, a, lda, b, ldb, c, ldc, d_status=None, stream=None) -> int:
    return library().gemm_tn_ex(dtype, m, n, k, a, lda, b, ldb, c, ldc, d_status, stream)


def gemm_tn_fused(dtype, m, n, k, a, lda, b, ldb, c, ldc, epilogue, d_status=None, stream=None) -> int:
    """D = act(alpha * A x B^T + beta * C + bias) over C (epilogue: GemmTnEpilogue)."""
    ep = ctypes.byref(epilogue) if epilogue is not None else None
    return library().gemm_tn_fused(dtype, m, n, k, a, lda, b, ldb, c, ldc, ep, d_status, stream)


def gemm_nn(dtype, m, n, k, a, lda, b, ldb, c, ldc, d_status=None, stream=None) -> int:
    """C = A x B with B stored [K, N] (N contiguous)."""
    return library().gemm_nn(dtype, m, n, k, a, lda, b, ldb, c, ldc, d_status, stream)


def gemm_tn_ex_noalloc(dtype, m, n, k, a, lda, b, ldb, c, ldc, d_status=None, stream=None) -> int:
    """gemm_tn_ex that allocates no device memory (see include/gemm_tn.h)."""
    return library().gemm_tn_ex_noalloc(dtype, m, n, k, a, lda, b, ldb, c, ldc, d_status, stream)


#: bytes of the static scratch gemm_tn_ex_noalloc may use (GEMM_TN_NOALLOC_SCRATCH_BYTES)
GEMM_TN_NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


def gemm_tn_host(dtype, m, n, k, a_host, b_host, c_host, stream=None) -> int:
    return library().gemm_tn_host(dtype, m, n, k, a_host, b_host, c_host, stream)


def flash_attn_fwd(dtype, batch, seq, heads, head_dim, q, k, v, o, softmax_scale=0.0, causal=1, d_status=None,
                   stream=None) -> int:
    """O = softmax(scale * Q K^T, mask) V on [batch, seq, heads, head_dim] arrays
    (see include/flash_attn.h)."""
    return library().flash_attn_fwd(dtype, batch, seq, heads, head_dim, q, k, v, o, float(softmax_scale),
                                    1 if causal else 0, d_status, stream)


def gemm_tn_select_config(dtype, m, n, k) -> int:
    return library().gemm_tn_select_config(dtype, m, n, k)


def gemm_tn_select_splits(dtype, m, n, k) -> int:
    return library().gemm_tn_select_splits(dtype, m, n, k)


def gemm_tn_last_config() -> int:
    """Configuration the calling thread's last GEMM call launched (-1: none)."""
    return library().gemm_tn_last_config()


def gemm_tn_workspace_pool() -> int | None:
    """Handle (cudaMemPool_t) of the library's workspace pool on the current
    device, or None without a usable device."""
    return library().gemm_tn_workspace_pool()


def gemm_tn_trim_workspace() -> int:
    """Return the workspace pool's unused memory on the current device."""
    return library().gemm_tn_trim_workspace()


def gemm_tn_multicast_allowed(a, b) -> int:
    """1 when both pointers are device memory of the current device (the
    multicast configuration may read them), else 0."""
    return library().gemm_tn_multicast_allowed(a, b)


def gemm_tn_num_configs() -> int:
    return library().gemm_tn_num_configs()


def gemm_tn_config_name(config: int) -> str:
    return library().gemm_tn_config_name(config).decode()


def gemm_tn_status_string(status: int) -> str:
    return library().gemm_tn_status_string(status).decode()


def gemm_tn_last_cuda_error() -> int:
    return library().gemm_tn_last_cuda_error()


def gemm_tn_last_error_message() -> str:
    return library().gemm_tn_last_error_message().decode()


def gemm_tn_version() -> int:
    return library().gemm_tn_version()


def gemm_tn_launch_count() -> int:
    """Kernels the library has launched in this process so far."""
    return library().gemm_tn_launch_count()


# ---------------------------------------------------------------- torch helpers

def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return GEMM_TN_F16
    if t.dtype == torch.bfloat16:
        return GEMM_TN_BF16
    raise TypeError(f"unsupported dtype {t.dtype}: expected float16 or bfloat16")


class _on_device:
    """Make `device` current for the call (the library launches on the
    current device), switching only when it is not current already; yields
    the raw handle of the device's current torch stream. Cheaper than
    torch.cuda.device() + torch.cuda.current_stream() on the common path."""

    __slots__ = ("index", "prev")

    def __init__(self, device):
        self.index = device.index if device.index is not None else 0
        self.prev = None

    def __enter__(self) -> int:
        import torch
        cur = torch._C._cuda_getDevice()
        if cur != self.index:
            self.prev = cur
            torch._C._cuda_setDevice(self.index)
        return torch._C._cuda_getCurrentRawStream(self.index)

    def __exit__(self, *exc):
        if self.prev is not None:
            import torch
            torch._C._cuda_setDevice(self.prev)
        return False


def _status_ptr(status, device):
    """Device pointer of the optional watchdog status word: a one-element (or
    longer) contiguous int32 tensor on the call's device, or None. The kernels
    write an int through it, so any other tensor is refused here."""
    import torch
    if status is None:
        return None
    if not isinstance(status, torch.Tensor) or status.device != device or status.dtype != torch.int32 or \
            status.numel() < 1 or not status.is_contiguous():
        raise ValueError(f"status must be a contiguous int32 tensor of at least one element on {device}")
    return status.data_ptr()


def _row_pitch(t, cols: int) -> int:
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
        raise ValueError("operands must be 2-D with unit stride along the last dimension")
    return t.stride(0) if t.shape[0] > 1 else max(cols, 1)


def mm_tn(a, b, out=None, status=None):
    """C = A x B^T on the GPU through gemm_tn_ex. a: [M, K], b: [N, K] CUDA
    tensors of the same fp16/bf16 dtype with unit stride along K; out: optional
    [M, N] tensor of that dtype with unit stride along N; status: optional
    one-element int32 CUDA tensor for the device watchdog. Runs on the
    current CUDA stream of a's device."""
    import torch
    if a.device.type != "cuda" or b.device != a.device:
        raise ValueError("a and b must be CUDA tensors on one device")
    if a.dtype != b.dtype:
        raise TypeError("a and b must have the same dtype")
    m, k = a.shape
    n, kb = b.shape
    if kb != k:
        raise ValueError(f"inner dimensions differ: {tuple(a.shape)} x {tuple(b.shape)}^T")
    if out is None:
        out = torch.empty((m, n), dtype=a.dtype, device=a.device)
    elif out.shape != (m, n) or out.dtype != a.dtype or out.device != a.device:
        raise ValueError("out must be [M, N] with the dtype and device of a")
    lda, ldb, ldc = _row_pitch(a, k), _row_pitch(b, k), _row_pitch(out, n)
    d_status = _status_ptr(status, a.device)
    with _on_device(a.device) as stream:
        rc = library().gemm_tn_ex(_dtype_code(a), m, n, k, a.data_ptr(), lda, b.data_ptr(), ldb, out.data_ptr(),
                                  ldc, d_status, stream)
    if rc != GEMM_TN_OK:
        raise GemmTnError(rc, "gemm_tn_ex")
    return out


_ACTIVATIONS = {"none": GEMM_TN_ACT_NONE, "relu": GEMM_TN_ACT_RELU, "gelu": GEMM_TN_ACT_GELU}


def mm_tn_fused(a, b, out=None, alpha=1.0, beta=0.0, bias=None, activation="none", out_fp32=False, status=None,
                out_dtype=None):
    """act(alpha * A x B^T + beta * out + bias) through gemm_tn_fused. a: [M, K],
    b: [N, K] CUDA fp16/bf16; bias: optional fp32 CUDA [N]; out: [M, N] of
    out_dtype (its contents are read when beta != 0). out_dtype: None for a's
    dtype, torch.float32 (or out_fp32=True), or torch.float8_e4m3fn for the
    saturating fp8 output (alpha then carries the quantisation scale)."""
    import torch
    if a.device.type != "cuda" or b.device != a.device:
        raise ValueError("a and b must be CUDA tensors on one device")
    if a.dtype != b.dtype:
        raise TypeError("a and b must have the same dtype")
    m, k = a.shape
    n, kb = b.shape
    if kb != k:
        raise ValueError(f"inner dimensions differ: {tuple(a.shape)} x {tuple(b.shape)}^T")
    if out_dtype is None:
        out_dtype = torch.float32 if out_fp32 else a.dtype
    elif out_fp32 and out_dtype != torch.float32:
        raise ValueError("out_fp32 contradicts out_dtype")
    codes = {a.dtype: GEMM_TN_OUT_INPUT, torch.float32: GEMM_TN_OUT_F32, torch.float8_e4m3fn: GEMM_TN_OUT_E4M3}
    if out_dtype not in codes:
        raise TypeError(f"unsupported output dtype {out_dtype}")
    if out is None:
        out = torch.zeros((m, n), dtype=out_dtype, device=a.device)
    elif out.shape != (m, n) or out.dtype != out_dtype or out.device != a.device:
        raise ValueError(f"out must be [M, N] of {out_dtype} on a's device")
    if bias is not None and (bias.dtype != torch.float32 or bias.shape != (n,) or bias.device != a.device or
                             not bias.is_contiguous()):
        raise ValueError("bias must be a contiguous CUDA fp32 [N] tensor on a's device")
    ep = GemmTnEpilogue(float(alpha), float(beta), bias.data_ptr() if bias is not None else None,
                        _ACTIVATIONS[activation], codes[out_dtype])
    lda, ldb, ldc = _row_pitch(a, k), _row_pitch(b, k), _row_pitch(out, n)
    d_status = _status_ptr(status, a.device)
    with _on_device(a.device) as stream:
        rc = gemm_tn_fused(_dtype_code(a), m, n, k, a.data_ptr(), lda, b.data_ptr(), ldb, out.data_ptr(), ldc, ep,
                           d_status, stream)
    if rc != GEMM_TN_OK:
        raise GemmTnError(rc, "gemm_tn_fused")
    return out


def mm_nn(a, b, out=None, status=None):
    """C = A x B on the GPU through gemm_nn. a: [M, K], b: [K, N] CUDA tensors
    of the same fp16/bf16 dtype with unit stride along their last dimension."""
    import torch
    if a.device.type != "cuda" or b.device != a.device:
        raise ValueError("a and b must be CUDA tensors on one device")
    if a.dtype != b.dtype:
        raise TypeError("a and b must have the same dtype")
    m, k = a.shape
    kb, n = b.shape
    if kb != k:
        raise ValueError(f"inner dimensions differ: {tuple(a.shape)} x {tuple(b.shape)}")
    if out is None:
        out = torch.empty((m, n), dtype=a.dtype, device=a.device)
    elif out.shape != (m, n) or out.dtype != a.dtype or out.device != a.device:
        raise ValueError("out must be [M, N] with the dtype and device of a")
    lda, ldb, ldc = _row_pitch(a, k), _row_pitch(b, n), _row_pitch(out, n)
    d_status = _status_ptr(status, a.device)
    with _on_device(a.device) as stream:
        rc = gemm_nn(_dtype_code(a), m, n, k, a.data_ptr(), lda, b.data_ptr(), ldb, out.data_ptr(), ldc,
                     d_status, stream)
    if rc != GEMM_TN_OK:
        raise GemmTnError(rc, "gemm_nn")
    return out


def mm_tn_host(a, b, out=None, device=None):
    """C = A x B^T through gemm_tn_host: a, b, out are contiguous CPU tensors
    (pinned or pageable); the call copies to the GPU, computes, copies back and
    waits."""
    import torch
    if a.device.type != "cpu" or b.device.type != "cpu":
        raise ValueError("mm_tn_host takes CPU tensors")
    if a.dim() != 2 or b.dim() != 2:
        raise ValueError("a and b must be 2-D")
    if a.dtype != b.dtype:
        raise TypeError("a and b must have the same dtype")
    dtype = _dtype_code(a)
    a = a.contiguous()
    b = b.contiguous()
    m, k = a.shape
    n, kb = b.shape
    if kb != k:
        raise ValueError(f"inner dimensions differ: {tuple(a.shape)} x {tuple(b.shape)}^T")
    if out is None:
        out = torch.empty((m, n), dtype=a.dtype)
    elif out.device.type != "cpu" or out.shape != (m, n) or out.dtype != a.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous CPU [M, N] tensor with the dtype of a")
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    stream = torch.cuda.current_stream(dev).cuda_stream
    with torch.cuda.device(dev):
        rc = gemm_tn_host(dtype, m, n, k, a.data_ptr(), b.data_ptr(), out.data_ptr(), stream)
    if rc != GEMM_TN_OK:
        raise GemmTnError(rc, "gemm_tn_host")
    return out


def flash_attn(q, k, v, causal=True, scale=None, out=None, status=None):
    """Attention forward pass through flash_attn_fwd. q, k, v: contiguous CUDA
    tensors [batch, seq, heads, head_dim] of one fp16/bf16 dtype (head_dim 64 or
    128, 16-byte aligned); scale: the factor on Q.K (None: 1/sqrt(head_dim));
    out: optional contiguous tensor of the same shape and dtype; status:
    optional one-element int32 CUDA tensor for the device watchdog. Runs on the
    current CUDA stream of q's device."""
    import torch
    if q.device.type != "cuda" or k.device != q.device or v.device != q.device:
        raise ValueError("q, k and v must be CUDA tensors on one device")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must have the same dtype")
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k and v must have one shape [batch, seq, heads, head_dim]")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k and v must be contiguous")
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or out.device != q.device or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor with q's shape, dtype and device")
    b, s, h, d = q.shape
    d_status = _status_ptr(status, q.device)
    with _on_device(q.device) as stream:
        rc = flash_attn_fwd(_dtype_code(q), b, s, h, d, q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                            0.0 if scale is None else float(scale), causal, d_status, stream)
    if rc != GEMM_TN_OK:
        raise GemmTnError(rc, "flash_attn_fwd")
    return out
