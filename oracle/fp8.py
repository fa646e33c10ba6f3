"""fp8 e4m3 encode / decode for the oracle -- TEST INFRASTRUCTURE ONLY.

The fused GEMM epilogue can store its result as fp8 e4m3, the quantised form
that "TileLang: a tile language one level below Triton" (exercise 4 of its
exercises) argues should be written by the operator producing the values rather
than by a separate bandwidth-bound pass. The format itself is not on that page;
these functions write out its definition (the "E4M3" fp8 format, OCP 8-bit
floating point specification):

  * bit 7 sign, bits 6-3 exponent e (bias 7), bits 2-0 mantissa m;
  * e = 0: subnormal, value m * 2^-9;
  * 0 < e: value (1 + m/8) * 2^(e-7), except e = 15 with m = 7, which is NaN
    (the format has no infinities); the largest finite value is 448 (0x7E).

Encoding rounds to the nearest representable value, ties to the even code
(mantissa lsb 0), and saturates: magnitudes of 448 and above (infinities too)
give +-448; NaN gives 0x7F. Negative values keep their sign bit, so a negative
value that rounds to zero encodes -0 (0x80).

Pinned by ``tests/test_oracle_pins.py``: landmark codes of the definition,
torch's own float8_e4m3fn conversion of every code and of random in-range
values, round trips of every finite code, and the ties-to-even rule at every
midpoint.
"""
from __future__ import annotations

import numpy as np

__all__ = ["E4M3_MAX", "e4m3_decode", "e4m3_encode", "e4m3_round"]

#: largest finite e4m3 magnitude, (1 + 6/8) * 2^8
E4M3_MAX = 448.0


def _decode_magnitude(code: np.ndarray) -> np.ndarray:
    """Value of the 7 magnitude bits (sign bit ignored)."""
    e = (code >> 3) & 0xF
    m = (code & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = m * 2.0 ** -9
    val = np.where(e == 0, sub, normal)
    return np.where((e == 15) & ((code & 0x7) == 7), np.nan, val)


def e4m3_decode(codes) -> np.ndarray:
    """e4m3 bytes (any integer array, or a torch uint8 / float8 tensor) to
    their exact fp64 values."""
    try:
        import torch
        if isinstance(codes, torch.Tensor):
            codes = codes.detach().cpu().contiguous().view(torch.uint8).numpy()
    except ImportError:  # pragma: no cover
        pass
    c = np.asarray(codes).astype(np.int64) & 0xFF
    mag = _decode_magnitude(c & 0x7F)
    return np.where((c & 0x80) != 0, -mag, mag)


# the 127 non-negative finite values, codes 0x00 ... 0x7E, in increasing order
_POS_VALUES = _decode_magnitude(np.arange(127, dtype=np.int64))


def e4m3_encode(x) -> np.ndarray:
    """fp64 values to e4m3 bytes (uint8): round to nearest, ties to the even
    code, saturating at +-448, NaN -> 0x7F."""
    v = np.asarray(x, dtype=np.float64)
    a = np.abs(v)
    nan = np.isnan(v)
    a_fin = np.where(nan, 0.0, np.minimum(a, E4M3_MAX))
    hi = np.searchsorted(_POS_VALUES, a_fin, side="left")     # _POS_VALUES[hi] >= a
    hi = np.minimum(hi, 126)
    lo = np.maximum(hi - 1, 0)
    d_lo = a_fin - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - a_fin
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    mag = np.where(take_hi, hi, lo)
    mag = np.where(a_fin == _POS_VALUES[hi], hi, mag)      # exact hits (and zero)
    code = mag | np.where(np.signbit(v), 0x80, 0)
    code = np.where(nan, 0x7F, code)
    return code.astype(np.uint8)


def e4m3_round(x) -> np.ndarray:
    """x rounded to the e4m3 value it encodes to (fp64)."""
    return e4m3_decode(e4m3_encode(x))
