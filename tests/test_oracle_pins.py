"""Pins for the fp64 oracle of C = A x B^T, against things other than itself.

* exact rational arithmetic (brute force) on tiny and odd shapes: every fp16 or
  bf16 value is a dyadic rational, so the true sum is known exactly;
* closed forms: identity and permutation matrices reproduce A exactly; all-ones
  operands give K everywhere; small-integer operands give the exact integer
  product (checked with integer matrix multiplication, a library routine);
* the pass criterion itself: the oracle rounded to the output dtype passes with
  a wide margin, a single element moved by twice its allowance fails, NaN fails;
* planted mistakes: deliberately wrong builds of the C loop (a dropped term, an
  un-transposed B, a flipped sign, swapped output indices) each fail at least
  one of the pins above.

"0. A Minimal Hopper Matmul", section "Block Tiling": C = A x B^T with A (M, K)
and B (N, K). "Tiling a matmul", section "Where it breaks" (numerical order):
tiling changes only the order of additions, so any correct order lands within
the summation error bound of the exact value.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import build as oracle_build

U = 2.0 ** -53  # unit roundoff of fp64


def _rand(shape, dtype, seed, kind="uniform"):
    g = np.random.Generator(np.random.PCG64(seed))
    x = g.uniform(-1.0, 1.0, size=shape).astype(np.float32) if kind == "uniform" else \
        g.integers(-2, 3, size=shape).astype(np.float32)
    return torch.from_numpy(x).to(dtype)


def _exact(a: torch.Tensor, b: torch.Tensor):
    """Exact C = A x B^T and sum |a*b| with Fractions."""
    A = [[Fraction(float(v)) for v in row] for row in a.to(torch.float64).tolist()]
    B = [[Fraction(float(v)) for v in row] for row in b.to(torch.float64).tolist()]
    M, N, K = len(A), len(B), a.shape[1]
    ref = [[sum((A[i][k] * B[j][k] for k in range(K)), Fraction(0)) for j in range(N)] for i in range(M)]
    mag = [[sum((abs(A[i][k] * B[j][k]) for k in range(K)), Fraction(0)) for j in range(N)] for i in range(M)]
    return ref, mag


def _gamma(k: int) -> float:
    """gamma_k = k u / (1 - k u): the recursive-summation error factor."""
    return k * U / (1.0 - k * U)


TINY = [(1, 1, 1), (2, 3, 1), (3, 2, 7), (7, 16, 17), (16, 7, 33), (17, 33, 16),
        (33, 17, 65), (1, 65, 127), (65, 1, 129), (2, 2, 129)]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("mnk", TINY)
def test_bruteforce_exact_rational(mnk, dtype):
    m, n, k = mnk
    a = _rand((m, k), dtype, 11 + m + 3 * n + 7 * k)
    b = _rand((n, k), dtype, 13 + m + 5 * n + 11 * k)
    ref, bound = oracle.gemm_tn_reference(a, b)
    exact, mag = _exact(a, b)
    g = _gamma(k)
    for i in range(m):
        for j in range(n):
            # products are exact in fp64; only the K-term summation rounds
            assert abs(Fraction(ref[i, j]) - exact[i][j]) <= Fraction(g) * mag[i][j]
            assert abs(Fraction(bound[i, j]) - mag[i][j]) <= Fraction(g) * mag[i][j]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_identity_reproduces_a_exactly(dtype):
    m, k = 37, 53
    a = _rand((m, k), dtype, 5)
    eye = torch.eye(k, dtype=dtype)
    ref, bound = oracle.gemm_tn_reference(a, eye)
    np.testing.assert_array_equal(ref, a.double().numpy())
    np.testing.assert_array_equal(bound, a.double().abs().numpy())


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_permutation_reproduces_columns_exactly(dtype):
    m, k = 29, 41
    a = _rand((m, k), dtype, 6)
    perm = np.random.Generator(np.random.PCG64(7)).permutation(k)
    p = torch.zeros((k, k), dtype=dtype)
    p[torch.arange(k), torch.from_numpy(perm)] = 1  # row j of B selects column perm[j] of A
    ref, _ = oracle.gemm_tn_reference(a, p)
    np.testing.assert_array_equal(ref, a.double().numpy()[:, perm])


@pytest.mark.parametrize("mnk", [(1, 1, 1), (5, 3, 256), (3, 5, 4097), (16, 16, 8192)])
def test_all_ones_gives_k(mnk):
    m, n, k = mnk
    ref, bound = oracle.gemm_tn_reference(torch.ones((m, k), dtype=torch.float16),
                                          torch.ones((n, k), dtype=torch.float16))
    assert (ref == k).all() and (bound == k).all()


@pytest.mark.parametrize("mnk", [(24, 24, 24), (31, 17, 45), (17, 31, 64), (40, 40, 300)])
def test_small_integers_give_exact_integer_product(mnk):
    m, n, k = mnk
    a = _rand((m, k), torch.float16, 100 + m, kind="int")
    b = _rand((n, k), torch.float16, 200 + n, kind="int")
    ref, bound = oracle.gemm_tn_reference(a, b)
    ai = a.to(torch.int64).numpy()
    bi = b.to(torch.int64).numpy()
    np.testing.assert_array_equal(ref, (ai @ bi.T).astype(np.float64))
    np.testing.assert_array_equal(bound, (np.abs(ai) @ np.abs(bi).T).astype(np.float64))
    if m == n == k:  # the product of a non-symmetric pair differs from A x B
        assert not np.array_equal(ref, (ai @ bi).astype(np.float64))


def test_thread_count_does_not_change_results():
    a = _rand((67, 129), torch.bfloat16, 1)
    b = _rand((45, 129), torch.bfloat16, 2)
    r1, b1 = oracle.gemm_tn_reference(a, b, nthreads=1)
    r8, b8 = oracle.gemm_tn_reference(a, b, nthreads=8)
    np.testing.assert_array_equal(r1, r8)
    np.testing.assert_array_equal(b1, b8)


def test_empty_shapes():
    ref, bound = oracle.gemm_tn_reference(torch.zeros((0, 5)), torch.zeros((3, 5)))
    assert ref.shape == (0, 3)
    ref, bound = oracle.gemm_tn_reference(torch.zeros((4, 0)), torch.zeros((3, 0)))
    assert ref.shape == (4, 3) and (ref == 0).all() and (bound == 0).all()


# ---------------------------------------------------------------- pass criterion

@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_criterion_accepts_rounded_oracle(dtype):
    a = _rand((64, 300), dtype, 3)
    b = _rand((48, 300), dtype, 4)
    ref, bound = oracle.gemm_tn_reference(a, b)
    rounded = torch.from_numpy(ref).to(dtype)
    rep = oracle.parity_report(rounded, ref, bound)
    assert rep.ok and rep.max_ratio < 0.25, rep


def test_criterion_rejects_perturbation_and_nan():
    a = _rand((16, 64), torch.float32, 8)
    b = _rand((16, 64), torch.float32, 9)
    ref, bound = oracle.gemm_tn_reference(a, b)
    c = ref.copy()
    c[3, 5] += 2.0 * (oracle.ALLOW_REL * bound[3, 5] + oracle.ALLOW_ABS)
    rep = oracle.parity_report(c, ref, bound)
    assert not rep.ok and rep.argmax == (3, 5) and rep.n_bad == 1
    c = ref.copy()
    c[0, 0] = np.nan
    assert not oracle.parity_report(c, ref, bound).ok
    c = ref.copy()
    c[1, 1] = np.inf
    assert not oracle.parity_report(c, ref, bound).ok
    assert oracle.parity_report(ref, ref, bound).ok


# ---------------------------------------------------------------- planted mistakes

def _pins_failed(lib) -> list[str]:
    """Run a compact version of the pins above against a given build; return
    the names of those that fail."""
    failed = []
    # all-ones closed form
    ref, _ = oracle.gemm_tn_reference(torch.ones((6, 33)), torch.ones((6, 33)), lib=lib)
    if not (ref == 33).all():
        failed.append("all_ones")
    # integer product, square and non-symmetric
    a = _rand((24, 24), torch.float16, 41, kind="int")
    b = _rand((24, 24), torch.float16, 42, kind="int")
    ref, _ = oracle.gemm_tn_reference(a, b, lib=lib)
    if not np.array_equal(ref, (a.long().numpy() @ b.long().numpy().T).astype(np.float64)):
        failed.append("integer_square")
    # brute force, one odd square shape
    a = _rand((7, 7), torch.float16, 43)
    b = _rand((7, 7), torch.float16, 44)
    ref, _ = oracle.gemm_tn_reference(a, b, lib=lib)
    exact, mag = _exact(a, b)
    if any(abs(Fraction(ref[i, j]) - exact[i][j]) > Fraction(_gamma(7)) * mag[i][j]
           for i in range(7) for j in range(7)):
        failed.append("bruteforce")
    return failed


def test_real_build_passes_compact_pins():
    assert _pins_failed(oracle.load_library()) == []


@pytest.mark.parametrize("plant", [1, 2, 3, 4])
def test_each_planted_mistake_is_caught(plant, tmp_path):
    lib = oracle.load_library(plant=plant, out_dir=tmp_path)
    assert _pins_failed(lib), f"planted mistake {plant} went unnoticed"
    assert oracle_build.library_path(plant, tmp_path).exists()


@pytest.mark.parametrize("mnk", [(24, 24, 24), (31, 17, 45), (17, 40, 9)])
def test_nn_reference_is_a_times_b(mnk):
    """C = A x B with B [K, N]: small integers give the exact integer product
    A @ B (and not A @ B^T on square shapes)."""
    m, n, k = mnk
    a = _rand((m, k), torch.float16, 300 + m, kind="int")
    b = _rand((k, n), torch.float16, 400 + n, kind="int")
    ref, bound = oracle.gemm_nn_reference(a, b)
    ai, bi = a.to(torch.int64).numpy(), b.to(torch.int64).numpy()
    np.testing.assert_array_equal(ref, (ai @ bi).astype(np.float64))
    np.testing.assert_array_equal(bound, (np.abs(ai) @ np.abs(bi)).astype(np.float64))
    if m == n == k:
        assert not np.array_equal(ref, (ai @ bi.T).astype(np.float64))


# ---------------------------------------------------------------- fused epilogue

def test_fused_reference_closed_forms():
    """Scale, add and activation pinned to values fixed by arithmetic."""
    a = _rand((8, 16), torch.float16, 500, kind="int")
    b = _rand((6, 16), torch.float16, 501, kind="int")
    exact = (a.long() @ b.long().T).double().numpy()
    # alpha scales exactly (powers of two), no epilogue terms otherwise
    d, pb = oracle.fused_reference(a, b, alpha=2.0)
    np.testing.assert_array_equal(d, 2.0 * exact)
    # alpha 0, beta 1: D = C_in + bias, exactly
    c_in = torch.arange(48, dtype=torch.float32).reshape(8, 6) - 20
    bias = torch.tensor([0.5, -1.0, 2.0, 0.0, -0.25, 4.0])
    d, pb = oracle.fused_reference(a, b, alpha=0.0, beta=1.0, c_in=c_in, bias=bias)
    np.testing.assert_array_equal(d, c_in.double().numpy() + bias.double().numpy()[None, :])
    # relu keeps the non-negative part
    d, _ = oracle.fused_reference(a, b, activation=oracle.ACT_RELU)
    np.testing.assert_array_equal(d, np.maximum(exact, 0.0))


def test_fused_reference_all_terms_and_bound():
    """Every term at once with exactly representable scales: D = 2 A B^T +
    0.5 C_in + bias and pre_bound = 2 sum|a b| + |0.5 C_in| + |bias|, both
    exact (integer operands, dyadic scales); B given [K, N] (b_kn) gives the
    same D."""
    a = _rand((8, 16), torch.float16, 502, kind="int")
    b = _rand((6, 16), torch.float16, 503, kind="int")
    exact = (a.long() @ b.long().T).double().numpy()
    abs_sum = (a.long().abs() @ b.long().abs().T).double().numpy()
    c_in = (torch.arange(48, dtype=torch.float32).reshape(8, 6) - 20) / 4
    bias = torch.tensor([0.5, -1.0, 2.0, 0.0, -0.25, 4.0])
    d, pb = oracle.fused_reference(a, b, alpha=2.0, beta=0.5, c_in=c_in, bias=bias)
    cin, bb = c_in.double().numpy(), bias.double().numpy()[None, :]
    np.testing.assert_array_equal(d, 2.0 * exact + 0.5 * cin + bb)
    np.testing.assert_array_equal(pb, 2.0 * abs_sum + np.abs(0.5 * cin) + np.abs(bb))
    d_kn, pb_kn = oracle.fused_reference(a, b.T.contiguous(), alpha=2.0, beta=0.5, c_in=c_in, bias=bias, b_kn=True)
    np.testing.assert_array_equal(d_kn, d)
    np.testing.assert_array_equal(pb_kn, pb)
    # a negative alpha flips D but not the bound
    d_neg, pb_neg = oracle.fused_reference(a, b, alpha=-2.0)
    np.testing.assert_array_equal(d_neg, -2.0 * exact)
    np.testing.assert_array_equal(pb_neg, 2.0 * abs_sum)


def test_gelu_reference_properties():
    """GELU(x) = x * Phi(x): GELU(0) = 0, GELU(x) - GELU(-x) = x, Phi(1) and
    Phi(2) from the normal CDF's tabulated values, and GELU(x) ~ x for large x."""
    x = np.array([0.0, 1.0, 2.0, -1.0, -2.0, 8.0, -8.0])
    g = oracle._activation(x, oracle.ACT_GELU)
    assert g[0] == 0.0
    np.testing.assert_allclose(g[1] - g[3], 1.0, rtol=0, atol=1e-15)
    np.testing.assert_allclose(g[2] - g[4], 2.0, rtol=0, atol=1e-15)
    np.testing.assert_allclose(g[1], 0.8413447460685429, rtol=1e-15)      # Phi(1)
    np.testing.assert_allclose(g[2] / 2.0, 0.9772498680518208, rtol=1e-15)  # Phi(2)
    assert abs(g[5] - 8.0) < 1e-13 and abs(g[6]) < 1e-13


def test_fused_tolerance_scales_with_the_activation_slope():
    ref = np.zeros((2, 2))
    pb = np.ones((2, 2))
    d = ref + 1.05 * (oracle.ALLOW_REL * 1.0 + oracle.ALLOW_ABS)   # 5% over the plain allowance
    assert not oracle.fused_parity_report(d, ref, pb, oracle.ACT_NONE).ok
    assert oracle.fused_parity_report(d, ref, pb, oracle.ACT_GELU).ok    # GELU allows 13% more


# ------------------------------------------------------------ fp8 e4m3 output

from oracle import fp8  # noqa: E402


def test_e4m3_decode_landmarks():
    """Codes whose values the format's definition fixes (sign, 4 exponent
    bits with bias 7, 3 mantissa bits; e = 15 with m = 7 is NaN)."""
    landmarks = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
                 0x39: 1.125, 0x40: 2.0, 0x77: 240.0, 0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0}
    for code, value in landmarks.items():
        assert fp8.e4m3_decode(np.array([code]))[0] == value, hex(code)
    assert np.isnan(fp8.e4m3_decode(np.array([0x7F, 0xFF]))).all()
    assert np.signbit(fp8.e4m3_decode(np.array([0x80]))[0])
    vals = fp8.e4m3_decode(np.arange(256))
    assert np.isnan(vals).sum() == 2
    assert len(np.unique(vals[~np.isnan(vals)])) == 253          # +0 and -0 compare equal


def test_e4m3_decode_matches_torch_for_every_code():
    """torch's float8_e4m3fn widening (a library routine) of all 256 codes."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    want = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = fp8.e4m3_decode(codes.numpy())
    assert np.array_equal(np.isnan(got), np.isnan(want))
    fin = ~np.isnan(want)
    assert np.array_equal(got[fin], want[fin])
    assert np.array_equal(np.signbit(got[fin]), np.signbit(want[fin]))


def test_e4m3_round_trip_and_ties_to_even():
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    assert np.array_equal(fp8.e4m3_encode(fp8.e4m3_decode(finite)), finite.astype(np.uint8))
    pos = fp8.e4m3_decode(np.arange(127))
    mid = (pos[:-1] + pos[1:]) / 2                                 # exact in fp64
    got = fp8.e4m3_encode(mid).astype(np.int64)
    lower = np.arange(126)
    assert np.array_equal(got, np.where(lower % 2 == 0, lower, lower + 1))
    assert fp8.e4m3_encode(np.array([1.0 + 1 / 16]))[0] == 0x38   # tie: 1.0 (m = 000), not 1.125
    assert fp8.e4m3_encode(np.array([1.0 + 3 / 16]))[0] == 0x3A   # tie: 1.25 (m = 010), not 1.125
    # just off a midpoint, the nearer neighbour wins whatever its parity
    assert fp8.e4m3_encode(np.array([1.0 + 1 / 16 + 1e-9]))[0] == 0x39


def test_e4m3_saturation_and_special_values():
    enc = fp8.e4m3_encode(np.array([448.0, 463.9, 464.0, 1e6, np.inf, -1e6, -np.inf, np.nan, -0.0, -1e-9, 2.0 ** -10]))
    assert enc.tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F, 0x80, 0x80, 0x00]
    # 3 * 2^-10 lies halfway between 2^-9 (0x01) and 2^-8 (0x02): the even code
    assert fp8.e4m3_encode(np.array([3 * 2.0 ** -10]))[0] == 0x02


def test_e4m3_encode_matches_torch_in_range():
    """torch's float8_e4m3fn rounding (a library routine) of fp32 values in the
    finite range, where it and the saturating encoder agree by definition."""
    g = np.random.Generator(np.random.PCG64(88))
    x = np.concatenate([g.uniform(-448, 448, 20000), g.standard_normal(20000) * 4,
                        g.uniform(-2.0 ** -5, 2.0 ** -5, 20000)]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.e4m3_encode(x.astype(np.float64)), want)


def test_e4m3_parity_allowance():
    """The e4m3 criterion accepts the oracle's own rounding of d (and of the
    saturated values) and rejects a code one step off where the step is larger
    than the fp32 allowance."""
    g = np.random.Generator(np.random.PCG64(5))
    d = np.concatenate([g.uniform(-600, 600, 4000), g.uniform(-1, 1, 4000)]).reshape(80, 100)
    pre_bound = np.abs(d)
    rep = oracle.fused_e4m3_parity_report(fp8.e4m3_encode(d), d, pre_bound)
    assert rep.ok, rep
    codes = fp8.e4m3_encode(d)
    bumped = codes.copy()
    big = int(np.argmax(np.where(np.abs(d) < 300, np.abs(d), 0)))      # code <= 0x7A: +2 stays finite
    bumped.flat[big] = codes.flat[big] + 2                              # two steps: over 2^-3 relative
    assert np.isfinite(fp8.e4m3_decode(bumped.flat[big:big + 1]))[0]
    assert not oracle.fused_e4m3_parity_report(bumped, d, np.zeros_like(d)).ok
    nan = codes.copy()
    nan.flat[7] = 0x7F
    assert not oracle.fused_e4m3_parity_report(nan, d, pre_bound).ok
