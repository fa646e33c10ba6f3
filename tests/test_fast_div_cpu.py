"""The tile scheduler divides by invariant integers with a multiply-high, an
add and a shift (Granlund and Montgomery, "Division by invariant integers
using multiplication", 1994, the round-up method; the kernels' FastDiv and the
host's make_fast_div). This checks the method itself against exact integer
division by brute force over the divisors and dividends the scheduler can see
(1 <= d < 2^31, 0 <= n < 2^31), including the powers of two and their
neighbours. The device side is covered by the GPU parity tests, whose shapes
run every raster group layout through it."""
import random


def make_fast_div(d):
    shift = 0
    while (1 << shift) < d:
        shift += 1
    mul = ((1 << 32) * ((1 << shift) - d)) // d + 1
    return mul, shift


def fast_div(n, mul, shift):
    t = (n * mul) >> 32          # umulhi
    s = t + n
    assert s < (1 << 32), "the 32-bit sum must not wrap"
    return s >> shift


def test_multiplier_fits_32_bits_and_division_is_exact():
    rng = random.Random(20261202)
    divisors = list(range(1, 600))
    divisors += [(1 << k) + o for k in range(1, 31) for o in (-1, 0, 1) if 0 < (1 << k) + o < (1 << 31)]
    divisors += [(1 << 31) - 1] + [rng.randrange(1, 1 << 31) for _ in range(400)]
    for d in divisors:
        mul, shift = make_fast_div(d)
        assert 0 < mul < (1 << 32)
        dividends = list(range(0, 300)) + [d - 1, d, d + 1, 2 * d - 1, 2 * d, 3 * d + 1]
        dividends += [(1 << 31) - 1, (1 << 31) - 2] + [rng.randrange(0, 1 << 31) for _ in range(40)]
        for n in dividends:
            if 0 <= n < (1 << 31):
                assert fast_div(n, mul, shift) == n // d, (n, d)


def test_group_coordinates_match_plain_division():
    """The raster's tile -> (row, column) with the constants the host computes
    (tiles per group, rows per group, the last group's rows) equals the plain
    definition for every tile of assorted grids and group sizes."""
    for num_m, num_n in [(1, 1), (1, 7), (7, 1), (5, 9), (32, 32), (13, 40), (33, 3)]:
        for group in [1, 2, 3, 4, 8, 16, 64]:
            g_m = min(group, num_m)
            last_first = (num_m - 1) // g_m * g_m
            dg, dr, dl = make_fast_div(g_m * num_n), make_fast_div(g_m), make_fast_div(num_m - last_first)
            for tile in range(num_m * num_n):
                g = fast_div(tile, *dg)
                first = g * g_m
                in_group = tile - g * g_m * num_n
                full = first + g_m <= num_m
                rows = g_m if full else num_m - first
                col = fast_div(in_group, *(dr if full else dl))
                tm, tn = first + (in_group - col * rows), col
                # the plain definition
                per_group = g_m * num_n
                g0 = tile // per_group
                rows0 = min(num_m - g0 * g_m, g_m)
                in0 = tile - g0 * per_group
                assert (tm, tn) == (g0 * g_m + in0 % rows0, in0 // rows0)
