"""The decode kernel divides by launch-fixed divisors (row costs of the line,
heads, window widths) with a multiply-high instead of a division: m =
ceil(2^64 / d) (m = 0 for d = 1), q = (x * m) >> 64, exact for 32-bit x;
a row-range offset of 2^32 or more takes a true division instead.  These
tests check that arithmetic, written here with Python's exact integers,
against floor division for every divisor the kernel uses and for dividends
at and around the points where an error would show: multiples of d and the
32-bit boundary."""
import random

MASK64 = (1 << 64) - 1


def fastdiv_m(d):
    # the host's make_fastdiv: ~0 / d + 1 in 64-bit unsigned arithmetic
    return 0 if d <= 1 else (MASK64 // d + 1) & MASK64


def fdiv32(x, d):
    m = fastdiv_m(d)
    return x if m == 0 else (x * m) >> 64


def _qblock_row_cost(k):
    return 132 * (k + 128) // 128


# row costs of the line (full-width / K_prun + V rows at k = 0..128, sealed
# block rows), head and (layer, sequence) counts, window widths
KERNEL_DIVISORS = sorted({2 * k + 256 for k in range(0, 129, 32)} | {_qblock_row_cost(k) for k in range(0, 129, 32)} |
                         {1, 2, 4, 7, 8, 28, 32, 64, 256, 512, 1024, 4096, 2048 * 64, 16 * 8})


def _dividends(d, rng, top):
    xs = {0, 1, d - 1, d, d + 1, 2 * d - 1, 2 * d, (1 << 32) - 1, top}
    for q in (1 << 20, (1 << 32) // d, top // d):
        xs.update({q * d - 1, q * d, q * d + 1})
    xs.update(rng.randrange(0, top + 1) for _ in range(200))
    return sorted(x for x in xs if 0 <= x <= top)


def test_all_divisors_are_exact_for_32_bit_dividends():
    # the form used for entry ids, window slots and head indices
    rng = random.Random(1)
    ds = KERNEL_DIVISORS + [rng.randrange(2, 1 << 32) for _ in range(50)] + [(1 << 32) - 1, 3, 5, 127]
    for d in ds:
        for x in _dividends(d, rng, (1 << 32) - 1):
            assert fdiv32(x, d) == x // d, (x, d)


def test_multiply_high_is_not_exact_past_32_bits():
    # why offsets of 2^32 or more take a true division: there the
    # multiply-high comes out one too large for some dividends
    rng = random.Random(3)
    bad = 0
    for d in KERNEL_DIVISORS:
        if d <= 1 or d & (d - 1) == 0:
            continue       # powers of two: m = 2^64 / d exactly
        for x in _dividends(d, rng, MASK64 - d):
            bad += fdiv32(x, d) != x // d
    assert bad > 0
