"""The decode kernel divides by per-call divisors (KV heads, row tiles,
split size, GQA group) with a multiply: q = high 64 bits of x * ceil(2^64 / d)
(d = 1: q = x), and query rows by G with (r * ceil(2^32 / G)) >> 32.  This
checks the exactness those replacements rely on, over every 32-bit x class
that could break it: multiples of d and their neighbours, the top of the
range, and every small x, for divisors across their whole range."""
import random

import pytest

M64 = (1 << 64) - 1


def q64(x, d):
    m = 0 if d <= 1 else M64 // d + 1          # the host's make_fastdiv
    return x if d <= 1 else (x * m) >> 64      # the device's fdiv


def q32(r, g):
    m = ((1 << 32) + g - 1) // g                # ceil(2^32 / G)
    return (r * m) >> 32


def _divisors():
    rnd = random.Random(7)
    ds = list(range(1, 4097)) + [1 << k for k in range(13, 32)] + [(1 << 32) - 1, (1 << 31) + 1]
    ds += [rnd.randrange(4097, 1 << 32) for _ in range(2000)]
    return ds


@pytest.mark.parametrize("chunk", range(4))
def test_fastdiv_is_exact_for_32_bit_dividends(chunk):
    rnd = random.Random(chunk)
    ds = _divisors()[chunk::4]
    for d in ds:
        xs = {0, 1, d - 1, d, d + 1, (1 << 32) - 1, (1 << 31) - 1}
        top = ((1 << 32) - 1) // d
        for k in (1, 2, 3, top - 1, top, rnd.randrange(1, top + 1)):
            for e in (-1, 0, 1):
                x = k * d + e
                if 0 <= x < (1 << 32):
                    xs.add(x)
        xs.update(rnd.randrange(0, 1 << 32) for _ in range(20))
        for x in xs:
            assert q64(x, d) == x // d, (x, d)


def test_row_division_by_the_group_is_exact():
    # rows r < 32 and groups G <= 32 (the decode's limits), and well beyond
    for g in range(1, 257):
        for r in range(0, 4096):
            assert q32(r, g) == r // g, (r, g)
