"""Host-side pins of the fixed-divisor division the kernels use for index
math (Granlund-Montgomery, "Division by invariant integers using
multiplication", section 4): the constants make_fastdiv computes, applied
with the device formula (mulhi(n, m) + n) >> s, equal n // d."""
import random

import pytest


def make_fastdiv(d):
    # the same recipe as kv4_internal.h, written from the paper's definition
    s = 0
    while (1 << s) < d:
        s += 1
    m = ((1 << 32) * ((1 << s) - d)) // d + 1
    return m, s


def apply(n, m, s):
    hi = (n * m) >> 32                 # __umulhi
    return ((hi + n) & 0xFFFFFFFF) >> s


@pytest.mark.parametrize("d", [1, 2, 3, 4, 5, 6, 7, 12, 16, 24, 64, 96, 100, 255, 256, 1600,
                               65535, 65536, 1 << 20, (1 << 31) - 1])
def test_fastdiv_edges(d):
    m, s = make_fastdiv(d)
    assert 0 <= m < (1 << 32)
    limit = (1 << 31) - 1
    cases = {0, 1, d - 1, d, d + 1, limit, limit - 1}
    for k in (1, 2, 3, 1000, limit // d):
        for delta in (-1, 0, 1):
            cases.add(k * d + delta)
    for n in cases:
        if 0 <= n <= limit:
            assert apply(n, m, s) == n // d, (n, d)


def test_fastdiv_random():
    rng = random.Random(7)
    for _ in range(200):
        d = rng.randrange(1, 1 << 31)
        m, s = make_fastdiv(d)
        for _ in range(200):
            n = rng.randrange(0, 1 << 31)
            assert apply(n, m, s) == n // d
