"""The kernels split a CTA index n into chunk and tile with one multiply:
q = floor(n * r / 2^64), r = floor((2^64 - 1) / d) + 1 for d >= 2 (the
device side of FastDiv in ez_common.cuh).  The claim is that q == n // d for
every 32-bit n and d; this checks it on the edge cases and random pairs with
Python integers (exact)."""
import random

M64 = (1 << 64) - 1


def fast_quot(n: int, d: int) -> int:
    if d == 1:
        return n
    r = M64 // d + 1
    assert r < (1 << 64)
    return (n * r) >> 64


def test_fastdiv_edges():
    ds = [1, 2, 3, 5, 7, 8, 9, 255, 256, 257, 1000, 8191, 8192, 8193, 16384, 65535, 65536, 65537,
          (1 << 31) - 1, 1 << 31, (1 << 31) + 1, (1 << 32) - 2, (1 << 32) - 1]
    ns = [0, 1, 2, 3, 1023, 1024, 65535, 65536, (1 << 31) - 1, 1 << 31, (1 << 32) - 2, (1 << 32) - 1]
    for d in ds:
        for n in ns + [d - 1, d, d + 1, 2 * d - 1, 2 * d, 3 * d - 1]:
            if 0 <= n < (1 << 32):
                assert fast_quot(n, d) == n // d, (n, d)


def test_fastdiv_random():
    rng = random.Random(12345)
    for _ in range(200_000):
        d = rng.randrange(1, 1 << 32) if rng.random() < 0.5 else rng.randrange(1, 1 << 16)
        n = rng.randrange(0, 1 << 32)
        assert fast_quot(n, d) == n // d, (n, d)
        # the worst n for d: the largest multiple of d minus one
        m = ((1 << 32) - 1) // d * d - 1
        if m >= 0:
            assert fast_quot(m, d) == m // d, (m, d)
