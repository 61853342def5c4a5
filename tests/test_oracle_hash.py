"""Hash-based change detection (CIERA's HashCache: two independent 64-bit
SplitMix64 hashes per block), oracle side.

Pins: the SplitMix64 generator's published first outputs (tests/golden);
payload equality with the direct exponent compare over cold and warm
iterations (the bitmap is the same unless a hash pair collides, p ~ 2^-128);
a change of any single exponent is always detected; mantissa-only changes
never mark a block."""
import os

import numpy as np
import pytest

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "splitmix64_seed0.txt")


def _flip(rng, x, rate):
    y = x.copy()
    e = (y >> 7) & 0xFF
    pick = (rng.random(x.size) < rate) & (e > 1) & (e < 254)
    e2 = np.where(rng.random(x.size) < 0.5, e - 1, e + 1)
    y[pick] = (y[pick] & 0x807F) | (e2[pick].astype(np.uint16) << 7)
    # mantissa noise on every value: must never mark a block on its own
    y = (y & 0xFF80) | (rng.integers(0, 128, x.size).astype(np.uint16))
    return y


def test_splitmix64_published_outputs(orc):
    with open(GOLDEN) as f:
        want = [int(l, 16) for l in f if l.strip() and not l.startswith("#")]
    assert orc.splitmix64(0, 3) == want


@pytest.mark.parametrize("n", [0, 1, 1000, 8197, 50_000])
@pytest.mark.parametrize("B", [8, 32, 256, 1024])
@pytest.mark.parametrize("coded", [False, True])
def test_hash_payload_equals_direct_compare(orc, n, B, coded):
    rng = np.random.default_rng(n + B + coded)
    xs = [synth.config2(max(n, 1), seed=5).numpy().view(np.uint16)[:n]]
    for rate in (0.0, 0.001, 0.02):
        xs.append(_flip(rng, xs[-1], rate))
    nb = -(-n // B)
    ecache = np.zeros(max(n, 1), np.uint8)
    hcache = np.zeros(2 * max(nb, 1), np.uint64)
    for it, x in enumerate(xs):
        a, sa = orc.reuse_encode(x, B, 3, ecache, cold=it == 0, coded=coded)
        b, sb = orc.reuse_encode_hash(x, B, 3, hcache, cold=it == 0, coded=coded)
        assert np.array_equal(a, b), it
        if coded:
            assert sa["E0"] == sb["E0"]
    # the cache holds the last tensor's block hashes
    for k in range(nb):
        assert int(hcache[2 * k]) == orc.block_hash(xs[-1], B, k, 0)
        assert int(hcache[2 * k + 1]) == orc.block_hash(xs[-1], B, k, 1)


def test_single_exponent_change_is_always_detected(orc):
    rng = np.random.default_rng(9)
    n, B = 4096, 256
    x = synth.config2(n, seed=6).numpy().view(np.uint16)
    h0 = [(orc.block_hash(x, B, k, 0), orc.block_hash(x, B, k, 1)) for k in range(n // B)]
    assert len(set(h0)) == len(h0)
    for v in rng.integers(0, n, 64):
        y = x.copy()
        e = (int(y[v]) >> 7) & 0xFF
        for d in (1, 2, 37):
            y[v] = (int(x[v]) & 0x807F) | (((e + d) & 0xFF) << 7)
            k = int(v) // B
            assert orc.block_hash(y, B, k, 0) != h0[k][0]
            assert orc.block_hash(y, B, k, 1) != h0[k][1]
    # only mantissas and signs changed: every hash stays
    y = x ^ np.uint16(0x807F)
    assert all((orc.block_hash(y, B, k, 0), orc.block_hash(y, B, k, 1)) == h0[k] for k in range(n // B))
