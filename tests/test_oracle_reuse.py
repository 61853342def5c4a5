"""Pins of the oracle's exponent-reuse codec (CIERA).

* Brute force on tiny shards: for every subset of changed positions the
  bitmap is the block-wise OR of the subset, the payload size is the closed
  form 64 + bitmap + sign+mantissa + B*changed (+ padding), and the decode
  rebuilds the current tensor while both caches end up equal to its
  exponents.
* Reuse rate: with i.i.d. exponent flips at rate c, a block of B values is
  reused with probability (1-c)^B (CIERA, block-partition paragraph); with
  20% of rows at 5c it is 0.8(1-c)^B + 0.2(1-5c)^B.
* Corrupted payloads are reported, never decoded past their bounds.
"""
import math

import numpy as np
import pytest
import torch

import synth


def cdiv(a, b):
    return -(-a // b)


def rup(a, b):
    return cdiv(a, b) * b


def exps(x):
    return ((x.astype(np.uint32) >> 7) & 0xFF).astype(np.uint8)


def bitmap_bits(pay, nb):
    bm = pay[64:64 + cdiv(nb, 8)]
    return [(int(bm[k // 8]) >> (k % 8)) & 1 for k in range(nb)]


@pytest.mark.parametrize("n", [1, 5, 8, 11])
@pytest.mark.parametrize("B", [1, 2, 3, 4, 8, 16])
def test_bruteforce_all_subsets(orc, n, B):
    rng = np.random.default_rng(n * 100 + B)
    prev = rng.integers(0, 65536, n, dtype=np.uint32).astype(np.uint16)
    nb = cdiv(n, B)
    for mask in range(1 << n):
        cur = prev.copy()
        for i in range(n):
            if (mask >> i) & 1:
                e = (int(cur[i]) >> 7) & 0xFF
                e2 = (e + 1 + int(rng.integers(0, 254))) % 256  # any other exponent
                cur[i] = (cur[i] & 0x807F) | (e2 << 7)
            else:
                cur[i] = (cur[i] & 0xFF80) | int(rng.integers(0, 128))  # mantissa drift
        send = exps(prev).copy()
        recv = exps(prev).copy()
        pay, _ = orc.reuse_encode(cur, B, 0, send)
        want = [int(any((mask >> i) & 1 for i in range(k * B, min((k + 1) * B, n))))
                for k in range(nb)]
        assert bitmap_bits(pay, nb) == want
        changed_len = sum(min((k + 1) * B, n) - k * B for k in range(nb) if want[k])
        assert pay.size == rup(64 + rup(cdiv(nb, 8), 16) + rup(n, 16) + rup(8 * cdiv(n, 8192), 16)
                               + changed_len, 128)
        assert np.array_equal(send, exps(cur))
        out, st = orc.reuse_decode(pay, n, B, 0, recv)
        assert st == 0 and np.array_equal(out, cur) and np.array_equal(recv, exps(cur))


def test_bruteforce_16_sampled_subsets(orc):
    n, rng = 16, np.random.default_rng(16)
    for B in (1, 2, 3, 4, 8, 16):
        for mask in list(rng.integers(0, 1 << n, 300)) + [0, (1 << n) - 1]:
            prev = rng.integers(0, 65536, n, dtype=np.uint32).astype(np.uint16)
            cur = prev.copy()
            for i in range(n):
                if (int(mask) >> i) & 1:
                    cur[i] ^= 0x0080     # flips the exponent's low bit
            send, recv = exps(prev).copy(), exps(prev).copy()
            pay, _ = orc.reuse_encode(cur, B, 0, send)
            nb = cdiv(n, B)
            want = [int(any((int(mask) >> i) & 1 for i in range(k * B, min((k + 1) * B, n))))
                    for k in range(nb)]
            assert bitmap_bits(pay, nb) == want
            out, st = orc.reuse_decode(pay, n, B, 0, recv)
            assert st == 0 and np.array_equal(out, cur)


def _reuse_rate(orc, x0, x1, B):
    n = x0.size
    send = exps(x0).copy()
    pay, _ = orc.reuse_encode(x1, B, 0, send)
    nb = cdiv(n, B)
    return 1.0 - int(pay[24:32].view(np.uint64)[0]) / nb, nb


@pytest.mark.parametrize("B", [64, 128, 256, 512, 1024])
def test_reuse_rate_uniform_flips(orc, B):
    c = 0.005
    n = 1 << 22
    x0 = synth.gaussian_bf16(n, 0.02, synth.key_of(21, 0))
    x1 = synth.flip_exponents(x0, torch.tensor(c, dtype=torch.float64), synth.key_of(21, 1))
    x0, x1 = x0.numpy().view(np.uint16), x1.numpy().view(np.uint16)
    rate, nb = _reuse_rate(orc, x0, x1, B)
    p = (1 - c) ** B
    assert abs(rate - p) < 5 * math.sqrt(p * (1 - p) / nb) + 1e-9
    # (1 - c)^B at c = 0.005 to four places
    table = {64: 0.7256, 128: 0.5264, 256: 0.2771, 512: 0.0768, 1024: 0.0059}
    assert p == pytest.approx(table[B], abs=1e-4)
    # the realised element change rate is c
    ch = np.count_nonzero(exps(x0) != exps(x1)) / n
    assert abs(ch - c) < 5 * math.sqrt(c * (1 - c) / n)


@pytest.mark.parametrize("B", [64, 256, 1024])
def test_reuse_rate_clustered_rows(orc, B):
    """20% of rows at 5c: rate 0.8 (1-c)^B + 0.2 (1-5c)^B (rows of 2048)."""
    c = 0.005
    seg = synth.Segment("expert_ffn", 2048, 2048, 0.02, 0.0, c)
    x0 = synth._segments_base([seg], synth.key_of(22, 0), "cpu")
    rate_t = synth._segments_rate([seg], x0.numel(), 1.0, True, synth.key_of(22, 7), "cpu")
    x1 = synth.flip_exponents(x0, rate_t, synth.key_of(22, 1))
    rate, nb = _reuse_rate(orc, x0.numpy().view(np.uint16), x1.numpy().view(np.uint16), B)
    p = 0.8 * (1 - c) ** B + 0.2 * (1 - 5 * c) ** B
    # rows (not blocks) are the independent unit of the hot/cold draw
    rows = 2048
    assert abs(rate - p) < 5 * math.sqrt(0.16 * ((1 - c) ** B - (1 - 5 * c) ** B) ** 2 / rows
                                          + p * (1 - p) / nb)


def test_norm_category_is_fully_reused(orc):
    seg = synth.Segment("norm", 1, 2048, 0.01, 1.0, 0.0)
    x0 = synth._segments_base([seg], synth.key_of(23, 0), "cpu")
    x1 = synth.flip_exponents(x0, torch.tensor(0.0, dtype=torch.float64), synth.key_of(23, 1))
    rate, _ = _reuse_rate(orc, x0.numpy().view(np.uint16), x1.numpy().view(np.uint16), 256)
    assert rate == 1.0


def _good_payload(orc, coded=False):
    rng = np.random.default_rng(31)
    n, B = 3000, 64
    prev = rng.integers(0, 65536, n, dtype=np.uint32).astype(np.uint16)
    cur = prev.copy()
    cur[::97] ^= 0x0100
    send = exps(prev).copy()
    pay, _ = orc.reuse_encode(cur, B, 2, send, coded=coded)
    return pay, prev, cur, n, B


@pytest.mark.parametrize("coded", [False, True])
def test_corrupt_reuse_payloads(orc, coded):
    pay, prev, cur, n, B = _good_payload(orc, coded)
    ok, st = orc.reuse_decode(pay.copy(), n, B, 2, exps(prev).copy())
    assert st == 0 and np.array_equal(ok, cur)
    cases = []
    bad = pay.copy(); bad[0] ^= 1; cases.append((bad, None, orc.BAD_HEADER))
    bad = pay.copy(); bad[4] = 1; cases.append((bad, None, orc.BAD_HEADER))
    bad = pay.copy(); bad[12] = 3; cases.append((bad, None, orc.BAD_HEADER))
    bad = pay.copy(); cases.append((bad, pay.size - 128, orc.BAD_SIZE))   # truncated
    bad = pay.copy(); bad[48] ^= 0x80; cases.append((bad, None, orc.BAD_SIZE))
    bad = pay.copy(); bad[64] ^= 0x01; cases.append((bad, None, orc.BAD_COUNT))  # bitmap bit
    bad = pay.copy(); bad[24] += 1; cases.append((bad, None, None))
    for b, avail, want in cases:
        _, st = orc.reuse_decode(b, n, B, 2, exps(prev).copy(), avail=avail)
        assert st != 0
        if want is not None:
            assert st & want, (st, want)
    assert orc.reuse_decode(pay[:10], n, B, 2, exps(prev).copy())[1] == orc.BAD_SIZE


def test_corrupt_code3_chunks(orc):
    rng = np.random.default_rng(41)
    x = (rng.normal(0, 0.02, 5000).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    slots, sizes, slot = orc.code3_encode(x, 2, orc.stats(x)["E0"])
    recv, offs = orc.compact(slots, sizes, slot)
    assert orc.code3_decode(recv, offs, x.size, 2)[1] == 0
    bad = recv.copy(); bad[0] = 0; assert orc.code3_decode(bad, offs, x.size, 2)[1] & orc.BAD_HEADER
    bad = recv.copy(); bad[32] = 1; assert orc.code3_decode(bad, offs, x.size, 2)[1] & orc.BAD_HEADER
    o2 = offs.copy(); o2[1] -= 128
    assert orc.code3_decode(recv, o2, x.size, 2)[1] & orc.BAD_SIZE
    # a plane bit set on an escape changes the escape count
    n_c = orc.shard_count(x.size, 2, 0)
    base = 128 + rup(n_c, 128)
    bad = recv.copy()
    codes0 = [(int(bad[base + p * rup(cdiv(n_c, 8), 128)]) & 1) for p in range(3)]
    if codes0 == [0, 0, 0]:
        bad[base] |= 1
    else:
        for p in range(3):
            bad[base + p * rup(cdiv(n_c, 8), 128)] &= 0xFE
    assert orc.code3_decode(bad, offs, x.size, 2)[1] & orc.BAD_COUNT
    # every bounded-size cut of the buffer is rejected, never read past
    for cut in (1, 127, 128, int(sizes[0]) - 1):
        o3 = np.array([0, cut, cut], np.uint64)
        assert orc.code3_decode(recv[:cut], o3, x.size, 2)[1] != 0


def test_empty_and_short_shards(orc):
    rng = np.random.default_rng(51)
    for n, W, B in [(0, 4, 64), (1, 1, 64), (100, 8, 16), (129, 2, 8), (1000, 3, 7)]:
        x = rng.integers(0, 65536, n, dtype=np.uint32).astype(np.uint16)
        send = np.zeros(max(n, 1), np.uint8)
        recv = np.zeros(max(n, 1), np.uint8)
        for cold in (True, False):
            slots, sizes, slot, _ = orc.reuse_encode_all(x, W, B, send, cold=cold)
            rb, offs = orc.compact(slots, sizes, slot)
            out, st = orc.gather_decode_reuse(rb, offs, n, W, B, recv)
            assert st == 0 and np.array_equal(out, x)
        st = orc.stats(x)
        slots, sizes, slot = orc.code3_encode(x, W, st["E0"])
        rb, offs = orc.compact(slots, sizes, slot)
        out, s = orc.code3_decode(rb, offs, n, W)
        assert s == 0 and np.array_equal(out, x)
        for r in range(W):
            if orc.shard_count(n, W, r) == 0:
                assert int(sizes[r]) == 128
