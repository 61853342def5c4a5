"""Pins of the CPU oracle's byte layouts and its lossless round trips.

What pins what:
* every one of the 65,536 BF16 patterns must come back bit for bit through
  both codecs (CIERA: "every gathered parameter is reconstructed
  bit-for-bit"), for every window base and several chunk / block sizes;
* the hand-worked bytes in tests/golden/format_examples.txt pin the code
  mapping, the bit order of the planes, the section offsets and the headers;
* escape counts are checked against a numpy histogram of the exponent field;
* payload sizes are checked against the pages' accounting (8 bits of
  sign+mantissa and 3 code bits per value plus 8 bits per escape; bitmap +
  sign+mantissa + changed exponents), with only header and padding on top.
"""
import os

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ALL = np.arange(65536, dtype=np.uint32).astype(np.uint16)


def cdiv(a, b):
    return -(-a // b)


def rup(a, b):
    return cdiv(a, b) * b


def exps(x):
    return ((x.astype(np.uint32) >> 7) & 0xFF).astype(np.uint8)


def load_examples():
    """Scalar rows by key; image rows (<name>_fill off len hex, <name>_bytes
    off hex...) by image name, in file order."""
    rows = {}
    byte_rows = {}
    with open(os.path.join(HERE, "golden", "format_examples.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key.endswith("_bytes"):
                byte_rows.setdefault(key[:-6], []).append(
                    (int(vals[0]), bytes(int(v, 16) for v in vals[1:])))
            elif key.endswith("_fill"):
                byte_rows.setdefault(key[:-5], []).append(
                    (int(vals[0]), bytes([int(vals[2], 16)]) * int(vals[1])))
            else:
                rows[key] = vals
    return rows, byte_rows


def expected_image(total, byte_rows):
    img = bytearray(total)
    for off, bs in byte_rows:
        img[off:off + len(bs)] = bs
    return bytes(img)


def multi_input(rows):
    x = np.full(int(rows["multi_n"][0]), 0x3C00, dtype=np.uint16)
    for item in rows["multi_special"]:
        j, bits = item.split(":")
        x[int(j)] = int(bits, 16)
    return x


def test_code3_golden_example(orc):
    rows, byte_rows = load_examples()
    x = np.array([int(v, 16) for v in rows["input"]], dtype=np.uint16)
    E0 = int(rows["code3_E0"][0])
    slots, sizes, slot = orc.code3_encode(x, 1, E0)
    total = int(rows["code3_total"][0])
    assert int(sizes[0]) == total
    assert bytes(slots[:total]) == expected_image(total, byte_rows["code3"])
    out, st = orc.code3_decode(slots, np.array([0, slot], np.uint64), x.size, 1)
    assert st == 0 and np.array_equal(out, x)


def test_reuse_golden_example(orc):
    rows, byte_rows = load_examples()
    x = np.array([int(v, 16) for v in rows["input"]], dtype=np.uint16)
    B = int(rows["reuse_B"][0])
    cache = exps(x).copy()
    cache[5] = int(rows["reuse_prev_exp5"][0])
    recv_cache = cache.copy()
    pay, _ = orc.reuse_encode(x, B, 0, cache)
    total = int(rows["reuse_total"][0])
    assert pay.size == total
    assert bytes(pay) == expected_image(total, byte_rows["reuse"])
    assert np.array_equal(cache, exps(x))
    out, st = orc.reuse_decode(pay, x.size, B, 0, recv_cache)
    assert st == 0 and np.array_equal(out, x) and np.array_equal(recv_cache, exps(x))


def test_code3_golden_index_example(orc):
    """Three 8192-value index entries, worked by hand."""
    rows, byte_rows = load_examples()
    x = multi_input(rows)
    slots, sizes, slot = orc.code3_encode(x, 1, int(rows["code3m_E0"][0]))
    total = int(rows["code3m_total"][0])
    assert int(sizes[0]) == total
    assert bytes(slots[:total]) == expected_image(total, byte_rows["code3m"])
    out, st = orc.code3_decode(slots, np.array([0, slot], np.uint64), x.size, 1)
    assert st == 0 and np.array_equal(out, x)


def test_reuse_golden_index_example(orc):
    rows, byte_rows = load_examples()
    x = np.full(int(rows["multi_n"][0]), 0x3C00, dtype=np.uint16)
    B = int(rows["reuse" + "m_B"][0])
    cache = exps(x).copy()
    cache[[int(v) for v in rows["reusem_prev0"]]] = 0
    recv_cache = cache.copy()
    pay, _ = orc.reuse_encode(x, B, 0, cache)
    total = int(rows["reusem_total"][0])
    assert pay.size == total
    assert bytes(pay) == expected_image(total, byte_rows["reusem"])
    out, st = orc.reuse_decode(pay, x.size, B, 0, recv_cache)
    assert st == 0 and np.array_equal(out, x) and np.array_equal(recv_cache, exps(x))


def test_index_entries_are_checked(orc):
    """A decoder that finds an index entry different from the count it
    derives itself reports a count error (code3 and reuse)."""
    rows, _ = load_examples()
    x = multi_input(rows)
    slots, sizes, slot = orc.code3_encode(x, 1, 120)
    bad = slots.copy()
    bad[23168 + 8] ^= 1
    _, st = orc.code3_decode(bad, np.array([0, slot], np.uint64), x.size, 1)
    assert st == orc.BAD_COUNT
    y = np.full(x.size, 0x3C00, dtype=np.uint16)
    cache = exps(y).copy()
    cache[[3, 8190]] = 0
    pay, _ = orc.reuse_encode(y, 8, 0, cache.copy())
    bad = pay.copy()
    bad[16736 + 16] ^= 1
    _, st = orc.reuse_decode(bad, y.size, 8, 0, cache.copy())
    assert st == orc.BAD_COUNT


@pytest.mark.parametrize("W", [1, 3, 8])
def test_code3_all_patterns_every_window(orc, W):
    """All 65,536 patterns (incl. +-0, subnormals, +-Inf, NaN payloads)
    round-trip for every window base E0 in 0..249."""
    e = exps(ALL)
    hist = np.bincount(e, minlength=256)
    L = orc.shard_len(ALL.size, W)
    for E0 in range(250):
        slots, sizes, slot = orc.code3_encode(ALL, W, E0)
        recv, offs = orc.compact(slots, sizes, slot)
        out, st = orc.code3_decode(recv, offs, ALL.size, W)
        assert st == 0
        assert np.array_equal(out, ALL), E0
        # escapes are exactly the values outside E0..E0+6 (numpy histogram)
        n_esc_total = 0
        for c in range(W):
            n_c = orc.shard_count(ALL.size, W, c)
            ec = e[c * L:c * L + n_c]
            n_esc = int(np.count_nonzero((ec < E0) | (ec > E0 + 6)))
            n_esc_total += n_esc
            hdr = slots[c * slot:c * slot + 128]
            assert int(hdr[16:24].view(np.uint64)[0]) == n_esc
            # the pages' accounting: 8 + 3 bits per value, 8 per escape,
            # plus a 128-B header and at most 127 B of padding per section
            payload_bits = 11 * n_c + 8 * n_esc
            assert payload_bits <= 8 * int(sizes[c]) <= payload_bits + 8 * (128 + 5 * 127)
        assert n_esc_total == ALL.size - int(hist[E0:E0 + 7].sum())


@pytest.mark.parametrize("B", [1, 7, 64, 256])
@pytest.mark.parametrize("coded", [False, True])
def test_reuse_all_patterns(orc, B, coded):
    """Every pattern survives a cold and then a warm reuse round trip."""
    rng = np.random.default_rng(B)
    W = 3
    n = ALL.size
    x0 = rng.permutation(ALL)
    send = np.zeros(n, np.uint8)
    recv = np.zeros(n, np.uint8)
    slots, sizes, slot, _ = orc.reuse_encode_all(x0, W, B, send, cold=True, coded=coded)
    rb, offs = orc.compact(slots, sizes, slot)
    out, st = orc.gather_decode_reuse(rb, offs, n, W, B, recv)
    assert st == 0 and np.array_equal(out, x0)
    assert np.array_equal(send, exps(x0)) and np.array_equal(recv, exps(x0))
    # cold payload size is the closed form with every block changed
    L = orc.shard_len(n, W)
    for r in range(W):
        n_r = orc.shard_count(n, W, r)
        nb = cdiv(n_r, B)
        raw = 64 + rup(cdiv(nb, 8), 16) + rup(n_r, 16) + rup(8 * cdiv(n_r, 8192), 16) + n_r
        if not coded:
            assert int(sizes[r]) == rup(raw, 128)
    # warm: another permutation of all patterns
    x1 = rng.permutation(ALL)
    slots, sizes, slot, _ = orc.reuse_encode_all(x1, W, B, send, cold=False, coded=coded)
    rb, offs = orc.compact(slots, sizes, slot)
    out, st = orc.gather_decode_reuse(rb, offs, n, W, B, recv)
    assert st == 0 and np.array_equal(out, x1)
    assert np.array_equal(recv, exps(x1))
    del L


def test_unchanged_iteration_sends_no_exponents(orc):
    rng = np.random.default_rng(5)
    x = rng.integers(0, 65536, 5000, dtype=np.uint32).astype(np.uint16)
    cache = exps(x).copy()
    pay, _ = orc.reuse_encode(x, 64, 0, cache)
    hdr = pay[:64]
    assert int(hdr[24:32].view(np.uint64)[0]) == 0          # n_changed
    nb = cdiv(5000, 64)
    assert pay.size == rup(64 + rup(cdiv(nb, 8), 16) + rup(5000, 16) + rup(8 * cdiv(5000, 8192), 16),
                           128)


def test_composed_matches_code3_of_exp_stream(orc):
    """The coded EXP section equals the code3 planes/escapes of the raw EXP
    stream under the same window (cross-check between the two codecs)."""
    import synth
    import torch
    x0 = synth.gaussian_bf16(40000, 0.02, synth.key_of(9, 0)).numpy().view(np.uint16)
    x1 = synth.flip_exponents(torch.from_numpy(x0.view(np.int16)),
                              torch.tensor(0.01, dtype=torch.float64),
                              synth.key_of(9, 1)).numpy().view(np.uint16)
    B = 64
    c_raw = exps(x0).copy()
    c_cod = exps(x0).copy()
    raw, _ = orc.reuse_encode(x1, B, 0, c_raw)
    cod, st = orc.reuse_encode(x1, B, 0, c_cod, coded=True)
    assert st["E0"] == orc.stats(x1)["E0"]
    m = int(raw[32:40].view(np.uint64)[0])
    nb = cdiv(x1.size, B)
    off_x = 64 + rup(cdiv(nb, 8), 16) + rup(x1.size, 16) + rup(8 * cdiv(x1.size, 8192), 16)
    off_c = 64 + rup(cdiv(nb, 8), 16) + rup(x1.size, 16) + rup(16 * cdiv(x1.size, 8192), 16)
    stream = raw[off_x:off_x + m]
    # a BF16 tensor whose exponents are the stream (sign+mantissa zero)
    xs = (stream.astype(np.uint16) << 7)
    slots, sizes, slot = orc.code3_encode(xs, 1, st["E0"])
    plane = rup(cdiv(m, 8), 16)
    p128 = rup(cdiv(m, 8), 128)
    base3 = 128 + rup(m, 128)
    for p in range(3):
        got = cod[off_c + p * plane:off_c + p * plane + (m + 7) // 8]
        want = slots[base3 + p * p128:base3 + p * p128 + (m + 7) // 8]
        assert np.array_equal(got, want)
    n_esc = int(cod[40:48].view(np.uint64)[0])
    assert n_esc == int(slots[16:24].view(np.uint64)[0])
    esc3 = base3 + 3 * p128 + rup(8 * cdiv(m, 8192), 128)
    esc_c3 = slots[esc3:esc3 + n_esc]
    assert np.array_equal(cod[off_c + 3 * plane:off_c + 3 * plane + n_esc], esc_c3)
    # and both decode to x1
    r1 = exps(x0).copy()
    r2 = exps(x0).copy()
    o1, s1 = orc.reuse_decode(raw, x1.size, B, 0, r1)
    o2, s2 = orc.reuse_decode(cod, x1.size, B, 0, r2)
    assert s1 == s2 == 0 and np.array_equal(o1, x1) and np.array_equal(o2, x1)
