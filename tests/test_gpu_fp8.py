"""GPU parity of the FP8 3-bit exponent codec (E5M2, E4M3) with the oracle,
through the C ABI (ez_fp8_stats, ez_fp8_encode, ez_fp8_decode and
ez_gather_decode on an FP8 plan).

* Statistics records bit for bit: every byte pattern, random bytes of many
  lengths, Gaussian tensors over a sigma sweep, the histogram window.
* Chunks byte for byte and size tables: every window base on all 256
  patterns, ragged W and lengths, empty and short chunks, a 2^24-value
  Gaussian tensor.
* Decoding: lossless, and the oracle's status bits on corrupt chunks.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import fbits

pytestmark = pytest.mark.gpu

FMTS = {"e5m2": (4, 1, 25), "e4m3": (5, 2, 9)}   # plan codec, oracle format code, largest E0


@pytest.fixture(scope="module")
def ez():
    from lossless_bf16_exponent_codec_gb300 import build
    build.build()
    from lossless_bf16_exponent_codec_gb300 import binding, codec
    return binding, codec


def dev8(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.uint8)).cuda()


def assert_fp8_stats_equal(g: dict, o: dict):
    nb = o["hist"].size          # 32 bins for E5M2, 16 for E4M3 (the record's other bins are 0)
    assert np.array_equal(g["hist"][:nb], o["hist"]), ("hist", g["hist"], o["hist"])
    assert not g["hist"][nb:].any()
    for k in ("n", "n_finite", "E0", "rule", "n_escape"):
        assert g[k] == o[k], (k, g[k], o[k])
    for k in ("s1", "s2", "var", "sigma", "K"):
        assert fbits(g[k]) == fbits(o[k]), (k, g[k], o[k])


def run_stats(ez, x: np.ndarray, codec: int, flags: int = 0) -> dict:
    _, cd = ez
    c = cd.Fp8Codec(max(x.size, 1), 1, codec, flags=flags)
    c.stats(dev8(x) if x.size else torch.zeros(16, dtype=torch.uint8, device="cuda"), x.size)
    torch.cuda.synchronize()
    return c.stats_of()


def inputs():
    rng = np.random.default_rng(8)
    yield "patterns", np.arange(256, dtype=np.uint8)
    for n in (1, 2, 17, 1000, 65537, (1 << 20) + 3):
        yield f"random{n}", rng.integers(0, 256, n).astype(np.uint8)


@pytest.mark.parametrize("fmt", list(FMTS))
def test_fp8_stats_patterns_and_random(ez, orc, fmt):
    codec, ofmt, _ = FMTS[fmt]
    for name, x in inputs():
        assert_fp8_stats_equal(run_stats(ez, x, codec), orc.fp8_stats(x, ofmt))


@pytest.mark.parametrize("fmt", list(FMTS))
@pytest.mark.parametrize("sigma", [2.0 ** -9, 0.02, 0.3, 1.0, 7.5, 40.0])
def test_fp8_stats_gaussian(ez, orc, fmt, sigma):
    codec, ofmt, _ = FMTS[fmt]
    x = synth.fp8_gaussian(300_007, sigma, fmt, seed=int(sigma * 1000) % 97).numpy()
    for mode in (0, 1):
        g = run_stats(ez, x, codec, flags=mode)
        assert_fp8_stats_equal(g, orc.fp8_stats(x, ofmt, window_mode=mode))


def test_fp8_stats_empty(ez, orc):
    for fmt, (codec, ofmt, _) in FMTS.items():
        assert_fp8_stats_equal(run_stats(ez, np.zeros(0, np.uint8), codec), orc.fp8_stats(np.zeros(0, np.uint8), ofmt))


def stats_record(binding, E0: int) -> torch.Tensor:
    """An ez_fp8_stats_t whose only meaningful field is E0 (the encoder reads
    nothing else)."""
    raw = np.zeros(binding.FP8_STATS_BYTES, np.uint8)
    raw[312:316] = np.frombuffer(np.uint32(E0).tobytes(), np.uint8)
    return dev8(raw)


def encode_compare(ez, orc, x: np.ndarray, W: int, fmt: str, E0: int):
    binding, cd = ez
    codec, ofmt, _ = FMTS[fmt]
    c = cd.Fp8Codec(x.size, W, codec)
    st = stats_record(binding, E0)
    xd = dev8(x) if x.size else torch.zeros(16, dtype=torch.uint8, device="cuda")
    binding.ez_fp8_encode(c.plan, xd, 0, W, st, c.out, c.out.numel(), c.sizes, c.status, c.ws, c.ws_bytes)
    torch.cuda.synchronize()
    assert c.status_word() == 0
    oslots, osizes, oslot = orc.fp8_encode(x, W, ofmt, E0)
    assert oslot == c.slot
    gs = c.sizes.cpu().numpy().astype(np.uint64)
    assert np.array_equal(gs, osizes), (gs, osizes)
    got = c.out.cpu().numpy()
    for r in range(W):
        k = int(osizes[r])
        a, b = got[r * c.slot:r * c.slot + k], oslots[r * oslot:r * oslot + k]
        if not np.array_equal(a, b):
            bad = np.nonzero(a != b)[0]
            raise AssertionError(f"{fmt} W={W} E0={E0} chunk {r}: {bad.size} bytes differ, first {bad[:8]}")
    # round trip through the gather-decode of the receive layout
    recv, offs = orc.compact(oslots, osizes, oslot)
    rd = dev8(recv if recv.size else np.zeros(16, np.uint8))
    od = torch.from_numpy(offs.astype(np.int64)).cuda()
    out = torch.zeros(max(x.size, 16), dtype=torch.uint8, device="cuda")
    c.clear_status()
    c.gather_decode(rd, od, out)
    torch.cuda.synchronize()
    assert c.status_word() == 0
    assert np.array_equal(out[:x.size].cpu().numpy(), x)
    return c, oslots, osizes, oslot


@pytest.mark.parametrize("fmt", list(FMTS))
def test_fp8_every_window_base_on_all_patterns(ez, orc, fmt):
    _, _, emax0 = FMTS[fmt]
    x = np.tile(np.arange(256, dtype=np.uint8), 37)   # 9472 values: two spans
    for E0 in range(emax0 + 1):
        encode_compare(ez, orc, x, 3, fmt, E0)


@pytest.mark.parametrize("fmt", list(FMTS))
@pytest.mark.parametrize("n,W", [(0, 1), (1, 1), (255, 2), (8192, 1), (8193, 3), (100_003, 8),
                                 (40_000, 16), ((1 << 20) + 77, 5)])
def test_fp8_round_trip_bytes(ez, orc, fmt, n, W):
    codec, ofmt, _ = FMTS[fmt]
    x = synth.fp8_gaussian(n, 1.0 if fmt == "e5m2" else 16.0, fmt, seed=n % 89).numpy()
    E0 = orc.fp8_stats(x, ofmt)["E0"]
    encode_compare(ez, orc, x, W, fmt, E0)


@pytest.mark.parametrize("fmt", list(FMTS))
def test_fp8_full_path_2p24(ez, orc, fmt):
    """Statistics on the device feed the encode; 2^24 Gaussian values with
    1% of entries x64 (escapes above the window), W = 8."""
    binding, cd = ez
    codec, ofmt, _ = FMTS[fmt]
    n, W = 1 << 24, 8
    sigma = 1.0 if fmt == "e5m2" else 16.0
    x = synth.fp8_gaussian(n, sigma, fmt, seed=3).numpy().copy()
    big = synth.fp8_gaussian(n // 100, sigma * 64, fmt, seed=4).numpy()
    x[np.arange(n // 100) * 100 + 7] = big
    c = cd.Fp8Codec(n, W, codec)
    xd = dev8(x)
    c.stats(xd)
    c.encode(xd)
    c.gather_decode()
    torch.cuda.synchronize()
    assert c.status_word() == 0
    ost = orc.fp8_stats(x, ofmt)
    assert_fp8_stats_equal(c.stats_of(), ost)
    oslots, osizes, oslot = orc.fp8_encode(x, W, ofmt, ost["E0"])
    assert np.array_equal(c.sizes.cpu().numpy().astype(np.uint64), osizes)
    got = c.out.cpu().numpy()
    for r in range(W):
        k = int(osizes[r])
        assert np.array_equal(got[r * c.slot:r * c.slot + k], oslots[r * oslot:r * oslot + k]), r
    assert np.array_equal(c.full[:n].cpu().numpy(), x)
    # the pages' factors, 6/8 (E5M2) and 7/8 (E4M3), plus one byte per escape
    # and the headers, index and padding (the x64 entries inflate sigma, so
    # the window sits higher and more of the bulk escapes)
    e = float(osizes.sum()) / n
    base = 0.75 if fmt == "e5m2" else 0.875
    assert base + ost["n_escape"] / n <= e < base + ost["n_escape"] / n + 0.002


@pytest.mark.parametrize("fmt", list(FMTS))
def test_fp8_corrupt_chunks(ez, orc, fmt):
    binding, cd = ez
    codec, ofmt, _ = FMTS[fmt]
    n, W = 20_000, 2
    x = synth.fp8_gaussian(n, 1.0 if fmt == "e5m2" else 16.0, fmt, seed=5).numpy()
    E0 = orc.fp8_stats(x, ofmt)["E0"]
    c, oslots, osizes, oslot = encode_compare(ez, orc, x, W, fmt, E0)
    recv, offs = orc.compact(oslots, osizes, oslot)
    nsm = 3 if fmt == "e5m2" else 4
    plane = ((c.L + 7) // 8 + 127) // 128 * 128       # chunk 0 holds L values
    idx0 = 128 + (nsm + 3) * plane                    # its escape index

    def put64(b, at, v):
        b[at:at + 8] = np.frombuffer(np.uint64(v).tobytes(), np.uint8)

    cases = {
        "magic": lambda b, o: b.__setitem__(0, ord("X")),
        "version": lambda b, o: b.__setitem__(4, 9),
        "format": lambda b, o: b.__setitem__(5, 3 - b[5]),
        "E0": lambda b, o: b.__setitem__(6, 40),
        "n_c": lambda b, o: b.__setitem__(8, b[8] ^ 1),
        "n_esc_big": lambda b, o: put64(b, 16, n + 5),
        "bytes": lambda b, o: b.__setitem__(24, b[24] ^ 128),
        "index": lambda b, o: b.__setitem__(idx0 + 8, b[idx0 + 8] ^ 1),
        "truncated": lambda b, o: o.__setitem__(2, o[2] - 128),
        "chunk_id": lambda b, o: b.__setitem__(32, 1),
    }
    for name, fn in cases.items():
        b = recv.copy()
        o = offs.copy()
        fn(b, o)
        _, want = orc.fp8_decode(b, o, n, W, ofmt)
        out = torch.zeros(n + 16, dtype=torch.uint8, device="cuda")
        c.clear_status()
        c.gather_decode(dev8(b), torch.from_numpy(o.astype(np.int64)).cuda(), out)
        torch.cuda.synchronize()
        got = c.status_word()
        assert want != 0, name
        assert got == want, (name, got, want)


def test_fp8_bad_window_base_is_reported(ez):
    binding, cd = ez
    c = cd.Fp8Codec(1000, 1, FMTS["e4m3"][0])
    x = torch.zeros(1008, dtype=torch.uint8, device="cuda")
    binding.ez_fp8_encode(c.plan, x, 0, 1, stats_record(binding, 10), c.out, c.out.numel(), c.sizes,
                          c.status, c.ws, c.ws_bytes)
    torch.cuda.synchronize()
    assert c.status_word() & binding.DSTAT_BAD_STATS
