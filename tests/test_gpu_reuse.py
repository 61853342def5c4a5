"""GPU parity of the exponent-reuse codec (a3 encode, a4 decode, a5 gather)
and of its 3-bit-coded variant, against the CPU oracle: payload bytes and
sizes, the sender and receiver caches, per-shard statistics and the decoded
tensor, over cold and warm iterations, every block size, ragged and empty
shards, and corrupted payloads."""
import numpy as np
import pytest
import torch

import synth
from gpu_util import assert_stats_equal, dev16, exps, host16, slots_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ez():
    from lossless_bf16_exponent_codec_gb300 import build
    build.build()
    from lossless_bf16_exponent_codec_gb300 import binding, codec
    return binding, codec


def codec_of(ez, n, W, B, coded):
    binding, codec = ez
    cid = binding.EZ_CODEC_REUSE_CODE3 if coded else binding.EZ_CODEC_REUSE
    return codec.Codec(n, W, B, cid)


def run_iterations(ez, orc, xs, W, B, coded, check_exchange=True, single=False):
    """Encode xs[0] cold, then each later tensor warm; decode each with the
    gather call; compare everything with the oracle at every step."""
    n = xs[0].size
    c = codec_of(ez, n, W, B, coded)
    o_send = np.zeros(n, np.uint8)
    o_recv = np.zeros(n, np.uint8)
    for it, x in enumerate(xs):
        cold = it == 0
        xd = dev16(x) if n else torch.zeros(8, dtype=torch.int16, device="cuda")
        c.encode_reuse(xd, cold=cold)
        torch.cuda.synchronize()
        assert c.status_word() == 0
        oslots, osizes, slot, osts = orc.reuse_encode_all(x, W, B, o_send, cold=cold, coded=coded)
        assert slot == c.slot
        slots_equal(c.out.cpu().numpy(), c.sizes.cpu().numpy(), oslots, osizes, slot, W)
        assert np.array_equal(c.send_cache.cpu().numpy()[:n], o_send)
        if coded:
            for r in range(W):
                if orc.shard_count(n, W, r):
                    assert_stats_equal(c.stats_of(r), osts[r])
        if single:
            L = c.L
            for r in range(W):
                nr = orc.shard_count(n, W, r)
                if nr == 0:
                    continue
                size = int(c.sizes[r].item())
                c.decode_reuse(c.out[r * c.slot:], size, r, c.recv_cache[r * L:],
                               c.full[r * L:])
            torch.cuda.synchronize()
        elif check_exchange and it % 2 == 1:
            recv, offs = c.exchange()
            c.gather_decode(recv, offs)
        else:
            c.gather_decode()
        torch.cuda.synchronize()
        assert c.status_word() == 0
        out = host16(c.full)[:n]
        assert np.array_equal(out, x), f"iteration {it}"
        o_out_recv = orc.compact(oslots, osizes, slot)
        od, ost = orc.gather_decode_reuse(o_out_recv[0], o_out_recv[1], n, W, B, o_recv)
        assert ost == 0 and np.array_equal(od, x)
        assert np.array_equal(c.recv_cache.cpu().numpy()[:n], o_recv)
    return c


@pytest.mark.parametrize("coded", [False, True])
@pytest.mark.parametrize("variant", ["literal", "1b"])
def test_config1(ez, orc, coded, variant):
    xs = [t.numpy().view(np.uint16) for t in synth.config1(iterations=3, variant=variant)]
    run_iterations(ez, orc, xs, 4, 256, coded)


def _flip_chain(n, c, iters, seed):
    x = synth.gaussian_bf16(n, 0.02, synth.key_of(seed, 0))
    out = [x]
    for t in range(iters):
        x = synth.flip_exponents(x, torch.tensor(c, dtype=torch.float64), synth.key_of(seed, 1 + t))
        out.append(x)
    return [t.numpy().view(np.uint16) for t in out]


@pytest.mark.parametrize("B", [8, 16, 32, 64, 128, 256, 512, 1024])
@pytest.mark.parametrize("coded", [False, True])
def test_block_sizes_ragged(ez, orc, B, coded):
    xs = _flip_chain(300007, 0.004, 2, 300 + B)
    run_iterations(ez, orc, xs, 3, B, coded)


@pytest.mark.parametrize("n,W,B", [(1, 1, 8), (100, 8, 8), (129, 4, 64), (8192, 1, 1024),
                                   (8193, 2, 1024), (70000, 32, 16), (16384 * 3 + 5, 5, 512)])
@pytest.mark.parametrize("coded", [False, True])
def test_edge_shapes(ez, orc, n, W, B, coded):
    rng = np.random.default_rng(n + W + B)
    x0 = rng.integers(0, 65536, n, dtype=np.uint32).astype(np.uint16)
    x1 = x0.copy()
    x1[rng.random(n) < 0.01] ^= 0x0080
    x2 = x1.copy()          # an iteration with nothing changed
    run_iterations(ez, orc, [x0, x1, x2], W, B, coded, single=(n % 2 == 0))


@pytest.mark.parametrize("B", [32, 256])
def test_coded_window_base_zero(ez, orc, B):
    """Values near zero (exponent fields 0..3): the shard windows start at
    E0 = 0, the decoders' other code -> exponent step."""
    rng = np.random.default_rng(77 + B)
    n, W = 3 * 8192 + 777, 4
    x0 = ((rng.integers(0, 2, n) << 15) | (rng.integers(0, 4, n) << 7) | rng.integers(0, 128, n)).astype(np.uint16)
    x1 = x0.copy()
    x1[rng.random(n) < 0.01] ^= 0x0080
    L = orc.shard_count(n, W, 0)
    assert orc.stats(x1[:L])["E0"] == 0
    run_iterations(ez, orc, [x0, x1], W, B, True)


def test_empty_tensor(ez, orc):
    for coded in (False, True):
        c = codec_of(ez, 0, 4, 64, coded)
        z = torch.zeros(8, dtype=torch.int16, device="cuda")
        c.encode_reuse(z, cold=True)
        c.gather_decode()
        torch.cuda.synchronize()
        assert c.status_word() == 0
        assert c.sizes.cpu().tolist() == [128] * 4


def test_all_patterns_coded_and_raw(ez, orc):
    rng = np.random.default_rng(1)
    allp = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    xs = [rng.permutation(allp) for _ in range(3)]
    for coded in (False, True):
        for B in (8, 256):
            run_iterations(ez, orc, xs, 3, B, coded)


def _payload_cases(pay: np.ndarray):
    cases = [("magic", lambda b: b.__setitem__(0, b[0] ^ 1), None),
             ("version", lambda b: b.__setitem__(4, 1), None),
             ("shard", lambda b: b.__setitem__(12, 3), None),
             ("total", lambda b: b.__setitem__(48, b[48] ^ 0x80), None),
             ("bitmap", lambda b: b.__setitem__(64, b[64] ^ 1), None),
             ("n_changed", lambda b: b.__setitem__(24, b[24] + 1), None),
             ("truncated", lambda b: None, pay.size - 128)]
    return cases


@pytest.mark.parametrize("coded", [False, True])
def test_corrupt_payloads_are_reported(ez, orc, coded):
    binding, codec = ez
    rng = np.random.default_rng(31)
    n, B, W = 3000, 64, 1
    prev = rng.integers(0, 65536, n, dtype=np.uint32).astype(np.uint16)
    cur = prev.copy()
    cur[::97] ^= 0x0100
    send = exps(prev).copy()
    pay, _ = orc.reuse_encode(cur, B, 0, send, coded=coded)
    c = codec_of(ez, n, W, B, coded)
    for name, mut, avail in _payload_cases(pay):
        bad = pay.copy()
        mut(bad)
        av = bad.size if avail is None else avail
        _, ost = orc.reuse_decode(bad, n, B, 0, exps(prev).copy(), avail=av)
        recv = torch.zeros(bad.size + 256, dtype=torch.uint8, device="cuda")
        recv[:bad.size].copy_(torch.from_numpy(bad))
        offs = torch.tensor([0, av], dtype=torch.int64, device="cuda")
        c.recv_cache[:n].copy_(torch.from_numpy(exps(prev)))
        c.clear_status()
        c.gather_decode(recv, offs)
        torch.cuda.synchronize()
        g = c.status_word()
        assert ost != 0 and g != 0, name
        assert g & ost, (name, g, ost)
    # a payload offset that is not 16-byte aligned is refused on the device
    recv = torch.zeros(pay.size + 256, dtype=torch.uint8, device="cuda")
    offs = torch.tensor([8, 8 + pay.size], dtype=torch.int64, device="cuda")
    c.clear_status()
    c.gather_decode(recv, offs)
    torch.cuda.synchronize()
    assert c.status_word() & binding.DSTAT_MISALIGNED


def test_corrupt_code3_chunks_are_reported(ez, orc):
    binding, codec = ez
    rng = np.random.default_rng(41)
    x = (rng.normal(0, 0.02, 20000).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    slots, sizes, slot = orc.code3_encode(x, 2, orc.stats(x)["E0"])
    recv, offs = orc.compact(slots, sizes, slot)
    c = codec.Codec(x.size, 2)

    def gpu_status(buf, o):
        d = torch.zeros(buf.size + 256, dtype=torch.uint8, device="cuda")
        d[:buf.size].copy_(torch.from_numpy(buf))
        c.clear_status()
        c.gather_decode(d, torch.from_numpy(o.astype(np.int64)).cuda())
        torch.cuda.synchronize()
        return c.status_word()

    assert gpu_status(recv, offs) == 0
    for mut in (lambda b: b.__setitem__(0, 0), lambda b: b.__setitem__(32, 1),
                lambda b: b.__setitem__(16, b[16] + 1)):
        bad = recv.copy()
        mut(bad)
        ost = orc.code3_decode(bad, offs, x.size, 2)[1]
        g = gpu_status(bad, offs)
        assert ost and g and (g & ost), (g, ost)
    o2 = offs.copy()
    o2[1] -= 128
    ost = orc.code3_decode(recv, o2, x.size, 2)[1]
    g = gpu_status(recv, o2)
    assert ost and (g & ost)


def test_coded_reuse_histogram_window(ez, orc):
    """The coded reuse encode with EZ_FLAG_WINDOW_HIST: each shard's window
    from its own histogram; payloads, caches and statistics as the oracle's
    window mode 1, cold then warm."""
    binding, codec = ez
    rng = np.random.default_rng(4)
    n, W, B = 150_001, 4, 256
    v = (1.0 + rng.normal(0, 0.01, n // 2)).astype(np.float32).view(np.uint32)
    norms = ((v + 0x7FFF + ((v >> 16) & 1)) >> 16).astype(np.uint16)
    x0 = np.concatenate([norms, synth.config2(n - n // 2, seed=4).numpy().view(np.uint16)])
    x1 = synth.scale_drift_bench(torch.from_numpy(x0.view(np.int16)), 1).numpy().view(np.uint16)
    c = codec.Codec(n, W, B, binding.EZ_CODEC_REUSE_CODE3, flags=binding.EZ_FLAG_WINDOW_HIST)
    o_send = np.zeros(n, np.uint8)
    for it, x in enumerate((x0, x1)):
        c.encode_reuse(dev16(x), cold=it == 0)
        torch.cuda.synchronize()
        assert c.status_word() == 0
        oslots, osizes, slot, osts = orc.reuse_encode_all(x, W, B, o_send, cold=it == 0, coded=True,
                                                          window_mode=1)
        slots_equal(c.out.cpu().numpy(), c.sizes.cpu().numpy(), oslots, osizes, slot, W)
        assert np.array_equal(c.send_cache.cpu().numpy()[:n], o_send)
        for r in range(W):
            assert_stats_equal(c.stats_of(r), osts[r])
            assert osts[r]["rule"] == 1
        c.gather_decode()
        torch.cuda.synchronize()
        assert c.status_word() == 0 and np.array_equal(host16(c.full)[:n], x)
