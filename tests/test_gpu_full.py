"""Full-size GPU checks on the workloads the benchmark and the configs name.

* The benchmark workload (2^26 values, W = 8, B = 256, exponent flips at
  c = 0.003 per iteration): every payload byte against the oracle, for the raw
  and the 3-bit-coded reuse codec.
* Config 3 (OLMoE-shaped layer set, 522,588,160 values, W = 1): all payload
  bytes against the oracle at B = 256; for every B in 64..1024 the lossless
  round trip and the payload size from changed-block counts taken with torch.
* Config 4 (DeepSeek-MoE-16B-shaped layers, 587,862,016 values): W in
  {4, 8, 16, 32}, B = 128, round trip and sizes; W = 32 byte-compared.
* Config 5 (2^30 values, 20 iterations, reuse + 3-bit coding, W = 8): round
  trip every iteration; shards 0 and 7 byte-compared with the oracle at
  iterations 1 and 11.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import assert_stats_equal, host16, slots_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ez():
    from lossless_bf16_exponent_codec_gb300 import build
    build.build()
    from lossless_bf16_exponent_codec_gb300 import binding, codec
    return binding, codec


def cdiv(a, b):
    return -(-a // b)


def rup(a, b):
    return cdiv(a, b) * b


def changed_blocks(x0: torch.Tensor, x1: torch.Tensor, n: int, W: int, L: int, B: int):
    """(n_changed, m) per shard from torch (independent of both codecs)."""
    e0 = (x0.to(torch.int32) >> 7) & 0xFF
    e1 = (x1.to(torch.int32) >> 7) & 0xFF
    diff = (e0 != e1)
    res = []
    for r in range(W):
        a = min(r * L, n)
        b = min(a + L, n)
        d = diff[a:b]
        ns = b - a
        nb = cdiv(ns, B)
        pad = torch.zeros(nb * B, dtype=torch.bool, device=d.device)
        pad[:ns] = d
        blk = pad.view(nb, B).any(1)
        nc = int(blk.sum().item())
        m = nc * B - ((nb * B - ns) if (nb and bool(blk[-1].item())) else 0)
        res.append((ns, nc, m))
    return res


def check_sizes(c, res, B):
    sizes = c.sizes.cpu().tolist()
    for r, (ns, nc, m) in enumerate(res):
        nb = cdiv(ns, B)
        raw = rup(64 + rup(cdiv(nb, 8), 16) + rup(ns, 16) + rup(8 * cdiv(ns, 8192), 16) + m, 128)
        assert sizes[r] == raw, (r, sizes[r], raw)


def reuse_codec(ez, n, W, B, coded):
    binding, codec = ez
    return codec.Codec(n, W, B, binding.EZ_CODEC_REUSE_CODE3 if coded else binding.EZ_CODEC_REUSE)


@pytest.mark.parametrize("coded", [False, True])
def test_bench_workload_bytes(ez, orc, coded):
    n, W, B = 1 << 26, 8, 256
    x0 = synth.config2(n, device="cuda")
    x1 = synth.scale_drift_bench(x0, 1)
    x2 = synth.scale_drift_bench(x1, 2)
    c = reuse_codec(ez, n, W, B, coded)
    o_send = np.zeros(n, np.uint8)
    for it, x in enumerate((x0, x1, x2)):
        c.encode_reuse(x, cold=(it == 0))
        c.gather_decode()
        torch.cuda.synchronize()
        assert c.status_word() == 0
        assert torch.equal(c.full[:n], x)
        xn = host16(x)
        oslots, osizes, slot, osts = orc.reuse_encode_all(xn, W, B, o_send, cold=(it == 0),
                                                         coded=coded)
        slots_equal(c.out.cpu().numpy(), c.sizes.cpu().numpy(), oslots, osizes, slot, W)
        if coded:
            for r in range(W):
                assert_stats_equal(c.stats_of(r), osts[r])
    assert np.array_equal(c.send_cache.cpu().numpy(), o_send)


def test_config3_block_sweep(ez, orc):
    n = 522588160
    x0 = synth.config3_base(device="cuda")
    assert x0.numel() == n
    x1 = synth.config3_step(x0)
    for B in (64, 128, 256, 512, 1024):
        c = reuse_codec(ez, n, 1, B, False)
        c.encode_reuse(x0, cold=True)
        c.gather_decode()
        c.encode_reuse(x1)
        c.gather_decode()
        torch.cuda.synchronize()
        assert c.status_word() == 0
        assert torch.equal(c.full[:n], x1)
        assert torch.equal(c.recv_cache[:n], ((x1.to(torch.int32) >> 7) & 0xFF).to(torch.uint8))
        check_sizes(c, changed_blocks(x0, x1, n, 1, c.L, B), B)
        if B == 256:
            send = ((host16(x0).astype(np.uint32) >> 7) & 0xFF).astype(np.uint8)
            oslots, osizes, slot, _ = orc.reuse_encode_all(host16(x1), 1, B, send)
            slots_equal(c.out.cpu().numpy(), c.sizes.cpu().numpy(), oslots, osizes, slot, 1)
        del c
        torch.cuda.empty_cache()


def test_config4_gather_widths(ez, orc):
    B = 128
    x0, x1 = synth.config4_layer(0, device="cuda")
    n = x0.numel()
    assert n == 587862016
    for W in (4, 8, 16, 32):
        c = reuse_codec(ez, n, W, B, False)
        c.encode_reuse(x0, cold=True)
        c.gather_decode()
        c.encode_reuse(x1)
        c.gather_decode()
        torch.cuda.synchronize()
        assert c.status_word() == 0
        assert torch.equal(c.full[:n], x1)
        check_sizes(c, changed_blocks(x0, x1, n, W, c.L, B), B)
        if W == 32:
            send = ((host16(x0).astype(np.uint32) >> 7) & 0xFF).astype(np.uint8)
            oslots, osizes, slot, _ = orc.reuse_encode_all(host16(x1), W, B, send)
            slots_equal(c.out.cpu().numpy(), c.sizes.cpu().numpy(), oslots, osizes, slot, W)
        del c
        torch.cuda.empty_cache()


def test_config5_twenty_iterations(ez, orc):
    n, W, B = 1 << 30, 8, 256
    c = reuse_codec(ez, n, W, B, True)
    x = synth.config5_base(device="cuda")
    c.encode_reuse(x, cold=True)
    c.gather_decode()
    torch.cuda.synchronize()
    assert c.status_word() == 0 and torch.equal(c.full[:n], x)
    L = c.L
    for t in range(1, 21):
        prev = x
        x = synth.config5_step(prev, t)
        if t in (1, 11):
            prev_e = ((host16(prev).astype(np.uint32) >> 7) & 0xFF).astype(np.uint8)
        c.encode_reuse(x)
        c.gather_decode()
        torch.cuda.synchronize()
        assert c.status_word() == 0, t
        assert torch.equal(c.full[:n], x), t
        if t in (1, 11):
            xn = host16(x)
            for r in (0, W - 1):
                send = prev_e[r * L:(r + 1) * L].copy()
                pay, st = orc.reuse_encode(xn[r * L:(r + 1) * L], B, r, send, coded=True)
                size = int(c.sizes[r].item())
                assert size == pay.size
                got = c.out[r * c.slot:r * c.slot + size].cpu().numpy()
                assert np.array_equal(got, pay), (t, r)
                assert_stats_equal(c.stats_of(r), st)
        del prev
