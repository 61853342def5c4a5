"""Full-size GPU checks on the workloads the benchmark and the configs name.

Every payload byte, every size, the sender cache after each encode and the
receiver cache after each gather-decode are compared with the oracle, which
runs the same iterations beside the GPU (one single-threaded oracle call per
shard, shards on parallel host threads; the oracle's receiver decodes its own
payloads, which equal the GPU's byte for byte).

* The benchmark workload (2^26 values, W = 8, B = 256, exponent flips at
  c = 0.003 per iteration), raw and 3-bit-coded reuse, cold then two warm
  iterations.
* Config 3 (OLMoE-shaped layer set, 522,588,160 values, W = 1): every B in
  {64, 128, 256, 512, 1024}, the cold iteration and the clustered-flip step.
* Config 4 (DeepSeek-MoE-16B-shaped layers, 587,862,016 values, B = 128): all
  four layers at every W in {4, 8, 16, 32}, cold and warm.
* Config 5 (2^30 values, W = 8, B = 256, reuse + 3-bit coding): the cold
  iteration and all 20 drift iterations (0.08% then 0.4% flips), every shard,
  with each shard's statistics record.
"""
import os

import numpy as np
import pytest
import torch

import synth
from gpu_util import assert_stats_equal, host16

pytestmark = pytest.mark.gpu

THREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module")
def ez():
    from lossless_bf16_exponent_codec_gb300 import build
    build.build()
    from lossless_bf16_exponent_codec_gb300 import binding, codec
    return binding, codec


def reuse_codec(ez, n, W, B, coded):
    binding, codec = ez
    return codec.Codec(n, W, B, binding.EZ_CODEC_REUSE_CODE3 if coded else binding.EZ_CODEC_REUSE)


class Lockstep:
    """One plan run on the GPU and on the oracle side by side: the oracle's
    sender and receiver caches follow the GPU's iteration by iteration."""

    def __init__(self, orc, c, coded):
        self.orc, self.c, self.coded = orc, c, coded
        self.send = np.zeros(c.n, np.uint8)
        self.recv = np.zeros(c.n, np.uint8)

    def step(self, x: torch.Tensor, cold: bool, tag=""):
        orc, c, n, W, B = self.orc, self.c, self.c.n, self.c.W, self.c.B
        c.clear_status()
        c.encode_reuse(x, cold=cold)
        xh = host16(x)
        slots, sizes, slot, sts = orc.reuse_encode_all(xh, W, B, self.send, cold=cold,
                                                       coded=self.coded, threads=THREADS)
        torch.cuda.synchronize()
        assert c.status_word() == 0, tag
        gs = c.sizes.cpu().tolist()
        assert gs == [int(s) for s in sizes], (tag, "sizes")
        for r in range(W):
            k = gs[r]
            got = c.out[r * c.slot:r * c.slot + k].cpu().numpy()
            want = slots[r * slot:r * slot + k]
            if not np.array_equal(got, want):
                bad = np.nonzero(got != want)[0]
                raise AssertionError(f"{tag} payload {r}: {bad.size} bytes differ, first at {bad[:8]}")
            if self.coded:
                assert_stats_equal(c.stats_of(r), sts[r])
        assert np.array_equal(c.send_cache[:n].cpu().numpy(), self.send), (tag, "sender cache")
        # receiver: the GPU gather-decodes its own slots, the oracle its own
        c.gather_decode()
        out, ost = orc.reuse_decode_all(slots, sizes, slot, n, W, B, self.recv, threads=THREADS)
        torch.cuda.synchronize()
        assert ost == 0 and c.status_word() == 0, tag
        assert np.array_equal(out, xh), (tag, "oracle round trip")
        assert torch.equal(c.full[:n], x), (tag, "decoded values")
        assert np.array_equal(c.recv_cache[:n].cpu().numpy(), self.recv), (tag, "receiver cache")
        return [int(s) for s in sizes]


@pytest.mark.parametrize("coded", [False, True])
def test_bench_workload_bytes(ez, orc, coded):
    n, W, B = 1 << 26, 8, 256
    c = reuse_codec(ez, n, W, B, coded)
    run = Lockstep(orc, c, coded)
    x = synth.config2(n, device="cuda")
    run.step(x, True, "cold")
    for t in (1, 2):
        x = synth.scale_drift_bench(x, t)
        run.step(x, False, f"t={t}")


def test_config3_block_sweep(ez, orc):
    n = 522588160
    x0 = synth.config3_base(device="cuda")
    assert x0.numel() == n
    x1 = synth.config3_step(x0)
    for B in (64, 128, 256, 512, 1024):
        c = reuse_codec(ez, n, 1, B, False)
        run = Lockstep(orc, c, False)
        run.step(x0, True, f"B={B} cold")
        sizes = run.step(x1, False, f"B={B} warm")
        assert sizes[0] < 2 * n
        del c, run
        torch.cuda.empty_cache()


@pytest.mark.parametrize("layer", [0, 1, 2, 3])
def test_config4_gather_widths(ez, orc, layer):
    B = 128
    x0, x1 = synth.config4_layer(layer, device="cuda")
    n = x0.numel()
    assert n == 587862016
    for W in (4, 8, 16, 32):
        c = reuse_codec(ez, n, W, B, False)
        run = Lockstep(orc, c, False)
        run.step(x0, True, f"layer {layer} W={W} cold")
        run.step(x1, False, f"layer {layer} W={W} warm")
        del c, run
        torch.cuda.empty_cache()


def test_config5_twenty_iterations(ez, orc):
    n, W, B = 1 << 30, 8, 256
    c = reuse_codec(ez, n, W, B, True)
    run = Lockstep(orc, c, True)
    x = synth.config5_base(device="cuda")
    run.step(x, True, "cold")
    ratios = []
    for t in range(1, 21):
        x = synth.config5_step(x, t)
        sizes = run.step(x, False, f"t={t}")
        ratios.append(2 * n / sum(sizes))
    # the 0.4% iterations change more blocks than the 0.08% ones
    assert min(ratios[:10]) > max(ratios[10:])

