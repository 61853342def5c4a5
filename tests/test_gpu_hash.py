"""GPU parity of hash-based change detection (EZ_FLAG_HASH_CACHE): over cold
and warm iterations, with exponent flips and mantissa noise, every payload
equals the oracle's hash-mode payload and the exponent-compare payload of
the same history, the sender's hash cache equals the oracle's block hashes,
and the receivers decode the tensor."""
import numpy as np
import pytest
import torch

import synth
from gpu_util import dev16, host16, slots_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ez():
    from lossless_bf16_exponent_codec_gb300 import build
    build.build()
    from lossless_bf16_exponent_codec_gb300 import binding, codec
    return binding, codec


def _flip(rng, x, rate):
    y = x.copy()
    e = (y >> 7) & 0xFF
    pick = (rng.random(x.size) < rate) & (e > 1) & (e < 254)
    e2 = np.where(rng.random(x.size) < 0.5, e - 1, e + 1)
    y[pick] = (y[pick] & 0x807F) | (e2[pick].astype(np.uint16) << 7)
    return (y & 0xFF80) | rng.integers(0, 128, x.size).astype(np.uint16)


@pytest.mark.parametrize("coded", [False, True])
@pytest.mark.parametrize("B", [8, 16, 32, 64, 256, 1024])
@pytest.mark.parametrize("n,W", [(50_001, 3), ((1 << 20) + 77, 8), (16_384, 1), (1000, 4)])
def test_hash_mode_parity(ez, orc, coded, B, n, W):
    binding, codec = ez
    cid = binding.EZ_CODEC_REUSE_CODE3 if coded else binding.EZ_CODEC_REUSE
    ch = codec.Codec(n, W, B, cid, flags=binding.EZ_FLAG_HASH_CACHE)
    cd = codec.Codec(n, W, B, cid)
    L = ch.L
    hstride = 16 * (-(-L // B))
    assert ch.geom["send_cache_bytes"] == W * hstride
    o_hash = np.zeros(W * hstride // 8, np.uint64)
    rng = np.random.default_rng(n + B + W + coded)
    xs = [synth.config2(n, seed=12).numpy().view(np.uint16)]
    for rate in (0.0, 0.001, 0.02):
        xs.append(_flip(rng, xs[-1], rate))
    for it, x in enumerate(xs):
        cold = it == 0
        for c in (ch, cd):
            c.encode_reuse(dev16(x), cold=cold)
        torch.cuda.synchronize()
        assert ch.status_word() == 0 and cd.status_word() == 0
        oslots = np.zeros(W * ch.slot, np.uint8)
        osizes = np.zeros(W, np.uint64)
        for r in range(W):
            a, b = min(r * L, n), min((r + 1) * L, n)
            hc = o_hash[r * hstride // 8:(r + 1) * hstride // 8]
            pay, _ = orc.reuse_encode_hash(x[a:b], B, r, hc, cold=cold, coded=coded)
            oslots[r * ch.slot:r * ch.slot + pay.size] = pay
            osizes[r] = pay.size
        slots_equal(ch.out.cpu().numpy(), ch.sizes.cpu().numpy(), oslots, osizes, ch.slot, W)
        slots_equal(cd.out.cpu().numpy(), cd.sizes.cpu().numpy(), oslots, osizes, ch.slot, W)
        got = ch.send_cache.cpu().numpy()[:W * hstride].view(np.uint64)
        for r in range(W):
            nb_r = -(-max(0, min(L, n - r * L)) // B)
            s = r * hstride // 8
            assert np.array_equal(got[s:s + 2 * nb_r], o_hash[s:s + 2 * nb_r]), (it, r)
        ch.gather_decode()
        torch.cuda.synchronize()
        assert ch.status_word() == 0 and np.array_equal(host16(ch.full)[:n], x), it


def test_hash_mode_plan_checks(ez):
    binding, codec = ez
    E = binding.EzError
    for bb in (8, 16):   # every reuse block size has hash mode
        binding.ez_plan_destroy(binding.ez_plan_create(1000, 2, bb, binding.EZ_CODEC_REUSE,
                                                       binding.EZ_FLAG_HASH_CACHE))
    with pytest.raises(E) as ei:
        binding.ez_plan_create(1000, 2, 4, binding.EZ_CODEC_REUSE, binding.EZ_FLAG_HASH_CACHE)
    assert ei.value.status == binding.EZ_ERR_UNSUPPORTED
    with pytest.raises(E) as ei:
        binding.ez_plan_create(1000, 2, 0, binding.EZ_CODEC_FP8_E5M2, binding.EZ_FLAG_HASH_CACHE)
    assert ei.value.status == binding.EZ_ERR_ARG
    with pytest.raises(E) as ei:
        binding.ez_plan_create(1000, 2, 0, binding.EZ_CODEC_CODE3, binding.EZ_FLAG_HASH_CACHE)
    assert ei.value.status == binding.EZ_ERR_ARG
