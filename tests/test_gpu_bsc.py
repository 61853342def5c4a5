"""The block change rate that drives the shard selection, read from the GPU
encoder's payload headers, equals the host count of changed blocks, and the
payload sizes equal the selection module's exact byte count."""
import numpy as np
import pytest
import torch

import synth
from lossless_bf16_exponent_codec_gb300 import bsc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ez():
    from lossless_bf16_exponent_codec_gb300 import build
    build.build()
    from lossless_bf16_exponent_codec_gb300 import binding, codec
    return binding, codec


@pytest.mark.parametrize("B", [64, 256, 1024])
def test_header_change_rate_matches_host(ez, B):
    binding, codec = ez
    n, W = (1 << 21) + 4099, 8
    x0 = synth.config2(n, device="cuda")
    x1 = synth.scale_drift_bench(x0, 1, rate=0.001)
    c = codec.Codec(n, W, B, binding.EZ_CODEC_REUSE)
    c.encode_reuse(x0, cold=True)
    c.encode_reuse(x1)
    torch.cuda.synchronize()
    assert c.status_word() == 0
    a = x0.cpu().numpy().view(np.uint16)
    b = x1.cpu().numpy().view(np.uint16)
    out = c.out.cpu().numpy()
    sizes = c.sizes.cpu().numpy()
    L = -(-n // W)
    L = -(-L // 128) * 128
    for r in range(W):
        lo, hi = r * L, min(n, (r + 1) * L)
        pay = out[r * c.slot:r * c.slot + int(sizes[r])]
        q_host = bsc.block_change_rate(a[lo:hi], b[lo:hi], B)
        assert bsc.change_rate_from_header(pay, hi - lo, B) == q_host
        nb = -(-(hi - lo) // B)
        n_changed = int(round(q_host * nb))
        d = np.zeros(nb * B, bool)
        d[:hi - lo] = ((a[lo:hi] ^ b[lo:hi]) & 0x7F80) != 0
        last = bool(d.reshape(nb, B)[-1].any())
        assert bsc.payload_bytes_exact(hi - lo, B, n_changed, last) == int(sizes[r])
