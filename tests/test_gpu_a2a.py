"""The device side of the compressed reduce-scatter on one GPU, W sources
emulated: each source's code3 encode, the receiver's decode of chunk `j` of
every source (one chunk per call) and the FP32 accumulate kernel give the
float32 sum of the sources' values in source order, bit for bit; and the
accumulate kernel alone matches numpy's float32 additions on every BF16
pattern."""
import numpy as np
import pytest
import torch

import synth
from gpu_util import dev16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ez():
    from lossless_bf16_exponent_codec_gb300 import build
    build.build()
    from lossless_bf16_exponent_codec_gb300 import binding, codec
    return binding, codec


def _f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("n,W", [((1 << 20) + 777, 4), (40_000, 3), (8192 * 3, 8)])
def test_reduce_scatter_local_step(ez, n, W):
    binding, codec = ez
    xs = [synth.config2(n, seed=20 + s, device="cuda") for s in range(W)]
    chunks = []
    for x in xs:
        c = codec.Codec(n, W)
        c.stats(x)
        c.encode_code3(x)
        torch.cuda.synchronize()
        assert c.status_word() == 0
        sizes = c.sizes.cpu().tolist()
        chunks.append([c.out[j * c.slot:j * c.slot + sizes[j]].clone() for j in range(W)])
    rx = codec.Codec(n, W)
    L = rx.L
    host = [x.cpu().numpy().view(np.uint16) for x in xs]
    for j in range(W):
        n_j = max(0, min(L, n - j * L))
        recv = torch.cat([chunks[s][j] for s in range(W)])
        offs = [0]
        for s in range(W):
            offs.append(offs[-1] + chunks[s][j].numel())
        acc = rx.reduce_received(recv, torch.tensor(offs, dtype=torch.int64), j)
        torch.cuda.synchronize()
        assert rx.status_word() == 0
        want = np.zeros(n_j, np.float32)
        for s in range(W):
            want = want + _f32(host[s][j * L:j * L + n_j])
        assert np.array_equal(acc.cpu().numpy().view(np.uint32), want.view(np.uint32)), j


@pytest.mark.parametrize("n,W", [((1 << 20) + 777, 4), (5_003, 2)])
def test_fused_decode_accumulate_equals_two_kernels(ez, n, W):
    """ez_decode_code3_accumulate gives the bits of ez_decode_code3 followed
    by ez_accumulate_bf16, for every chunk (ragged last chunks included)."""
    binding, codec = ez
    xs = [synth.config2(n, seed=40 + s, device="cuda") for s in range(3)]
    c = codec.Codec(n, W)
    L = c.L
    for j in range(W):
        n_j = max(0, min(L, n - j * L))
        fused = torch.zeros(max(L, 4), dtype=torch.float32, device="cuda")
        two = torch.zeros(max(L, 4), dtype=torch.float32, device="cuda")
        tmp = torch.zeros(max(L, 8), dtype=torch.int16, device="cuda")
        for s, x in enumerate(xs):
            c.stats(x)
            c.encode_code3(x)
            size = int(c.sizes[j].item())
            chunk = c.out[j * c.slot:j * c.slot + size].clone()
            one = torch.tensor([0, size], dtype=torch.int64, device="cuda")
            binding.ez_decode_code3_accumulate(c.plan, chunk, one, j, 1, fused, s == 0, c.status,
                                               c.ws, c.ws_bytes)
            binding.ez_decode_code3(c.plan, chunk, one, j, 1, tmp, c.status, c.ws, c.ws_bytes)
            binding.ez_accumulate_bf16(two, tmp, n_j, s == 0)
        torch.cuda.synchronize()
        assert c.status_word() == 0
        assert torch.equal(fused[:n_j].view(torch.int32), two[:n_j].view(torch.int32)), j


def test_accumulate_kernel_all_patterns(ez):
    binding, codec = ez
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    rng = np.random.default_rng(5)
    a = pats[rng.permutation(65536)]
    b = pats[rng.permutation(65536)]
    for n in (65536, 65531, 7, 1):
        xa, xb = dev16(a[:n]), dev16(b[:n])
        acc = torch.zeros(max(n, 4), dtype=torch.float32, device="cuda")
        binding.ez_accumulate_bf16(acc, xa, n, True)
        binding.ez_accumulate_bf16(acc, xb, n, False)
        torch.cuda.synchronize()
        with np.errstate(invalid="ignore", over="ignore"):
            want = (np.float32(0) + _f32(a[:n])) + _f32(b[:n])
        got = acc[:n].cpu().numpy()
        nan = np.isnan(want)
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32)), n


def test_accumulate_argument_checks(ez):
    binding, codec = ez
    acc = torch.zeros(64, dtype=torch.float32, device="cuda")
    x = torch.zeros(64, dtype=torch.int16, device="cuda")
    binding.ez_accumulate_bf16(acc, x, 0, True)           # n = 0: nothing to do
    with pytest.raises(binding.EzError):
        binding.ez_accumulate_bf16(acc[1:], x, 8, True)   # misaligned accumulator
    with pytest.raises(binding.EzError):
        binding.ez_accumulate_bf16(acc, x[1:], 8, True)   # misaligned input


def test_device_collectives_one_rank_nccl(ez):
    """The full device path (encode, NCCL all-to-all of one rank, decode or
    FP32 sum) on a one-rank process group: the all-to-all returns the
    tensor, the reduce-scatter its float32 values."""
    import os
    import socket
    import torch.distributed as dist
    from lossless_bf16_exponent_codec_gb300 import dist as zd
    binding, codec = ez
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        n = 300_001
        x = synth.config2(n, seed=31, device="cuda")
        xh = x.cpu().numpy().view(np.uint16)
        for design in (1, 2):
            c = codec.Codec(n, 1)
            out = zd.alltoall_code3(c, x, design=design)
            assert torch.equal(out[:n], x)
            c = codec.Codec(n, 1)
            acc = zd.reduce_scatter_code3(c, x, design=design)
            want = np.float32(0) + _f32(xh)
            assert np.array_equal(acc.cpu().numpy().view(np.uint32), want.view(np.uint32))
    finally:
        dist.destroy_process_group()


def test_fused_decode_leaves_sums_of_a_bad_chunk_untouched(ez):
    """A chunk that fails its header checks adds nothing and is reported."""
    binding, codec = ez
    n, W = 40_000, 2
    x = synth.config2(n, seed=50, device="cuda")
    c = codec.Codec(n, W)
    c.stats(x)
    c.encode_code3(x)
    size = int(c.sizes[1].item())
    chunk = c.out[c.slot:c.slot + size].clone()
    chunk[0] ^= 0xFF                                   # magic broken
    one = torch.tensor([0, size], dtype=torch.int64, device="cuda")
    acc = torch.full((c.L,), 3.5, dtype=torch.float32, device="cuda")
    c.clear_status()
    binding.ez_decode_code3_accumulate(c.plan, chunk, one, 1, 1, acc, False, c.status, c.ws, c.ws_bytes)
    torch.cuda.synchronize()
    assert c.status_word() & binding.DSTAT_BAD_HEADER
    assert torch.all(acc == 3.5)
