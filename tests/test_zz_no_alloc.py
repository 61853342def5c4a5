"""ez_encode_code3_noalloc: the code3 encode whose scratch is the library's
fixed device array instead of a caller workspace.

On the GPU it must give the same payload bytes, sizes and status as
ez_encode_code3 on the same input, for two calls in a row whose inputs
differ (the second call runs on scratch the first one left behind).  On the
host, plans whose encode scratch exceeds the array are rejected before any
CUDA call.  This file is collected last so that its first call may come
either in a fresh process or after every other test."""
import pytest
import torch

import synth


@pytest.fixture(scope="module")
def ez():
    from lossless_bf16_exponent_codec_gb300 import build
    build.build()
    from lossless_bf16_exponent_codec_gb300 import binding, codec
    return binding, codec


@pytest.mark.gpu
@pytest.mark.parametrize("n,W", [(200_003, 4), ((1 << 22) + 77, 8), (40_000, 1)])
def test_noalloc_matches_workspace_encode(ez, n, W):
    binding, codec = ez
    c = codec.Codec(n, W)
    x0 = synth.config2(n, device="cuda")
    x1 = synth.scale_drift_bench(x0, 1, rate=0.01)
    # expected: the workspace encoder, one input after the other
    ref = []
    for x in (x0, x1):
        c.stats(x)
        c.clear_status()
        c.out.zero_()
        c.encode_code3(x)
        torch.cuda.synchronize()
        assert c.status_word() == 0
        st = c.stats_buf[:binding.STATS_BYTES].clone()
        ref.append((c.out.clone(), c.sizes.clone(), st))
    # the no-alloc entry point: two calls in a row, no synchronisation between
    outs = [torch.zeros_like(c.out) for _ in ref]
    sizes = [torch.zeros_like(c.sizes) for _ in ref]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for (o_ref, s_ref, st), o, sz, x in zip(ref, outs, sizes, (x0, x1)):
        binding.ez_encode_code3_noalloc(c.plan, x, 0, W, st, o, o.numel(), sz, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for (o_ref, s_ref, _), o, sz in zip(ref, outs, sizes):
        assert torch.equal(sz, s_ref)
        for r in range(W):
            k = int(s_ref[r].item())
            assert torch.equal(o[r * c.slot:r * c.slot + k], o_ref[r * c.slot:r * c.slot + k])


@pytest.mark.gpu
def test_noalloc_chunk_subrange(ez):
    """Chunks [3, 5) of 8: the scratch holds per-chunk state for the encoded
    chunks only (indexed from `first`), so a sub-range must give the same
    bytes as the workspace encoder on the same sub-range, twice in a row."""
    binding, codec = ez
    n, W, first, count = (1 << 21) + 4099, 8, 3, 2
    c = codec.Codec(n, W)
    x = synth.config2(n, device="cuda")
    c.stats(x)
    sub = x[first * c.L:]
    c.out.zero_()
    binding.ez_encode_code3(c.plan, sub, first, count, c.stats_buf, c.out, c.out.numel(), c.sizes,
                            c.status, c.ws, c.ws_bytes)
    torch.cuda.synchronize()
    assert c.status_word() == 0
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        o = torch.zeros_like(c.out)
        sz = torch.zeros_like(c.sizes)
        binding.ez_encode_code3_noalloc(c.plan, sub, first, count, c.stats_buf, o, o.numel(), sz,
                                        status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(sz[:count], c.sizes[:count])
        for i in range(count):
            k = int(c.sizes[i].item())
            assert k > 0
            assert torch.equal(o[i * c.slot:i * c.slot + k], c.out[i * c.slot:i * c.slot + k])


def test_noalloc_rejects_oversized_plans(ez):
    """Sizes beyond EZ_NOALLOC_SCRATCH_BYTES give EZ_ERR_CAPACITY before any
    device work; the pointers below are aligned placeholders that are never
    dereferenced on that path (this test runs without a GPU)."""
    binding, _ = ez
    fake = 1 << 20
    for n, W in [(1 << 40, 8),          # 1 GiB of look-back state
                 (1 << 33, 1),          # one chunk of 2^33 values: 8 MiB
                 (1 << 20, 65536)]:     # per-chunk counters and records
        plan = binding.ez_plan_create(n, W, 0, binding.EZ_CODEC_CODE3)
        try:
            slot = binding.ez_plan_sizes(plan)["slot_bytes"]
            with pytest.raises(binding.EzError) as ei:
                binding.ez_encode_code3_noalloc(plan, fake, 0, W, fake, fake, slot * W, fake,
                                                fake, 0)
            assert ei.value.status == binding.EZ_ERR_CAPACITY
        finally:
            binding.ez_plan_destroy(plan)
    plan = binding.ez_plan_create(1000, 2, 0, binding.EZ_CODEC_CODE3)
    try:
        with pytest.raises(binding.EzError) as ei:
            binding.ez_encode_code3_noalloc(plan, fake, 0, 2, None, fake, 1 << 30, fake, fake, 0)
        assert ei.value.status == binding.EZ_ERR_ARG
    finally:
        binding.ez_plan_destroy(plan)
