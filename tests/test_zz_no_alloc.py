"""ez_gather_decode_noalloc: the gather-decode whose scratch is the library's
fixed device array instead of a caller workspace.

On the GPU it must give the same decoded tensor, receiver cache and status as
ez_gather_decode on the same payloads, for two calls in a row whose inputs
differ (the second call runs on scratch the first one left behind).  On the
host, plans whose decode scratch exceeds the array are rejected before any
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


def payloads(c, xs, reuse):
    """Encode each tensor with the workspace entry points (the first one
    cold) and lay its payloads out as an allgather would deliver them."""
    out = []
    for it, x in enumerate(xs):
        if reuse:
            c.encode_reuse(x, cold=it == 0)
        else:
            c.stats(x)
            c.encode_code3(x)
        torch.cuda.synchronize()
        assert c.status_word() == 0
        out.append(c.exchange())
    return out


@pytest.mark.gpu
@pytest.mark.parametrize("codec_id", [1, 2, 3])
@pytest.mark.parametrize("n,W,B", [(200_003, 4, 64), ((1 << 22) + 77, 8, 256)])
def test_noalloc_matches_workspace_gather(ez, codec_id, n, W, B):
    binding, codec = ez
    reuse = codec_id != binding.EZ_CODEC_CODE3
    c = codec.Codec(n, W, B if reuse else 0, codec_id)
    x0 = synth.config2(n, device="cuda")
    x1 = synth.scale_drift_bench(x0, 1, rate=0.01)
    got = payloads(c, [x0, x1], reuse)

    def fresh():
        return torch.zeros(max(n, 8), dtype=torch.uint8, device="cuda") if reuse else None

    # expected: the workspace gather-decode, iteration by iteration
    ref_cache = fresh()
    ref_out = []
    for recv, offs in got:
        o = torch.full((n,), -1, dtype=torch.int16, device="cuda")
        c.clear_status()
        c.gather_decode(recv, offs, ref_cache, o)
        torch.cuda.synchronize()
        assert c.status_word() == 0
        ref_out.append(o)
    assert torch.equal(ref_out[0], x0) and torch.equal(ref_out[1], x1)

    # the no-alloc entry point: two calls in a row, no synchronisation between
    cache = fresh()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = [torch.full((n,), -1, dtype=torch.int16, device="cuda") for _ in got]
    for (recv, offs), o in zip(got, outs):
        binding.ez_gather_decode_noalloc(c.plan, recv, offs, cache, o, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for o, r in zip(outs, ref_out):
        assert torch.equal(o, r)
    if reuse:
        assert torch.equal(cache, ref_cache)


def test_noalloc_rejects_oversized_plans(ez):
    """Sizes beyond EZ_NOALLOC_SCRATCH_BYTES give EZ_ERR_CAPACITY before any
    device work; the pointers below are aligned placeholders that are never
    dereferenced on that path (this test runs without a GPU)."""
    binding, _ = ez
    fake = 1 << 20
    for n, W, B, cid in [(1 << 40, 8, 0, 1),            # 1 GiB of look-back state
                         (1 << 31, 8, 256, 2),          # two 2 MiB state arrays
                         (1 << 20, 65536, 64, 3)]:      # per-shard records
        plan = binding.ez_plan_create(n, W, B, cid)
        try:
            with pytest.raises(binding.EzError) as ei:
                binding.ez_gather_decode_noalloc(plan, fake, fake, fake, fake, fake, 0)
            assert ei.value.status == binding.EZ_ERR_CAPACITY
        finally:
            binding.ez_plan_destroy(plan)
    plan = binding.ez_plan_create(1000, 2, 0, 1)
    try:
        with pytest.raises(binding.EzError) as ei:
            binding.ez_gather_decode_noalloc(plan, None, fake, None, fake, fake, 0)
        assert ei.value.status == binding.EZ_ERR_ARG
    finally:
        binding.ez_plan_destroy(plan)
