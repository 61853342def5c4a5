"""Concurrency and repetition on the GPU.

The encoders launch their later kernels as programmatic dependent launches
(each waits for the kernels before it in its stream); two codecs driven on two
CUDA streams at once must give exactly what they give alone.  Repeated cold
and warm reuse encodes of the same tensors must give the same payload bytes
every time (a race inside a kernel shows up as a payload that changes between
repetitions or a decode that differs from the input)."""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ez():
    from lossless_bf16_exponent_codec_gb300 import build
    build.build()
    from lossless_bf16_exponent_codec_gb300 import binding, codec
    return binding, codec


def _run_all(ez, x0, x1, n, W, B, stream=None):
    """code3 encode + gather decode, then raw and coded reuse encodes of x0
    (cold) and x1 (warm) with their gather decodes, all on `stream`; returns
    every payload slot array, size table, decoded tensor and status word."""
    binding, codec = ez
    out = {}
    ctx = torch.cuda.stream(stream) if stream is not None else torch.cuda.stream(torch.cuda.current_stream())
    with ctx:
        c3 = codec.Codec(n, W)
        s = torch.cuda.current_stream()
        c3.stats(x1, stream=s)
        c3.encode_code3(x1, stream=s)
        c3.gather_decode(stream=s)
        out["c3"] = c3
        for name, cid in (("raw", binding.EZ_CODEC_REUSE), ("coded", binding.EZ_CODEC_REUSE_CODE3)):
            c = codec.Codec(n, W, B, cid)
            c.encode_reuse(x0, cold=True, stream=s)
            c.gather_decode(stream=s)
            c.encode_reuse(x1, stream=s)
            c.gather_decode(stream=s)
            out[name] = c
    return out


def _snapshot(res, n):
    return {k: (c.out.clone(), c.sizes.clone(), c.full[:n].clone(), c.status_word()) for k, c in res.items()}


def test_two_streams_match_one(ez):
    n, W, B = (1 << 22) + 333, 8, 256
    x0 = synth.config2(n, device="cuda")
    x1 = synth.scale_drift_bench(x0, 1)
    y0 = synth.config2(n, seed=9, device="cuda")
    y1 = synth.scale_drift_bench(y0, 1)
    ref_x = _snapshot(_run_all(ez, x0, x1, n, W, B), n)
    ref_y = _snapshot(_run_all(ez, y0, y1, n, W, B), n)
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    res_x = _run_all(ez, x0, x1, n, W, B, stream=sa)
    res_y = _run_all(ez, y0, y1, n, W, B, stream=sb)
    torch.cuda.synchronize()
    for ref, res, want in ((ref_x, res_x, x1), (ref_y, res_y, y1)):
        got = _snapshot(res, n)
        for k in ref:
            out_r, sz_r, full_r, st_r = ref[k]
            out_g, sz_g, full_g, st_g = got[k]
            assert st_r == 0 and st_g == 0, k
            assert torch.equal(sz_r, sz_g), k
            assert torch.equal(full_g, want), k
            slot = res[k].slot
            for r in range(W):
                m = int(sz_r[r].item())
                assert torch.equal(out_r[r * slot:r * slot + m], out_g[r * slot:r * slot + m]), (k, r)


@pytest.mark.parametrize("coded", [False, True])
def test_repeated_encodes_are_identical(ez, coded):
    binding, codec = ez
    n, W, B = (1 << 23) + 77, 8, 256
    x0 = synth.config2(n, device="cuda")
    x1 = synth.scale_drift_bench(x0, 1)
    cid = binding.EZ_CODEC_REUSE_CODE3 if coded else binding.EZ_CODEC_REUSE
    first = None
    for rep in range(6):
        c = codec.Codec(n, W, B, cid)
        c.encode_reuse(x0, cold=True)
        c.gather_decode()
        c.encode_reuse(x1)
        c.gather_decode()
        torch.cuda.synchronize()
        assert c.status_word() == 0, rep
        assert torch.equal(c.full[:n], x1), rep
        sizes = c.sizes.clone()
        pay = [c.out[r * c.slot:r * c.slot + int(sizes[r].item())].clone() for r in range(W)]
        if first is None:
            first = (sizes, pay)
        else:
            assert torch.equal(first[0], sizes), rep
            for r in range(W):
                assert torch.equal(first[1][r], pay[r]), (rep, r)
        del c
