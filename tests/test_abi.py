"""The C-ABI library loads, exports every entry point include/expzip.h
declares, and rejects bad host-side arguments before touching a GPU.  Its
geometry (shard length, worst-case slot sizes) is checked against the
oracle's own formulas.  No compute call is made here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    from lossless_bf16_exponent_codec_gb300 import build
    build.build()
    from lossless_bf16_exponent_codec_gb300 import binding
    return binding


def declared_entry_points():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        with open(os.path.join(ROOT, "include", h)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(ez_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(B):
    names = declared_entry_points()
    assert len(names) >= 11
    lib = ctypes.CDLL(B.LIB_PATH)
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(B.ENTRY_POINTS)


def test_plan_validation(B):
    E = B.EzError
    for bad in [dict(n=10, W=0), dict(n=1 << 41, W=1), dict(n=10, W=70000),
                dict(n=10, W=1, codec=9), dict(n=10, W=1, flags=2),
                dict(n=10, W=1, flags=B.EZ_FLAG_WINDOW_HIST | 4),
                dict(n=10, W=1, codec=B.EZ_CODEC_REUSE, B=0)]:
        with pytest.raises(E) as ei:
            B.ez_plan_create(**bad)
        assert ei.value.status == B.EZ_ERR_ARG
    B.ez_plan_destroy(B.ez_plan_create(10, 1, 0, B.EZ_CODEC_CODE3, B.EZ_FLAG_WINDOW_HIST))
    for bb in (4, 12, 2048):
        with pytest.raises(E) as ei:
            B.ez_plan_create(1000, 2, bb, B.EZ_CODEC_REUSE)
        assert ei.value.status == B.EZ_ERR_UNSUPPORTED
    assert B.ez_version() == 0x000300
    for codec in (B.EZ_CODEC_FP8_E5M2, B.EZ_CODEC_FP8_E4M3):
        with pytest.raises(E) as ei:
            B.ez_plan_create(10, 1, 0, codec, B.EZ_FLAG_HASH_CACHE)
        assert ei.value.status == B.EZ_ERR_ARG
        B.ez_plan_destroy(B.ez_plan_create(10, 1, 0, codec, B.EZ_FLAG_WINDOW_HIST))
    assert B.status_str(0) == "ok"


@pytest.mark.parametrize("n,W", [(0, 1), (1, 1), (1000, 3), (1 << 20, 4), (1 << 26, 8),
                                 (587862016, 32), (1 << 30, 8), (100, 8)])
def test_geometry_matches_oracle(B, orc, n, W):
    p = B.ez_plan_create(n, W, 0, B.EZ_CODEC_CODE3)
    s = B.ez_plan_sizes(p)
    assert s["shard_len"] == orc.shard_len(n, W)
    assert s["slot_bytes"] == orc.code3_slot_bytes(n, W)
    assert s["cache_bytes"] == 0 and s["workspace_bytes"] % 256 == 0
    B.ez_plan_destroy(p)
    for bb in (8, 64, 256, 1024):
        for codec, coded in ((B.EZ_CODEC_REUSE, False), (B.EZ_CODEC_REUSE_CODE3, True)):
            p = B.ez_plan_create(n, W, bb, codec)
            s = B.ez_plan_sizes(p)
            assert s["slot_bytes"] == orc.reuse_slot_bytes(n, W, bb, coded)
            assert s["cache_bytes"] == n
            B.ez_plan_destroy(p)
    for codec, fmt in ((B.EZ_CODEC_FP8_E5M2, orc.FP8_E5M2), (B.EZ_CODEC_FP8_E4M3, orc.FP8_E4M3)):
        p = B.ez_plan_create(n, W, 0, codec)
        s = B.ez_plan_sizes(p)
        L = orc.shard_len(n, W)
        assert s["shard_len"] == L
        assert s["slot_bytes"] == orc.fp8_chunk_bytes(L, L, fmt)
        assert s["cache_bytes"] == 0 and s["send_cache_bytes"] == 0
        B.ez_plan_destroy(p)


def test_host_argument_checks_need_no_gpu(B):
    """NULL, misaligned, short workspace and bad ranges are refused on the
    host; none of these reaches the CUDA runtime."""
    p = B.ez_plan_create(1 << 16, 4, 0, B.EZ_CODEC_CODE3)
    s = B.ez_plan_sizes(p)
    ws, good = 1 << 20, 1 << 24       # fake, 256-aligned addresses never dereferenced
    E = B.EzError

    def rc(fn, *a):
        try:
            fn(*a)
        except E as e:
            return e.status
        return 0

    assert rc(B.ez_stats, p, good, 100, None, ws, s["workspace_bytes"], 0) == B.EZ_ERR_ARG
    assert rc(B.ez_stats, p, good + 2, 100, good, ws, s["workspace_bytes"], 0) == B.EZ_ERR_ARG
    assert rc(B.ez_stats, p, good, 100, good, ws + 16, s["workspace_bytes"], 0) == B.EZ_ERR_ARG
    assert rc(B.ez_stats, p, good, 100, good, ws, s["workspace_bytes"] - 1, 0) == B.EZ_ERR_CAPACITY
    assert rc(B.ez_encode_code3, p, good, 0, 5, good, good, 1 << 30, good, good, ws,
              s["workspace_bytes"], 0) == B.EZ_ERR_ARG          # range past W
    assert rc(B.ez_encode_code3, p, good, 0, 4, good, good, s["slot_bytes"] * 4 - 1, good, good,
              ws, s["workspace_bytes"], 0) == B.EZ_ERR_CAPACITY
    assert rc(B.ez_decode_code3, p, good, good + 4, 0, 4, good, good, ws,
              s["workspace_bytes"], 0) == B.EZ_ERR_ARG          # offsets misaligned
    assert rc(B.ez_encode_reuse, p, good, 0, 1, good, 0, good, 1 << 30, good, None, good, ws,
              s["workspace_bytes"], 0) == B.EZ_ERR_ARG          # code3 plan
    assert rc(B.ez_gather_decode, p, None, good, None, good, good, ws,
              s["workspace_bytes"], 0) == B.EZ_ERR_ARG
    B.ez_plan_destroy(p)
    q = B.ez_plan_create(1 << 16, 4, 64, B.EZ_CODEC_REUSE)
    sq = B.ez_plan_sizes(q)
    assert rc(B.ez_decode_reuse, q, good, 4096, 4, good, good, good, ws,
              sq["workspace_bytes"], 0) == B.EZ_ERR_ARG         # shard >= W
    assert rc(B.ez_gather_decode, q, good, good, None, good, good, ws,
              sq["workspace_bytes"], 0) == B.EZ_ERR_ARG         # reuse needs a cache
    assert rc(B.ez_encode_code3, q, good, 0, 1, good, good, 1 << 30, good, good, ws,
              sq["workspace_bytes"], 0) == B.EZ_ERR_ARG         # reuse plan
    B.ez_plan_destroy(q)
