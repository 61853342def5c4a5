"""Compressed all-to-all (Designs 1 and 2) and reduce-scatter (all-to-all
plus a local FP32 sum) across three gloo ranks on CPU, the oracle standing
in for the device codec: every rank gets chunk `rank` of every source back
bit for bit, the two designs move the same bytes, and the reduce-scatter
result equals the float32 sum of the sources' values in source order.
Plus the switcher's line fit and decision (closed forms)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from lossless_bf16_exponent_codec_gb300.dist import CollectiveSwitcher


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def worker(rank: int, world: int, port: int, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    try:
        dist.init_process_group("gloo", rank=rank, world_size=world)
        res = [_round(rank, world, n) for n in (50_001, 200)]   # 200: the last rank's chunk is empty
        q.put((rank,) + tuple(all(r[i] for r in res) for i in range(4)))
    except Exception as e:  # report, never hang the parent
        q.put((rank, repr(e), None, None, None))
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


def _round(rank, world, n):
    import oracle
    import synth
    from lossless_bf16_exponent_codec_gb300 import dist as zd
    xs = [synth.config2(n, seed=10 + s).numpy().view(np.uint16) for s in range(world)]
    L = oracle.shard_len(n, world)
    n_me = oracle.shard_count(n, world, rank)
    x = xs[rank]
    slots, sizes, slot = oracle.code3_encode(x, world, oracle.stats(x)["E0"])
    chunks = [torch.from_numpy(slots[j * slot:j * slot + int(sizes[j])].copy()) for j in range(world)]
    static = [zd.code3_static_bytes(oracle.shard_count(n, world, j)) for j in range(world)]
    got = {}
    for design in (1, 2):
        recv, offs = zd.alltoall_payloads(chunks, design=design,
                                          static_bytes=static if design == 2 else None)
        r, o = recv.numpy(), offs.tolist()
        dec = []
        ok = True
        for s in range(world):
            out, st = oracle.code3_decode_chunk(r[o[s]:o[s + 1]], n, world, rank)
            ok = ok and st == 0 and np.array_equal(out, xs[s][rank * L:rank * L + n_me])
            dec.append(torch.from_numpy(out.view(np.int16).copy()))
        got[design] = (ok, r[:o[-1]].copy(), dec)
    same = np.array_equal(got[1][1], got[2][1])
    summed = zd.reduce_decoded(got[1][2]).numpy()
    want = np.zeros(n_me, np.float32)
    for s in range(world):
        want = want + _f32(xs[s][rank * L:rank * L + n_me])
    rs_ok = np.array_equal(summed.view(np.uint32), want.view(np.uint32))
    return got[1][0], got[2][0], same, rs_ok


def test_alltoall_and_reduce_scatter_three_ranks():
    world = 3
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    ps = [ctx.Process(target=worker, args=(r, world, port, q)) for r in range(world)]
    for p in ps:
        p.start()
    res = [q.get(timeout=240) for _ in ps]
    for p in ps:
        p.join(timeout=60)
    for rank, d1, d2, same, rs in sorted(res, key=lambda t: t[0]):
        assert d1 is True, (rank, d1)
        assert d2 is True and same is True and rs is True, (rank, d2, same, rs)


def test_static_part_is_the_chunk_without_escapes(orc):
    from lossless_bf16_exponent_codec_gb300.dist import code3_static_bytes
    for n_c in (0, 1, 127, 128, 129, 8191, 8192, 8193, 70001, 1 << 20):
        assert code3_static_bytes(n_c) == orc.code3_chunk_bytes(n_c, 0)
        assert orc.code3_chunk_bytes(n_c, 1) == code3_static_bytes(n_c) + 128


def test_single_chunk_decode_equals_whole_decode(orc):
    import synth
    n, W = 30_000, 4
    x = synth.config2(n, seed=3).numpy().view(np.uint16)
    slots, sizes, slot = orc.code3_encode(x, W, orc.stats(x)["E0"])
    L = orc.shard_len(n, W)
    for c in range(W):
        out, st = orc.code3_decode_chunk(slots[c * slot:c * slot + int(sizes[c])], n, W, c)
        assert st == 0 and np.array_equal(out, x[c * L:c * L + orc.shard_count(n, W, c)])
    # a chunk presented under another index is refused by its header
    out, st = orc.code3_decode_chunk(slots[:int(sizes[0])], n, W, 1)
    assert st != 0


def test_switcher_fit_and_decision():
    rs = [(d, 20e-6 + d / 40e9) for d in (1e6, 4e6, 16e6, 64e6)]
    a2a = [(d, 35e-6 + d / 30e9) for d in (1e6, 4e6, 16e6)]
    sw = CollectiveSwitcher(rs, a2a)
    assert sw.a_rs == pytest.approx(20e-6) and sw.b_rs == pytest.approx(1 / 40e9)
    assert sw.a_a2a == pytest.approx(35e-6) and sw.b_a2a == pytest.approx(1 / 30e9)
    # T_A2A < T_RS  <=>  d (1/40e9 - e s / 30e9) > 15e-6
    e, s = 0.72, 0.5
    d_star = 15e-6 / (1 / 40e9 - e * s / 30e9)
    assert not sw.compress(0.9 * d_star, e, s)
    assert sw.compress(1.1 * d_star, e, s)
    # with BF16 on both paths (s = 1) and e = 0.72 the compressed path's slope
    # is 0.72/30e9 < 1/40e9 only barely; it needs a larger message
    d1 = 15e-6 / (1 / 40e9 - e / 30e9)
    assert d1 > d_star and sw.compress(1.01 * d1, e, 1.0) and not sw.compress(0.99 * d1, e, 1.0)
    with pytest.raises(ValueError):
        CollectiveSwitcher([(1, 1.0)], a2a)
