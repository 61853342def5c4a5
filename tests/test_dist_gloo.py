"""The multi-rank path on CPU: two gloo ranks, each encoding its own shard
(the CPU oracle stands in for the device encoder), exchange sizes and
payloads with dist.allgather_payloads (ZipCCL 3.2: all-gather sizes, then
blocks) and decode all of them; both ranks must get the whole tensor back
bit for bit, for the code3 and the reuse codecs.  Also the benchmark's
multi-rank helpers (barrier, max over ranks) under gloo."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def worker(rank: int, world: int, port: int, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    try:
        dist.init_process_group("gloo", rank=rank, world_size=world)
        import oracle
        import synth
        from lossless_bf16_exponent_codec_gb300.dist import allgather_payloads
        n = 70_001
        x = synth.config2(n, seed=7).numpy().view(np.uint16)
        L = oracle.shard_len(n, world)
        # code3: this rank's chunk, window from the whole tensor's statistics
        E0 = oracle.stats(x)["E0"]
        slots, sizes, slot = oracle.code3_encode(x, world, E0)
        mine = torch.from_numpy(slots[rank * slot:rank * slot + int(sizes[rank])].copy())
        recv, offs = allgather_payloads(mine)
        out, st = oracle.code3_decode(recv.numpy(), offs.numpy().astype(np.uint64), n, world)
        ok3 = st == 0 and np.array_equal(out, x)
        # reuse (cold, B = 64): this rank's shard and its sender cache
        a, b = rank * L, min((rank + 1) * L, n)
        send = np.zeros(max(b - a, 1), np.uint8)
        pay, _ = oracle.reuse_encode(x[a:b], 64, rank, send, cold=True)
        recv, offs = allgather_payloads(torch.from_numpy(pay.copy()))
        cache = np.zeros(n, np.uint8)
        out, st = oracle.gather_decode_reuse(recv.numpy(), offs.numpy().astype(np.uint64), n,
                                             world, 64, cache)
        okr = st == 0 and np.array_equal(out, x)
        # the benchmark's helpers
        import bench
        bench.barrier(world)
        mx = bench.reduce_max(world, float(rank + 1))
        q.put((rank, ok3, okr, mx))
    except Exception as e:  # report, never hang the parent
        q.put((rank, repr(e), None, None))
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


def test_two_gloo_ranks_exchange_and_decode():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        r, ok3, okr, mx = q.get(timeout=240)
        res[r] = (ok3, okr, mx)
    for p in procs:
        p.join(timeout=60)
    for r in range(world):
        ok3, okr, mx = res[r]
        assert ok3 is True, res
        assert okr is True, res
        assert mx == float(world)
