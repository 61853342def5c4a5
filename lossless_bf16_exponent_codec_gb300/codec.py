"""Device buffers for one plan, and the calls of the hot path on them.

A thin convenience layer over the C ABI (binding.py): it allocates, with
torch, the buffers include/expzip.h asks the caller to own (workspace, slots,
size table, status word, caches, gathered output) and forwards each call.
"""
from __future__ import annotations

import torch

from . import binding as B


class Codec:
    def __init__(self, n: int, W: int, B_block: int = 0, codec: int = B.EZ_CODEC_CODE3,
                 device: str = "cuda", flags: int = 0):
        self.n, self.W, self.B, self.codec = n, W, B_block, codec
        self.device = torch.device(device)
        self.plan = B.ez_plan_create(n, W, B_block, codec, flags)
        self.geom = B.ez_plan_sizes(self.plan)
        self.L = self.geom["shard_len"]
        self.slot = self.geom["slot_bytes"]
        self.ws_bytes = self.geom["workspace_bytes"]
        dev = self.device
        self.ws = torch.zeros(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.stats_buf = torch.zeros(W * B.STATS_BYTES, dtype=torch.uint8, device=dev)
        self.out = torch.zeros(W * self.slot, dtype=torch.uint8, device=dev)
        self.sizes = torch.zeros(W, dtype=torch.int64, device=dev)
        self.slot_offsets = (torch.arange(W + 1, dtype=torch.int64) * self.slot).to(dev)
        self.full = torch.zeros(max(n, 1), dtype=torch.int16, device=dev)
        if codec != B.EZ_CODEC_CODE3:
            # exponent cache (1 byte per value) or, with EZ_FLAG_HASH_CACHE,
            # two u64 hashes per block
            self.send_cache = torch.zeros(max(self.geom["send_cache_bytes"], 16), dtype=torch.uint8,
                                          device=dev)
            self.recv_cache = torch.zeros(max(n, 8), dtype=torch.uint8, device=dev)

    def __del__(self):
        try:
            B.ez_plan_destroy(self.plan)
        except Exception:
            pass

    # a1
    def stats(self, x: torch.Tensor, n_values: int | None = None, stream=None) -> None:
        nv = x.numel() if n_values is None else n_values
        B.ez_stats(self.plan, x, nv, self.stats_buf, self.ws, self.ws_bytes, stream)

    # a2
    def encode_code3(self, x: torch.Tensor, first: int = 0, count: int | None = None,
                     stream=None) -> None:
        count = self.W - first if count is None else count
        B.ez_encode_code3(self.plan, x, first, count, self.stats_buf, self.out,
                          self.out.numel(), self.sizes, self.status, self.ws, self.ws_bytes,
                          stream)

    # a6
    def decode_code3(self, inp: torch.Tensor, offsets: torch.Tensor, first: int = 0,
                     count: int | None = None, out: torch.Tensor | None = None,
                     stream=None) -> torch.Tensor:
        count = self.W - first if count is None else count
        out = self.full if out is None else out
        B.ez_decode_code3(self.plan, inp, offsets, first, count, out, self.status, self.ws,
                          self.ws_bytes, stream)
        return out

    # a3
    def encode_reuse(self, x: torch.Tensor, cold: bool = False, first: int = 0,
                     count: int | None = None, cache: torch.Tensor | None = None,
                     with_stats: bool = True, stream=None) -> None:
        count = self.W - first if count is None else count
        cache = self.send_cache if cache is None else cache
        stats = self.stats_buf if (with_stats and self.codec == B.EZ_CODEC_REUSE_CODE3) else None
        B.ez_encode_reuse(self.plan, x, first, count, cache, cold, self.out, self.out.numel(),
                          self.sizes, stats, self.status, self.ws, self.ws_bytes, stream)

    # a4
    def decode_reuse(self, payload: torch.Tensor, payload_bytes: int, shard: int,
                     cache: torch.Tensor, out: torch.Tensor, stream=None) -> None:
        B.ez_decode_reuse(self.plan, payload, payload_bytes, shard, cache, out, self.status,
                          self.ws, self.ws_bytes, stream)

    # a5
    def gather_decode(self, recv: torch.Tensor | None = None, offsets: torch.Tensor | None = None,
                      cache: torch.Tensor | None = None, out: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
        recv = self.out if recv is None else recv
        offsets = self.slot_offsets if offsets is None else offsets
        out = self.full if out is None else out
        if self.codec != B.EZ_CODEC_CODE3:
            cache = self.recv_cache if cache is None else cache
        B.ez_gather_decode(self.plan, recv, offsets, cache, out, self.status, self.ws,
                           self.ws_bytes, stream)
        return out

    def exchange(self) -> tuple[torch.Tensor, torch.Tensor]:
        """The receive side of an allgather of variable-size payloads: read
        the size table, lay payload r at the exclusive prefix sum of the
        sizes (one device copy per payload, as the collective would)."""
        sizes = self.sizes.cpu().tolist()
        offs = [0]
        for s in sizes:
            offs.append(offs[-1] + s)
        recv = torch.zeros(max(offs[-1], 16), dtype=torch.uint8, device=self.device)
        for r, s in enumerate(sizes):
            recv[offs[r]:offs[r] + s].copy_(self.out[r * self.slot:r * self.slot + s])
        return recv, torch.tensor(offs, dtype=torch.int64, device=self.device)

    def stats_of(self, i: int = 0) -> dict:
        return B.parse_stats(self.stats_buf[i * B.STATS_BYTES:(i + 1) * B.STATS_BYTES])

    def status_word(self) -> int:
        return int(self.status.item())

    def clear_status(self) -> None:
        self.status.zero_()

    # zipcclReduceScatter, the local step
    def reduce_received(self, recv: torch.Tensor, offsets: torch.Tensor, me: int,
                        stream=None) -> torch.Tensor:
        """Decode the W code3 chunks this rank received in an all-to-all
        (chunk ``me`` of every source, back to back in source order at
        ``offsets``) and sum them in FP32 in source order, the decoder adding
        each chunk into the accumulator.  Returns the FP32 sums of chunk
        ``me``."""
        offs = offsets.cpu().tolist()
        n_me = max(0, min(self.L, self.n - me * self.L))
        acc = torch.zeros(max(self.L, 4), dtype=torch.float32, device=self.device)
        for s in range(self.W):
            one = torch.tensor([0, offs[s + 1] - offs[s]], dtype=torch.int64, device=self.device)
            B.ez_decode_code3_accumulate(self.plan, recv[offs[s]:], one, me, 1, acc, s == 0,
                                         self.status, self.ws, self.ws_bytes, stream)
        return acc[:n_me]


class Fp8Codec:
    """Buffers and calls of one FP8 plan (EZ_CODEC_FP8_E5M2 / _E4M3): the
    tensor is n FP8 values passed as their raw bytes (uint8)."""

    def __init__(self, n: int, W: int, codec: int = B.EZ_CODEC_FP8_E5M2, device: str = "cuda",
                 flags: int = 0):
        self.n, self.W, self.codec = n, W, codec
        self.device = torch.device(device)
        self.plan = B.ez_plan_create(n, W, 0, codec, flags)
        self.geom = B.ez_plan_sizes(self.plan)
        self.L = self.geom["shard_len"]
        self.slot = self.geom["slot_bytes"]
        self.ws_bytes = self.geom["workspace_bytes"]
        dev = self.device
        self.ws = torch.zeros(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.stats_buf = torch.zeros(B.FP8_STATS_BYTES, dtype=torch.uint8, device=dev)
        self.out = torch.zeros(W * self.slot, dtype=torch.uint8, device=dev)
        self.sizes = torch.zeros(W, dtype=torch.int64, device=dev)
        self.slot_offsets = (torch.arange(W + 1, dtype=torch.int64) * self.slot).to(dev)
        self.full = torch.zeros(max(n, 16), dtype=torch.uint8, device=dev)

    def __del__(self):
        try:
            B.ez_plan_destroy(self.plan)
        except Exception:
            pass

    def stats(self, x: torch.Tensor, n_values: int | None = None, stream=None) -> None:
        nv = x.numel() if n_values is None else n_values
        B.ez_fp8_stats(self.plan, x, nv, self.stats_buf, self.ws, self.ws_bytes, stream)

    def encode(self, x: torch.Tensor, first: int = 0, count: int | None = None, stream=None) -> None:
        count = self.W - first if count is None else count
        B.ez_fp8_encode(self.plan, x, first, count, self.stats_buf, self.out, self.out.numel(),
                        self.sizes, self.status, self.ws, self.ws_bytes, stream)

    def decode(self, inp: torch.Tensor, offsets: torch.Tensor, first: int = 0, count: int | None = None,
               out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        count = self.W - first if count is None else count
        out = self.full if out is None else out
        B.ez_fp8_decode(self.plan, inp, offsets, first, count, out, self.status, self.ws, self.ws_bytes,
                        stream)
        return out

    def gather_decode(self, recv: torch.Tensor | None = None, offsets: torch.Tensor | None = None,
                      out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        recv = self.out if recv is None else recv
        offsets = self.slot_offsets if offsets is None else offsets
        out = self.full if out is None else out
        B.ez_gather_decode(self.plan, recv, offsets, None, out, self.status, self.ws, self.ws_bytes, stream)
        return out

    def stats_of(self) -> dict:
        return B.parse_fp8_stats(self.stats_buf)

    def status_word(self) -> int:
        return int(self.status.item())

    def clear_status(self) -> None:
        self.status.zero_()
