"""The exchange step of a compressed all-gather across ranks.

ZipCCL research digest 3.2 (zipcclAllGather): each rank compresses its own
chunk, the ranks all-gather the compressed sizes, then all-gather the
compressed blocks, and every rank decompresses all of them.  The codec calls
(encode on the rank's shard, gather-decode of the W payloads) are the
library's; this module only moves the bytes with torch.distributed, so it
runs over NCCL for device tensors and over gloo for host tensors alike.

Payload sizes are multiples of 128 bytes, so laying the received payloads
back to back keeps every offset 16-byte aligned, as the decoders require.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def allgather_sizes(nbytes: int, device, group=None) -> list[int]:
    """Every rank's payload size (the first all-gather of 3.2)."""
    world = dist.get_world_size(group)
    mine = torch.tensor([nbytes], dtype=torch.int64, device=device)
    sizes = [torch.zeros(1, dtype=torch.int64, device=device) for _ in range(world)]
    dist.all_gather(sizes, mine, group=group)
    return [int(s.item()) for s in sizes]


def allgather_payloads(payload: torch.Tensor, group=None) -> tuple[torch.Tensor, torch.Tensor]:
    """All-gather variable-size uint8 payloads (one per rank).

    Returns the received bytes laid out back to back in rank order and the
    W+1 int64 offsets the gather-decode takes (on the payload's device)."""
    if payload.dtype != torch.uint8 or payload.dim() != 1:
        raise ValueError("payload must be a 1-D uint8 tensor")
    device = payload.device
    sizes = allgather_sizes(payload.numel(), device, group)
    if any(s % 128 for s in sizes):
        raise ValueError(f"payload sizes must be multiples of 128 bytes: {sizes}")
    cap = max(max(sizes), 128)
    send = torch.zeros(cap, dtype=torch.uint8, device=device)
    send[:payload.numel()] = payload
    bufs = [torch.empty(cap, dtype=torch.uint8, device=device) for _ in sizes]
    dist.all_gather(bufs, send, group=group)
    offs = [0]
    for s in sizes:
        offs.append(offs[-1] + s)
    recv = torch.cat([b[:s] for b, s in zip(bufs, sizes)]) if offs[-1] else \
        torch.zeros(16, dtype=torch.uint8, device=device)
    return recv, torch.tensor(offs, dtype=torch.int64, device=device)
