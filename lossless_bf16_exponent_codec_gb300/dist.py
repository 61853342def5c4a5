"""The exchange steps of the compressed collectives across ranks: all-gather,
all-to-all (Designs 1 and 2) and reduce-scatter, and the switcher between the
compressed and the native reduce-scatter.

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


# ---- compressed all-to-all and reduce-scatter (ZipCCL 3.2) ------------------
#
# zipcclAlltoAll: rank r holds one compressed chunk per peer (the code3
# encoder's per-peer chunks: chunk j goes to rank j).  Design 1 exchanges the
# chunk sizes, then the chunks.  Design 2 first moves each chunk's static
# part, whose size is known before compression (header, sign+mantissa bytes,
# the three code planes and the index of a code3 chunk), then the sizes and
# bytes of the dynamic part (the escapes); a rank that is ready early moves
# most of its bytes before any size is known.  zipcclReduceScatter is the
# all-to-all followed by a local decode and a sum in higher precision (FP32),
# so no addition ever happens on compressed data.  The receiver lays the W
# chunks it gets back to back in source-rank order, static part then dynamic
# part, so each chunk is contiguous and 128-byte aligned as the decoder wants.


def _rup(x: int, a: int) -> int:
    return -(-x // a) * a


def code3_static_bytes(n_c: int) -> int:
    """Bytes of a code3 chunk of n_c values before its escapes: header 128,
    sign+mantissa, three planes, index (one u64 per 8192 values), each
    section padded to 128 bytes (the format in the C header)."""
    return 128 + _rup(n_c, 128) + 3 * _rup(-(-n_c // 8), 128) + _rup(8 * -(-n_c // 8192), 128)


def _a2a_sizes(sizes: list[int], device, group=None) -> list[int]:
    world = dist.get_world_size(group)
    send = torch.tensor(sizes, dtype=torch.int64, device=device)
    recv = torch.empty(world, dtype=torch.int64, device=device)
    dist.all_to_all_single(recv, send, group=group)
    return [int(v) for v in recv.tolist()]


def _a2a_bytes(parts: list[torch.Tensor], recv_sizes: list[int], device, group=None) -> list[torch.Tensor]:
    send_sizes = [int(p.numel()) for p in parts]
    send = torch.cat(parts) if sum(send_sizes) else torch.zeros(0, dtype=torch.uint8, device=device)
    recv = torch.empty(sum(recv_sizes), dtype=torch.uint8, device=device)
    dist.all_to_all_single(recv, send, output_split_sizes=recv_sizes, input_split_sizes=send_sizes,
                           group=group)
    out, o = [], 0
    for s in recv_sizes:
        out.append(recv[o:o + s])
        o += s
    return out


def alltoall_payloads(chunks: list[torch.Tensor], design: int = 1, static_bytes: list[int] | None = None,
                      group=None) -> tuple[torch.Tensor, torch.Tensor]:
    """Variable-size all-to-all of uint8 chunks: chunks[j] goes to rank j.

    design 1: the sizes, then the chunks.  design 2: the static parts
    (static_bytes[j] bytes of chunks[j]; the same for every sender of chunk j,
    so the receiver knows its own), then the dynamic parts' sizes and bytes.
    Returns the received chunks back to back in source order and the W+1
    int64 offsets (on the chunks' device)."""
    world = dist.get_world_size(group)
    me = dist.get_rank(group)
    if len(chunks) != world:
        raise ValueError("one chunk per rank")
    device = chunks[0].device
    for c in chunks:
        if c.dtype != torch.uint8 or c.dim() != 1 or c.numel() % 128:
            raise ValueError("chunks must be 1-D uint8 tensors, multiples of 128 bytes")
    if design == 1:
        rsz = _a2a_sizes([int(c.numel()) for c in chunks], device, group)
        got = _a2a_bytes(list(chunks), rsz, device, group)
    elif design == 2:
        if static_bytes is None or len(static_bytes) != world:
            raise ValueError("design 2 needs the static size of every chunk")
        for c, s in zip(chunks, static_bytes):
            if s % 128 or s > c.numel():
                raise ValueError("static part must be a 128-byte multiple within the chunk")
        stat = _a2a_bytes([c[:s] for c, s in zip(chunks, static_bytes)], [static_bytes[me]] * world,
                          device, group)
        dyn_send = [c[s:] for c, s in zip(chunks, static_bytes)]
        rsz = _a2a_sizes([int(d.numel()) for d in dyn_send], device, group)
        dyn = _a2a_bytes(dyn_send, rsz, device, group)
        got = [torch.cat([a, b]) for a, b in zip(stat, dyn)]
    else:
        raise ValueError("design is 1 or 2")
    offs = [0]
    for g in got:
        offs.append(offs[-1] + int(g.numel()))
    recv = torch.cat(got) if offs[-1] else torch.zeros(16, dtype=torch.uint8, device=device)
    return recv, torch.tensor(offs, dtype=torch.int64, device=device)


def reduce_decoded(decoded: list[torch.Tensor], accumulate=None) -> torch.Tensor:
    """The local step of the compressed reduce-scatter: the W decoded BF16
    chunks (raw bits, int16) summed in FP32, in source-rank order.
    ``accumulate(acc, x, first)`` does acc = (0 if first else acc) + x on the
    device (the library's kernel); without it (host tensors) the sum runs in
    numpy float32, one addition per source in the same order."""
    if not decoded:
        raise ValueError("nothing to reduce")
    n = decoded[0].numel()
    if accumulate is not None:
        acc = torch.empty(n, dtype=torch.float32, device=decoded[0].device)
        for i, d in enumerate(decoded):
            accumulate(acc, d, i == 0)
        return acc
    import numpy as np
    acc = np.zeros(n, dtype=np.float32)
    for d in decoded:
        v = (d.numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32)
        acc = acc + v
    return torch.from_numpy(acc)


class CollectiveSwitcher:
    """The adaptive choice between the native reduce-scatter and the
    compressed all-to-all plus local sum:

        T_RS(d)  = alpha_RS  + beta_RS  d
        T_A2A(d) = alpha_A2A + beta_A2A e s d

    with d the data size, e the compression factor (compressed over original)
    and s the precision factor (0.5 for FP32 traffic replaced by BF16, 1 when
    the native path is BF16 too).  alpha and beta of each path are fitted by
    least squares to latencies measured at start-up; the compressed path is
    taken only when T_A2A < T_RS."""

    def __init__(self, rs_samples, a2a_samples):
        self.a_rs, self.b_rs = self.fit(rs_samples)
        self.a_a2a, self.b_a2a = self.fit(a2a_samples)

    @staticmethod
    def fit(samples) -> tuple[float, float]:
        """Least-squares line t = alpha + beta d through (d, t) samples of
        the path as timed (the all-to-all timed on payloads of d bytes)."""
        pts = [(float(d), float(t)) for d, t in samples]
        if len(pts) < 2 or len({d for d, _ in pts}) < 2:
            raise ValueError("need two or more distinct sizes")
        m = len(pts)
        sd = sum(d for d, _ in pts)
        st = sum(t for _, t in pts)
        sdd = sum(d * d for d, _ in pts)
        sdt = sum(d * t for d, t in pts)
        beta = (m * sdt - sd * st) / (m * sdd - sd * sd)
        alpha = (st - beta * sd) / m
        return alpha, beta

    def t_rs(self, d: float) -> float:
        return self.a_rs + self.b_rs * d

    def t_a2a(self, d: float, e: float, s: float) -> float:
        return self.a_a2a + self.b_a2a * e * s * d

    def compress(self, d: float, e: float, s: float = 0.5) -> bool:
        return self.t_a2a(d, e, s) < self.t_rs(d)


def _code3_chunks(codec, x: torch.Tensor, stream=None) -> list[torch.Tensor]:
    """This rank's tensor coded into W per-peer chunks (window from its own
    statistics); reading the size table is the host sync the collective's
    size exchange needs anyway."""
    codec.stats(x, stream=stream)
    codec.encode_code3(x, stream=stream)
    sizes = codec.sizes.cpu().tolist()
    if codec.status_word():
        raise RuntimeError(f"encode status {codec.status_word():#x}")
    return [codec.out[j * codec.slot:j * codec.slot + sizes[j]] for j in range(codec.W)]


def alltoall_code3(codec, x: torch.Tensor, design: int = 1, group=None) -> torch.Tensor:
    """zipcclAlltoAll on device tensors: chunk j of this rank's x goes to rank
    j; returns the W chunks received (chunk `rank` of every source), decoded
    into codec.L-value rows in source order (BF16 bits, int16)."""
    me = dist.get_rank(group)
    chunks = _code3_chunks(codec, x)
    static = [code3_static_bytes(max(0, min(codec.L, codec.n - j * codec.L))) for j in range(codec.W)]
    recv, offs = alltoall_payloads(chunks, design=design, static_bytes=static if design == 2 else None,
                                   group=group)
    out = torch.zeros(codec.W * max(codec.L, 1), dtype=torch.int16, device=x.device)
    o = offs.cpu().tolist()
    for s in range(codec.W):
        one = torch.tensor([0, o[s + 1] - o[s]], dtype=torch.int64, device=x.device)
        codec.decode_code3(recv[o[s]:], one, first=me, count=1, out=out[s * codec.L:])
    if codec.status_word():
        raise RuntimeError(f"decode status {codec.status_word():#x}")
    return out


def reduce_scatter_code3(codec, x: torch.Tensor, design: int = 1, group=None) -> torch.Tensor:
    """zipcclReduceScatter on device tensors: the compressed all-to-all, then
    the W received chunks decoded and summed in FP32 in source order (the
    library's kernels).  Returns this rank's chunk of the sum (FP32)."""
    me = dist.get_rank(group)
    chunks = _code3_chunks(codec, x)
    static = [code3_static_bytes(max(0, min(codec.L, codec.n - j * codec.L))) for j in range(codec.W)]
    recv, offs = alltoall_payloads(chunks, design=design, static_bytes=static if design == 2 else None,
                                   group=group)
    acc = codec.reduce_received(recv, offs, me)
    if codec.status_word():
        raise RuntimeError(f"decode status {codec.status_word():#x}")
    return acc
