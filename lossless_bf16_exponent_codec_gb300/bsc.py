"""Benefit-driven selective compression: which shards to all-gather with
exponent reuse.

CIERA, the paragraphs on selective compression and the gain formula.  For a
shard i of N values in b-bit precision (16 for BF16), split into blocks of B
values:

    S      = N b / 8                     bytes of the shard
    S_e    = N e / 8                     exponent bytes (e = 8 for BF16)
    S_sm   = S - S_e                     sign+mantissa bytes
    S_b    = ceil(N / B)                 blocks
    S_bm   = ceil(S_b / 8)               bitmap bytes
    P      = S_sm + S_bm + q S_e         expected payload per iteration, with
                                         q the shard's block change rate

    g      = Comm(S) - (Comm(P) + T_hash + T_cmp + T_decmp)
    M      = (W - 1) S_e                 receiver cache footprint per GPU

Comm maps a per-GPU payload size to the all-gather latency.  With the
sender's work on a stream of its own, T_hash and T_cmp are off the critical
path and only T_decmp counts (the default here).  Shards with g <= 0 are
dropped; the rest are taken in descending order of g / M until the cache
budget is exhausted, and the selection stays fixed for the run.

Readings where the pages leave a step open:

* "until the cache budget is exhausted": shards are taken in ranked order
  and the selection stops at the first shard whose footprint no longer fits
  (no skipping ahead to smaller shards).  Equal ratios keep the input order.
* T_decmp is the receiver's reconstruction of the gathered tensor, W shards
  of N values, at a measured decode throughput G_d in uncompressed bytes per
  second: T_decmp = W S / G_d.
* P is the pages' expected payload; the library's payload adds a 64-byte
  header, one index entry per 8192 values and padding to 16 and 128 bytes
  (``payload_bytes_exact`` gives those bytes for a known changed-block count).
* The block change rate q is the fraction of blocks with at least one changed
  exponent between two iterations (``block_change_rate``), or read from the
  changed-block counts the encoder writes into its payload headers.
"""
from __future__ import annotations

import bisect
from dataclasses import dataclass
from typing import Callable, List, Optional, Sequence

import numpy as np

KTILE = 8192


@dataclass(frozen=True)
class Shard:
    name: str
    n_values: int
    q: float                 # block change rate per iteration, 0..1
    bits: int = 16
    exp_bits: int = 8


@dataclass(frozen=True)
class Sizes:
    S: int
    S_e: int
    S_sm: int
    S_b: int
    S_bm: int
    payload: float           # S_sm + S_bm + q S_e


def sizes(sh: Shard, B: int) -> Sizes:
    if sh.n_values < 0 or B <= 0 or not 0.0 <= sh.q <= 1.0:
        raise ValueError("bad shard")
    S = sh.n_values * sh.bits // 8
    S_e = sh.n_values * sh.exp_bits // 8
    S_sm = S - S_e
    S_b = -(-sh.n_values // B)
    S_bm = -(-S_b // 8)
    return Sizes(S, S_e, S_sm, S_b, S_bm, S_sm + S_bm + sh.q * S_e)


def _rup(x: int, a: int) -> int:
    return -(-x // a) * a


def payload_bytes_exact(n_values: int, B: int, n_changed: int, last_block_changed: bool) -> int:
    """Bytes of the library's raw reuse payload for one shard (header 64 |
    bitmap | SM | index | EXP, see the C header), given its changed-block
    count; the exponent stream holds B bytes per changed block, fewer for a
    changed partial last block."""
    nb = -(-n_values // B)
    m = n_changed * B
    if last_block_changed and n_values:
        m -= nb * B - n_values
    off_sm = 64 + _rup(-(-nb // 8), 16)
    off_idx = off_sm + _rup(n_values, 16)
    off_exp = off_idx + _rup(8 * -(-n_values // KTILE), 16)
    return _rup(off_exp + m, 128)


class LinearComm:
    """Comm(d) = alpha + d / bw (seconds, bytes, bytes per second)."""

    def __init__(self, alpha: float, bw: float):
        if bw <= 0 or alpha < 0:
            raise ValueError("bad link model")
        self.alpha, self.bw = alpha, bw

    def __call__(self, d: float) -> float:
        return self.alpha + d / self.bw


class TableComm:
    """Comm from measured (payload bytes, latency) points: piecewise linear
    between them, the end segments extended beyond the first and last point."""

    def __init__(self, points: Sequence[tuple]):
        pts = sorted((float(d), float(t)) for d, t in points)
        if len(pts) < 2 or len({d for d, _ in pts}) != len(pts):
            raise ValueError("need two or more distinct sizes")
        self.d = [d for d, _ in pts]
        self.t = [t for _, t in pts]

    def __call__(self, d: float) -> float:
        i = bisect.bisect_right(self.d, d) - 1
        i = min(max(i, 0), len(self.d) - 2)
        d0, d1, t0, t1 = self.d[i], self.d[i + 1], self.t[i], self.t[i + 1]
        return t0 + (t1 - t0) * (d - d0) / (d1 - d0)


def decmp_time(sh: Shard, W: int, decode_Bps: float) -> float:
    """Receiver reconstruction of the gathered tensor: W S bytes at decode_Bps."""
    return W * sizes(sh, 1).S / decode_Bps


def gain(sh: Shard, B: int, comm: Callable[[float], float], t_decmp: float,
         t_hash: float = 0.0, t_cmp: float = 0.0, pipelined: bool = True) -> float:
    """g_i; with ``pipelined`` the sender's hash and compress times are off the
    critical path and do not count."""
    z = sizes(sh, B)
    extra = t_decmp + (0.0 if pipelined else t_hash + t_cmp)
    return comm(z.S) - (comm(z.payload) + extra)


@dataclass(frozen=True)
class Choice:
    shard: Shard
    gain: float
    footprint: int           # M = (W - 1) S_e
    selected: bool


def select(shards: Sequence[Shard], B: int, W: int, budget_bytes: float,
           comm: Callable[[float], float], decode_Bps: float,
           t_hash: Optional[Sequence[float]] = None, t_cmp: Optional[Sequence[float]] = None,
           pipelined: bool = True) -> List[Choice]:
    """Rank the shards with positive gain by g / M and take them in that
    order while their footprints fit the budget.  Returns one Choice per
    shard, in ranked order (positive gains first), then the rest in input
    order."""
    if W < 2:
        raise ValueError("an all-gather needs W >= 2")
    rows = []
    for i, sh in enumerate(shards):
        th = t_hash[i] if t_hash is not None else 0.0
        tc = t_cmp[i] if t_cmp is not None else 0.0
        g = gain(sh, B, comm, decmp_time(sh, W, decode_Bps), th, tc, pipelined)
        M = (W - 1) * sizes(sh, B).S_e
        rows.append((i, sh, g, M))
    pos = [r for r in rows if r[2] > 0 and r[3] > 0]
    pos.sort(key=lambda r: (-(r[2] / r[3]), r[0]))
    out, used, full = [], 0.0, False
    for i, sh, g, M in pos:
        take = not full and used + M <= budget_bytes
        if take:
            used += M
        else:
            full = True
        out.append(Choice(sh, g, M, take))
    out += [Choice(sh, g, M, False) for i, sh, g, M in rows if not (g > 0 and M > 0)]
    return out


def block_change_rate(prev_bits: np.ndarray, cur_bits: np.ndarray, B: int) -> float:
    """Fraction of blocks of B values (the last one may be partial) with at
    least one exponent that differs between two BF16 tensors (raw bits)."""
    a = np.asarray(prev_bits).view(np.uint16)
    b = np.asarray(cur_bits).view(np.uint16)
    if a.shape != b.shape or a.ndim != 1:
        raise ValueError("two flat tensors of one shape")
    n = a.size
    if n == 0:
        return 0.0
    diff = ((a ^ b) & 0x7F80) != 0
    nb = -(-n // B)
    pad = np.zeros(nb * B, dtype=bool)
    pad[:n] = diff
    return float(pad.reshape(nb, B).any(axis=1).mean())


def change_rate_from_header(payload: bytes | np.ndarray, n_values: int, B: int) -> float:
    """q of one shard from the changed-block count in its reuse payload header
    (little-endian u64 at bytes 24..31)."""
    h = np.frombuffer(bytes(np.asarray(payload, dtype=np.uint8)[:32]), dtype="<u8")
    nb = -(-n_values // B)
    return float(h[3]) / nb if nb else 0.0


def shards_from_categories(q_by_category: dict, n_by_category: dict) -> List[Shard]:
    """One shard per category from per-category change rates and sizes."""
    return [Shard(k, int(n_by_category[k]), float(q)) for k, q in q_by_category.items()]
