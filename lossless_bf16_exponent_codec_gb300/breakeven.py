"""Break-even link bandwidth of a compressed collective.

ZipCCL research digest, section 3.3 (the paper's Eqs. 8-9) and the Panel 1
caption: with message size d per GPU, bottleneck bandwidth B, N GPUs and
codec throughputs G_c (compress) and G_d (decompress),

    all-gather : T_zip = d/(N G_c) + d/G_d + e d/B     (compress 1/N, decompress all)
    all-to-all : T_zip = d/G_c     + d/G_d + e d/B
    plain      : T_nccl = d/B

where e is the compression factor (compressed over original size).  Setting
T_zip = T_nccl gives the bandwidth below which compression pays:

    B*_AG  = (1 - e) / (1/(N G_c) + 1/G_d)   -> (1-e) G / (1 + 1/N) when G_c = G_d = G
    B*_A2A = (1 - e) / (1/G_c + 1/G_d)       -> (1-e) G / 2
"""
from __future__ import annotations

import math


def t_nccl(d: float, B: float) -> float:
    return d / B


def t_zip_allgather(d: float, N: int, Gc: float, Gd: float, B: float, e: float) -> float:
    return d / (N * Gc) + d / Gd + e * d / B


def t_zip_alltoall(d: float, Gc: float, Gd: float, B: float, e: float) -> float:
    return d / Gc + d / Gd + e * d / B


def break_even_allgather(e: float, Gc: float, Gd: float, N: float = math.inf) -> float:
    """B*_AG in the units of Gc/Gd; N = inf gives the many-GPU limit."""
    inv = (0.0 if math.isinf(N) else 1.0 / (N * Gc)) + 1.0 / Gd
    return (1.0 - e) / inv


def break_even_alltoall(e: float, Gc: float, Gd: float) -> float:
    return (1.0 - e) / (1.0 / Gc + 1.0 / Gd)


def speedup_allgather(d: float, N: int, Gc: float, Gd: float, B: float, e: float) -> float:
    return t_nccl(d, B) / t_zip_allgather(d, N, Gc, Gd, B, e)
