"""Seeded synthetic BF16 weight tensors for the exponent codecs.

This module holds no codec arithmetic.  It only draws the inputs that both the
CPU oracle and the CUDA library are fed, so both sides see the same bits.

Randomness is counter based, so any element can be drawn on its own, on the
CPU or on a CUDA device, in any chunking:

* ``word(key, i)`` is the i-th output of a SplitMix64 generator seeded with
  ``key`` (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): F(key + (i + 1) * gamma mod 2**64), with
  gamma = 0x9E3779B97F4A7C15 and F the SplitMix64 output mix.  The
  integer steps are exact on every device.
* Uniforms use the top 53 bits; normals use the Box-Muller transform in
  float64.  The float64 ``log``/``cos`` of a CUDA device may differ from the
  CPU's in the last place, so a tensor drawn on a GPU can differ from the same
  tensor drawn on the CPU in rare elements.  Every test feeds ONE drawn tensor
  to both sides, so this never affects parity.
* Rounding to BF16 is a direct round-to-nearest-even from float64 (one
  rounding), done on the integer bits.

BF16 tensors are returned as ``torch.int16`` tensors holding the raw bits.

Workloads (shapes and drift models follow the codec pages' experiments; the
trained checkpoints and datasets they measured are not available, so these
synthetic tensors stand in for them):

* config 1 -- one tensor of 2**20 values from N(0, 0.02); iteration t adds an
  update u ~ N(0, 1e-4*|w| + 1e-6) in float32 and rounds back to BF16.
* config 2 -- 2**26 values from N(0, 0.02); a seeded 0.5% of entries times
  100, a disjoint 0.1% set to +0.0.
* config 3 -- an OLMoE-1B-7B-shaped layer set (expert FFN, attention, router,
  LayerNorm, embedding) in one flat buffer; per-category exponent flips,
  20% of rows at 5x the category rate.
* config 4 -- four DeepSeek-MoE-16B-shaped layers; per-category flips.
* config 5 -- 2**30 values in the config-3 mix, 20 iterations of flips at a
  mean rate of 0.08% (1-10) then 0.4% (11-20).
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import List, Sequence, Tuple

import numpy as np

import torch

__all__ = [
    "word", "uniform", "normal", "round_bf16", "gaussian_bf16",
    "flip_exponents", "lr_update", "Segment", "olmoe_segments",
    "deepseek_layer_segments", "config1", "config2", "config3_base",
    "config3_step", "config4_layer", "config5_base", "config5_step",
    "config5_rate_factor", "scale_drift_bench", "pow2_bf16", "rounding_tie_cases",
]

_M64 = (1 << 64) - 1
_GAMMA = 0x9E3779B97F4A7C15
_MIX1 = 0xBF58476D1CE4E5B9
_MIX2 = 0x94D049BB133111EB


def _s64(c: int) -> int:
    """Two's-complement int64 value of an unsigned 64-bit constant."""
    c &= _M64
    return c - (1 << 64) if c >= (1 << 63) else c


def _srl(x: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return (x >> s) & ((1 << (64 - s)) - 1)


def _mix(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _srl(z, 30)) * _s64(_MIX1)
    z = (z ^ _srl(z, 27)) * _s64(_MIX2)
    return z ^ _srl(z, 31)


def _mix_int(z: int) -> int:
    z &= _M64
    z = ((z ^ (z >> 30)) * _MIX1) & _M64
    z = ((z ^ (z >> 27)) * _MIX2) & _M64
    return z ^ (z >> 31)


def key_of(*parts: int) -> int:
    """Fold integers (seed, stream ids) into one 64-bit generator key."""
    k = 0x243F6A8885A308D3
    for p in parts:
        k = _mix_int(k + (p & _M64) * _GAMMA + _GAMMA)
    return k


def word(key: int, idx: torch.Tensor) -> torch.Tensor:
    """idx-th SplitMix64 output for ``key`` (int64 bit patterns)."""
    idx = idx.to(torch.int64)
    return _mix(idx * _s64(_GAMMA) + _s64(key + _GAMMA))


def uniform(key: int, idx: torch.Tensor) -> torch.Tensor:
    """Uniform float64 in (0, 1) from the top 53 bits of ``word``."""
    w = _srl(word(key, idx), 11)
    return (w.to(torch.float64) + 0.5) * (2.0 ** -53)


def normal(key: int, idx: torch.Tensor) -> torch.Tensor:
    """Standard normal float64 by Box-Muller from words 2*idx and 2*idx+1."""
    u1 = uniform(key, 2 * idx)
    u2 = uniform(key, 2 * idx + 1)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


def round_bf16(x: torch.Tensor) -> torch.Tensor:
    """float64 -> BF16 bits (int16), one round-to-nearest-even step.

    Works on the float64 bit pattern: keeps 7 fraction bits, rounds the other
    45 to nearest, ties to even; a carry into the exponent field is the
    correct next binade (and 0x7F80 = inf on overflow).  Magnitudes below
    2**-126 are rounded on the 2**-133 grid of BF16 subnormals.  NaN inputs
    are not expected from the generators and are not handled.
    """
    x = x.to(torch.float64)
    b = x.view(torch.int64)
    sign = _srl(b, 63) << 15
    e11 = _srl(b, 52) & 0x7FF
    frac = b & ((1 << 52) - 1)
    e8 = e11 - 1023 + 127
    m7 = _srl(frac, 45)
    rem = frac & ((1 << 45) - 1)
    half = 1 << 44
    up = (rem > half) | ((rem == half) & ((m7 & 1) == 1))
    normal_bits = ((e8 << 7) | m7) + up.to(torch.int64)
    normal_bits = torch.clamp(normal_bits, max=0x7F80)
    # below the normal range: integer count of 2**-133 quanta, ties to even
    q = torch.round(torch.abs(x) * (2.0 ** 133)).to(torch.int64)
    bits = torch.where(e8 >= 1, normal_bits, q)
    bits = bits | sign
    return bits.to(torch.int32).to(torch.int16)


def gaussian_bf16(n: int, sigma: float, key: int, device="cpu",
                  mean: float = 0.0, start: int = 0,
                  chunk: int = 1 << 24) -> torch.Tensor:
    """n BF16 values mean + sigma*z, element i drawn from counter start+i."""
    out = torch.empty(n, dtype=torch.int16, device=device)
    for a in range(0, n, chunk):
        b = min(n, a + chunk)
        idx = torch.arange(start + a, start + b, dtype=torch.int64, device=device)
        out[a:b] = round_bf16(mean + sigma * normal(key, idx))
    return out


# --------------------------------------------------------------------------
# drift models
# --------------------------------------------------------------------------

def flip_exponents(bits: torch.Tensor, rate: torch.Tensor, key: int,
                   start: int = 0, redraw_mantissa: bool = True,
                   chunk: int = 1 << 24) -> torch.Tensor:
    """One training-like step on raw BF16 bits, drawn per element.

    An element flips with probability ``rate`` (a per-element float64 tensor
    or a scalar tensor): its 8-bit exponent field moves to E+1 or E-1 on a
    fair coin, forced to +1 at E <= 1 and to -1 at E >= 254; sign and
    mantissa are kept.  Independently, with probability 1/2 every element's
    7 mantissa bits are redrawn, so sign+mantissa bytes keep changing as in
    training while the exponent changes only at the flipped elements.
    """
    n = bits.numel()
    out = torch.empty_like(bits)
    dev = bits.device
    for a in range(0, n, chunk):
        b = min(n, a + chunk)
        idx = torch.arange(start + a, start + b, dtype=torch.int64, device=dev)
        h = bits[a:b].to(torch.int32) & 0xFFFF
        w0 = word(key, 3 * idx)
        w1 = word(key, 3 * idx + 1)
        w2 = word(key, 3 * idx + 2)
        u = (_srl(w0, 11).to(torch.float64) + 0.5) * (2.0 ** -53)
        r = rate if rate.dim() == 0 else rate[a:b]
        flip = u < r
        e = (h >> 7) & 0xFF
        up = (w1 & 1) == 1
        up = torch.where(e <= 1, torch.ones_like(up), up)
        up = torch.where(e >= 254, torch.zeros_like(up), up)
        e2 = torch.where(up, e + 1, e - 1)
        e = torch.where(flip, e2, e)
        m = h & 0x7F
        if redraw_mantissa:
            redraw = ((w1 >> 1) & 1) == 1
            m = torch.where(redraw, (w2 & 0x7F).to(torch.int32), m)
        h2 = (h & 0x8000) | (e << 7) | m
        out[a:b] = h2.to(torch.int16)
    return out


def lr_update(bits: torch.Tensor, scale_rel: float, scale_abs: float,
              key: int, chunk: int = 1 << 24) -> torch.Tensor:
    """w_t = bf16(f32(w) + f32(u)), u ~ N(0, scale_rel*|w| + scale_abs).

    The second argument of N(.,.) is read as the standard deviation; the
    update is added in float32 and the sum rounded to BF16 (nearest even).
    """
    n = bits.numel()
    out = torch.empty_like(bits)
    dev = bits.device
    for a in range(0, n, chunk):
        b = min(n, a + chunk)
        idx = torch.arange(a, b, dtype=torch.int64, device=dev)
        w32 = (bits[a:b].to(torch.int32) << 16).view(torch.float32)
        sd = scale_rel * torch.abs(w32.to(torch.float64)) + scale_abs
        u32 = (normal(key, idx) * sd).to(torch.float32)
        s32 = w32 + u32
        out[a:b] = s32.to(torch.bfloat16).view(torch.int16)
    return out


# --------------------------------------------------------------------------
# MoE-shaped layer sets
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class Segment:
    """One weight matrix of a flat parameter buffer."""
    category: str        # expert_ffn | attention | router | norm | embedding
    rows: int
    cols: int
    sigma: float         # init std
    mean: float          # init mean (1.0 for norms)
    rate: float          # per-element exponent flip rate

    @property
    def numel(self) -> int:
        return self.rows * self.cols


def olmoe_segments() -> List[Segment]:
    """OLMoE-1B-7B-shaped layer set (522,588,160 values)."""
    segs: List[Segment] = []
    for _ in range(64 * 3):
        segs.append(Segment("expert_ffn", 2048, 1024, 0.02, 0.0, 0.005))
    for _ in range(4):
        segs.append(Segment("attention", 2048, 2048, 0.02, 0.0, 0.003))
    segs.append(Segment("router", 2048, 64, 0.02, 0.0, 0.01))
    for _ in range(2):
        segs.append(Segment("norm", 1, 2048, 0.01, 1.0, 0.0))
    segs.append(Segment("embedding", 50304, 2048, 0.02, 0.0, 0.001))
    return segs


def deepseek_layer_segments() -> List[Segment]:
    """One DeepSeek-MoE-16B-shaped layer (587,862,016 values)."""
    segs: List[Segment] = []
    for _ in range(66 * 3):
        segs.append(Segment("expert_ffn", 2048, 1408, 0.02, 0.0, 0.005))
    for _ in range(4):
        segs.append(Segment("attention", 2048, 2048, 0.02, 0.0, 0.003))
    segs.append(Segment("router", 2048, 64, 0.02, 0.0, 0.01))
    for _ in range(2):
        segs.append(Segment("norm", 1, 2048, 0.01, 1.0, 0.0))
    return segs


def _segments_base(segs: Sequence[Segment], key: int, device,
                   limit: int | None = None) -> torch.Tensor:
    total = sum(s.numel for s in segs)
    n = total if limit is None else limit
    out = torch.empty(n, dtype=torch.int16, device=device)
    pos = 0
    i = 0
    while pos < n:
        s = segs[i % len(segs)]
        take = min(s.numel, n - pos)
        out[pos:pos + take] = gaussian_bf16(take, s.sigma, key, device,
                                            mean=s.mean, start=pos)
        pos += take
        i += 1
    return out


def _segments_rate(segs: Sequence[Segment], n: int, factor: float,
                   cluster: bool, key: int, device) -> torch.Tensor:
    """Per-element flip rate; with ``cluster`` a seeded 20% of each matrix's
    rows (first dimension) get 5x the category rate."""
    rate = torch.empty(n, dtype=torch.float64, device=device)
    pos = 0
    i = 0
    row_base = 0
    while pos < n:
        s = segs[i % len(segs)]
        take = min(s.numel, n - pos)
        r = torch.full((take,), s.rate * factor, dtype=torch.float64, device=device)
        if cluster and s.rate > 0:
            nrows = (take + s.cols - 1) // s.cols
            ridx = torch.arange(row_base, row_base + nrows, dtype=torch.int64,
                                device=device)
            hot = uniform(key, ridx) < 0.2
            mult = torch.where(hot, 5.0, 1.0).to(torch.float64)
            r = r * mult.repeat_interleave(s.cols)[:take]
            row_base += nrows
        rate[pos:pos + take] = r
        pos += take
        i += 1
    return rate


def config1(n: int = 1 << 20, iterations: int = 1, variant: str = "literal",
            seed: int = 1, device="cpu") -> List[torch.Tensor]:
    """Config 1: [w_0, w_1, ..., w_iterations] for the tiny reuse case.

    ``variant`` "literal" draws u ~ N(0, 1e-4|w| + 1e-6) (second argument read
    as a standard deviation); "1b" uses 2.3e-3|w| + 1e-6, a scale that
    realises an exponent change rate near 0.3%.
    """
    rel = {"literal": 1e-4, "1b": 2.3e-3}[variant]
    ws = [gaussian_bf16(n, 0.02, key_of(seed, 0), device)]
    for t in range(1, iterations + 1):
        ws.append(lr_update(ws[-1], rel, 1e-6, key_of(seed, 100 + t)))
    return ws


def config2(n: int = 1 << 26, seed: int = 2, device="cpu") -> torch.Tensor:
    """Config 2: N(0, 0.02) with 0.5% of entries x100 and 0.1% set to +0."""
    out = torch.empty(n, dtype=torch.int16, device=device)
    k_val, k_sel = key_of(seed, 0), key_of(seed, 1)
    chunk = 1 << 24
    for a in range(0, n, chunk):
        b = min(n, a + chunk)
        idx = torch.arange(a, b, dtype=torch.int64, device=device)
        x = 0.02 * normal(k_val, idx)
        u = uniform(k_sel, idx)
        x = torch.where(u < 0.005, x * 100.0, x)
        bits = round_bf16(x)
        zero = (u >= 0.005) & (u < 0.006)
        out[a:b] = torch.where(zero, torch.zeros_like(bits), bits)
    return out


def scale_drift_bench(bits: torch.Tensor, t: int, rate: float = 0.003,
                      seed: int = 2) -> torch.Tensor:
    """Uniform i.i.d. exponent flips at ``rate`` (iteration t of a chain)."""
    r = torch.tensor(rate, dtype=torch.float64, device=bits.device)
    return flip_exponents(bits, r, key_of(seed, 1000 + t))


def config3_base(seed: int = 3, device="cpu") -> torch.Tensor:
    return _segments_base(olmoe_segments(), key_of(seed, 0), device)


def config3_step(bits: torch.Tensor, t: int = 1, seed: int = 3,
                 cluster: bool = True) -> torch.Tensor:
    segs = olmoe_segments()
    rate = _segments_rate(segs, bits.numel(), 1.0, cluster,
                          key_of(seed, 7), bits.device)
    return flip_exponents(bits, rate, key_of(seed, 100 + t))


def config4_layer(layer: int, seed: int = 4, device="cpu"
                  ) -> Tuple[torch.Tensor, torch.Tensor]:
    """(w_{t-1}, w_t) for one DeepSeek-MoE-16B-shaped layer."""
    segs = deepseek_layer_segments()
    base = _segments_base(segs, key_of(seed, layer, 0), device)
    rate = _segments_rate(segs, base.numel(), 1.0, False,
                          key_of(seed, layer, 7), device)
    return base, flip_exponents(base, rate, key_of(seed, layer, 1))


CONFIG5_N = 1 << 30


def config5_rate_factor(target_mean: float, n: int = CONFIG5_N) -> float:
    """Common factor on the config-3 category rates so that the expected
    element-weighted flip rate (with 20% of rows at 5x) is ``target_mean``."""
    segs = olmoe_segments()
    acc, pos, i = 0.0, 0, 0
    while pos < n:
        s = segs[i % len(segs)]
        take = min(s.numel, n - pos)
        acc += take * s.rate * (0.8 * 1.0 + 0.2 * 5.0)
        pos += take
        i += 1
    return target_mean * n / acc


def config5_base(n: int = CONFIG5_N, seed: int = 5, device="cpu") -> torch.Tensor:
    return _segments_base(olmoe_segments(), key_of(seed, 0), device, limit=n)


def config5_step(bits: torch.Tensor, t: int, seed: int = 5) -> torch.Tensor:
    """Iteration t (1-based) of config 5: mean flip rate 0.08% for t <= 10,
    0.4% after."""
    target = 0.0008 if t <= 10 else 0.004
    f = config5_rate_factor(target, bits.numel())
    rate = _segments_rate(olmoe_segments(), bits.numel(), f, True,
                          key_of(seed, 7), bits.device)
    return flip_exponents(bits, rate, key_of(seed, 100 + t))


def fp8_gaussian(n: int, sigma: float, fmt: str, seed: int = 6, device="cpu",
                 mean: float = 0.0) -> torch.Tensor:
    """n FP8 values (raw bytes, uint8) of mean + sigma*z, z the counter-based
    normals of ``key_of(seed, 8)``, rounded to float32 and then to the FP8
    format ('e5m2' or 'e4m3', torch's round-to-nearest-even casts; E4M3 is
    the OCP E4M3 with no infinities)."""
    z = normal(key_of(seed, 8), torch.arange(n, dtype=torch.int64, device=device))
    dt = torch.float8_e5m2 if fmt == "e5m2" else torch.float8_e4m3fn
    return (z * sigma + mean).to(torch.float32).to(dt).view(torch.uint8)


def pow2_bf16(e: int, negative: bool = False) -> int:
    """BF16 bits of +-2^e for a normal exponent e (-126 <= e <= 127)."""
    assert -126 <= e <= 127
    return ((e + 127) << 7) | (0x8000 if negative else 0)


def rounding_tie_cases() -> List[Tuple[str, np.ndarray]]:
    """Small tensors whose exact sum or sum of squares lies exactly halfway
    between two doubles, or a hair above it, at several scales (so that the
    deciding bit falls at different 32-bit word boundaries of a fixed-point
    accumulator).  Powers of two only, so the exact sums are plain to state:
    s1 = 2^k (1 + 2^-53) is a tie, 2^k (1 + 2^-52 + 2^-53) a tie next to an
    odd last bit, and s2 = 2^2k (1 + 2^-53) a tie of the squares."""
    cases = []
    for k in (-30, -16, 0, 16, 48, 100):
        for neg in (False, True):
            p = lambda e: pow2_bf16(e, neg)
            s = "-" if neg else "+"
            cases.append((f"s1 tie even k={k}{s}", [p(k), p(k - 53)]))
            cases.append((f"s1 tie odd k={k}{s}", [p(k), p(k - 52), p(k - 53)]))
            cases.append((f"s1 above tie k={k}{s}", [p(k), p(k - 53), p(k - 90)]))
            cases.append((f"s1 tie from halves k={k}{s}", [p(k), p(k - 54), p(k - 54)]))
        cases.append((f"s2 tie even k={k}", [pow2_bf16(k), pow2_bf16(k - 27), pow2_bf16(k - 27, True)]))
        cases.append((f"s2 tie odd k={k}", [pow2_bf16(k), pow2_bf16(k - 26), pow2_bf16(k - 27),
                                            pow2_bf16(k - 27)]))
        cases.append((f"s2 above tie k={k}", [pow2_bf16(k), pow2_bf16(k - 27), pow2_bf16(k - 27),
                                              pow2_bf16(k - 60)]))
    return [(name, np.array(v, dtype=np.uint16)) for name, v in cases]
