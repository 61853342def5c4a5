"""Benefit-driven selective compression (host logic).

Pinned to the formulas of CIERA's gain paragraphs (sizes, expected payload,
gain, footprint, ranking), to the oracle's payloads (exact byte counts and
changed-block counts), and to the outcomes the pages report: low-change
categories (expert FFN, layer norm) are chosen and high-change ones
(attention, routing gate) are skipped over a slow inter-node link, and no
shard pays off on a fast intra-node link."""
import math

import numpy as np
import pytest

import synth
from lossless_bf16_exponent_codec_gb300 import bsc


def _bf16(rng, n, sigma=0.02):
    return (rng.normal(0, sigma, n).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _flip(rng, x, rate):
    """Move a seeded fraction of exponents by one binade (never to 0 or 255)."""
    y = x.copy()
    e = (y >> 7) & 0xFF
    pick = (rng.random(x.size) < rate) & (e > 1) & (e < 254)
    e2 = np.where(rng.random(x.size) < 0.5, e - 1, e + 1)
    y[pick] = (y[pick] & 0x807F) | (e2[pick].astype(np.uint16) << 7)
    return y


def _changed_blocks(a, b, B):
    n = a.size
    nb = -(-n // B)
    d = np.zeros(nb * B, dtype=bool)
    d[:n] = ((a ^ b) & 0x7F80) != 0
    return d.reshape(nb, B).any(axis=1) if nb else np.zeros(0, bool)


def test_sizes_closed_form():
    z = bsc.sizes(bsc.Shard("a", 1000, 0.25), 256)
    assert (z.S, z.S_e, z.S_sm, z.S_b, z.S_bm) == (2000, 1000, 1000, 4, 1)
    assert z.payload == 1000 + 1 + 250
    z = bsc.sizes(bsc.Shard("b", 2 ** 20, 0.0), 512)
    assert (z.S_b, z.S_bm, z.payload) == (2048, 256, 2 ** 20 + 256)
    z = bsc.sizes(bsc.Shard("c", 7, 1.0), 8)
    assert (z.S, z.S_b, z.S_bm, z.payload) == (14, 1, 1, 15)


@pytest.mark.parametrize("n", [0, 1, 255, 256, 257, 8192, 8193, 40000])
@pytest.mark.parametrize("B", [8, 64, 256, 1024])
def test_change_rate_and_exact_bytes_match_the_oracle(orc, n, B):
    rng = np.random.default_rng(n * 7 + B)
    x0 = _bf16(rng, n)
    x1 = _flip(rng, x0, 0.002)
    cache = np.zeros(max(n, 1), np.uint8)
    orc.reuse_encode(x0, B, 0, cache, cold=True)
    pay, _ = orc.reuse_encode(x1, B, 0, cache)
    ch = _changed_blocks(x0, x1, B)
    n_changed = int(np.frombuffer(pay[24:32].tobytes(), "<u8")[0])
    assert n_changed == int(ch.sum())
    q = bsc.block_change_rate(x0, x1, B)
    assert q == (ch.mean() if ch.size else 0.0)
    assert bsc.change_rate_from_header(pay, n, B) == q
    last = bool(ch[-1]) if ch.size else False
    assert bsc.payload_bytes_exact(n, B, n_changed, last) == pay.size


def test_gain_with_a_linear_link_is_the_saved_bytes_over_the_bandwidth():
    sh = bsc.Shard("s", 1 << 24, 0.3)
    comm = bsc.LinearComm(alpha=20e-6, bw=8e9)
    W, Gd = 8, 1.5e12
    z = bsc.sizes(sh, 512)
    td = bsc.decmp_time(sh, W, Gd)
    assert td == W * z.S / Gd
    g = bsc.gain(sh, 512, comm, td)
    assert g == pytest.approx((z.S - z.payload) / 8e9 - td, rel=1e-12)   # alpha cancels
    # the sender's hash and compress times count only without pipelining
    assert bsc.gain(sh, 512, comm, td, t_hash=1e-3, t_cmp=2e-3) == g
    assert bsc.gain(sh, 512, comm, td, 1e-3, 2e-3, pipelined=False) == pytest.approx(g - 3e-3)


def test_table_comm_interpolates_and_extends():
    c = bsc.TableComm([(1e7, 1010e-6), (0, 10e-6), (1e6, 110e-6)])
    assert c(0) == 10e-6 and c(1e6) == 110e-6
    assert c(5e5) == pytest.approx(60e-6)
    assert c(2e7) == pytest.approx(2010e-6)          # last segment, extended
    lin = bsc.LinearComm(5e-6, 50e9)
    t = bsc.TableComm([(d, lin(d)) for d in (0, 1e5, 1e8)])
    for d in (3e4, 7e6, 5e8):
        assert t(d) == pytest.approx(lin(d), rel=1e-12)
    with pytest.raises(ValueError):
        bsc.TableComm([(1, 1.0)])


def test_every_block_changing_never_pays():
    comm = bsc.LinearComm(0.0, 1e9)
    for n in (8, 1000, 1 << 22):
        sh = bsc.Shard("all", n, 1.0)
        assert bsc.sizes(sh, 64).payload > bsc.sizes(sh, 64).S
        assert bsc.gain(sh, 64, comm, 0.0) < 0
    choice = bsc.select([bsc.Shard("all", 1 << 20, 1.0)], 64, 4, 1e18, comm, 1e15)
    assert not choice[0].selected


def test_selection_ranks_by_gain_per_cache_byte_and_stops_at_the_budget():
    comm = bsc.LinearComm(0.0, 10e9)
    W, Gd, B = 4, 1e18, 256            # decode cost negligible: g = (S - P) / bw
    shards = [bsc.Shard("a", 1 << 20, 0.5), bsc.Shard("b", 1 << 18, 0.1),
              bsc.Shard("c", 1 << 22, 0.2), bsc.Shard("d", 1 << 16, 0.9),
              bsc.Shard("e", 1 << 18, 0.1), bsc.Shard("f", 1 << 16, 1.0)]
    # g / M = (S_e (1 - q) - S_bm) / bw / ((W - 1) S_e): smaller q ranks first
    M = {s.name: (W - 1) * bsc.sizes(s, B).S_e for s in shards}
    budget = M["b"] + M["e"] + M["c"] + M["a"] // 2
    out = bsc.select(shards, B, W, budget, comm, Gd)
    order = [c.shard.name for c in out]
    assert order[:5] == ["b", "e", "c", "a", "d"]    # b and e tie: input order
    assert order[5] == "f"                           # g < 0: listed last
    sel = [c.shard.name for c in out if c.selected]
    assert sel == ["b", "e", "c"]                    # a no longer fits, and d is not taken after it
    for c in out:
        z = bsc.sizes(c.shard, B)
        assert c.gain == pytest.approx((z.S - z.payload) / 10e9 - W * z.S / Gd)
        assert c.footprint == M[c.shard.name]


def test_pages_outcomes_for_olmoe_categories():
    # category medians of the block change rate at B = 512 for OLMoE-1B-7B
    # (the pages' per-category figure), sizes of the OLMoE-shaped layer set
    q = {"expert_ffn": 0.22, "attention": 0.96, "router": 0.94, "norm": 0.64, "embedding": 0.65}
    n = {}
    for s in synth.olmoe_segments():
        n[s.category] = n.get(s.category, 0) + s.numel
    shards = bsc.shards_from_categories(q, n)
    Gd = 2.0e12            # order of this library's measured gather-decode throughput (bytes/s)
    # inter-node all-gather at the pages' measured ~8 GB/s bus bandwidth
    inter = bsc.select(shards, 512, 16, math.inf, bsc.LinearComm(50e-6, 8e9), Gd)
    chosen = {c.shard.name for c in inter if c.selected}
    assert {"expert_ffn", "norm"} <= chosen
    assert "attention" not in chosen and "router" not in chosen
    # within a node on NVLink (600 GB/s): no shard pays for its reconstruction
    intra = bsc.select(shards, 512, 4, math.inf, bsc.LinearComm(10e-6, 600e9), Gd)
    assert not any(c.selected for c in intra)


def test_bad_inputs():
    with pytest.raises(ValueError):
        bsc.sizes(bsc.Shard("x", 10, 1.5), 8)
    with pytest.raises(ValueError):
        bsc.select([], 8, 1, 1.0, bsc.LinearComm(0, 1), 1.0)
    with pytest.raises(ValueError):
        bsc.block_change_rate(np.zeros(4, np.uint16), np.zeros(5, np.uint16), 8)
