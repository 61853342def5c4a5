"""The break-even calculator reproduces the ZipCCL digest's printed numbers
(section 3.3 Panel 1 caption; section 5 Table 2 arithmetic), stored in
tests/golden/zipccl_breakeven.txt."""
import os

import pytest

from lossless_bf16_exponent_codec_gb300 import breakeven as be

HERE = os.path.dirname(os.path.abspath(__file__))


def golden():
    vals = {}
    with open(os.path.join(HERE, "golden", "zipccl_breakeven.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                k, v = line.split()
                vals[k] = float(v)
    return vals


def test_paper_break_even_points():
    g = golden()
    bag = be.break_even_allgather(g["e"], g["G_GBs"], g["G_GBs"])
    ba2a = be.break_even_alltoall(g["e"], g["G_GBs"], g["G_GBs"])
    assert bag == pytest.approx(g["BAG_GBs"], rel=0.02)     # ~360 GB/s
    assert ba2a == pytest.approx(g["BA2A_GBs"], rel=0.02)   # ~180 GB/s
    # finite N: (1-e) G / (1 + 1/N)
    assert be.break_even_allgather(0.72, 1300, 1300, N=8) == pytest.approx(0.28 * 1300 / 1.125)


def test_rdma_allgather_speedup_and_codec_time():
    g = golden()
    d = 1.0  # GB
    s = be.speedup_allgather(d, int(g["N_rdma"]), g["G2_GBs"], g["G2_GBs"], g["B_rdma_GBs"], g["e2"])
    assert round(s, 2) == g["speedup_rdma_ag"]
    codec_ms = 1e3 * (d / (g["N_rdma"] * g["G2_GBs"]) + d / g["G2_GBs"])
    assert codec_ms == pytest.approx(0.85, abs=0.01)         # "about 0.85 ms"
    # e implied by Table 2: (T_zip - codec) / T_nccl
    assert (g["t_zip_ms"] - 0.84) / g["t_nccl_ms"] == pytest.approx(0.73, abs=0.005)
    assert g["t_nccl_ms"] / g["t_zip_ms"] == pytest.approx(1.30, abs=0.005)


def test_break_even_is_the_crossing_point():
    for e in (0.6, 0.7, 0.8):
        for N in (2, 8, 64):
            b = be.break_even_allgather(e, 1000.0, 1500.0, N)
            assert be.t_zip_allgather(1.0, N, 1000.0, 1500.0, b, e) == pytest.approx(be.t_nccl(1.0, b))
            assert be.speedup_allgather(1.0, N, 1000.0, 1500.0, 0.9 * b, e) > 1.0
            assert be.speedup_allgather(1.0, N, 1000.0, 1500.0, 1.1 * b, e) < 1.0
