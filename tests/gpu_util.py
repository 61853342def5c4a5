"""Helpers of the GPU parity tests: run the CUDA path through the C ABI and
compare it with the CPU oracle on the same seeded inputs."""
import struct

import numpy as np
import torch


def dev16(x: np.ndarray) -> torch.Tensor:
    """uint16 numpy -> int16 CUDA tensor (raw BF16 bits)."""
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda()


def host16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().view(np.uint16)


def fbits(v: float) -> int:
    return struct.unpack("<Q", struct.pack("<d", v))[0]


def assert_stats_equal(g: dict, o: dict):
    """Every field bit for bit (doubles compared by their bit patterns)."""
    assert np.array_equal(g["hist"], o["hist"]), "histogram"
    for k in ("n", "n_finite", "E0", "rule", "n_escape"):
        assert g[k] == o[k], (k, g[k], o[k])
    for k in ("s1", "s2", "var", "sigma", "K"):
        assert fbits(g[k]) == fbits(o[k]), (k, g[k], o[k])


def slots_equal(gslots: np.ndarray, gsizes, oslots: np.ndarray, osizes, slot: int, W: int):
    gs = [int(s) for s in gsizes]
    os_ = [int(s) for s in osizes]
    assert gs == os_, ("sizes", gs, os_)
    for r in range(W):
        a = gslots[r * slot:r * slot + gs[r]]
        b = oslots[r * slot:r * slot + os_[r]]
        if not np.array_equal(a, b):
            bad = np.nonzero(a != b)[0]
            raise AssertionError(f"payload {r}: {bad.size} bytes differ, first at {bad[:8]}")


def exps(x: np.ndarray) -> np.ndarray:
    return ((x.astype(np.uint32) >> 7) & 0xFF).astype(np.uint8)
