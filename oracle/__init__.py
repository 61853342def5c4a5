"""CPU oracle of the lossless BF16 exponent codecs -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The library itself never does.

The oracle is ``ezoracle.c``: plain single-threaded C that walks the values one
at a time in the order the pages describe (CIERA's exponent-reuse codec and
ZipCCL's 3-bit exponent code; see the header of ``ezoracle.c`` for the byte
layouts and the passages each step follows).  This module only compiles it
with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ezoracle.c")
_SO = os.path.join(_HERE, "libezoracle.so")
_lib = None

BAD_HEADER, BAD_SIZE, BAD_COUNT = 1, 2, 4


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FMA contraction, IEEE doubles)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "ezoracle.h"))):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-Wall", "-ffp-contract=off",
                               "-fno-fast-math", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


class _Stats(ctypes.Structure):
    _fields_ = [("hist", ctypes.c_uint64 * 256), ("n", ctypes.c_uint64),
                ("n_finite", ctypes.c_uint64), ("s1", ctypes.c_double),
                ("s2", ctypes.c_double), ("var", ctypes.c_double),
                ("sigma", ctypes.c_double), ("K", ctypes.c_double),
                ("E0", ctypes.c_uint32), ("rule", ctypes.c_uint32),
                ("n_escape", ctypes.c_uint64)]


class _Fp8Stats(ctypes.Structure):
    _fields_ = [("hist", ctypes.c_uint64 * 32), ("n", ctypes.c_uint64),
                ("n_finite", ctypes.c_uint64), ("s1", ctypes.c_double),
                ("s2", ctypes.c_double), ("var", ctypes.c_double),
                ("sigma", ctypes.c_double), ("K", ctypes.c_double),
                ("E0", ctypes.c_uint32), ("rule", ctypes.c_uint32),
                ("n_escape", ctypes.c_uint64)]


FP8_E5M2, FP8_E4M3 = 1, 2


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        u64, u32, vp, i32 = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_void_p, ctypes.c_int
        sig = {
            "orc_shard_len": (u64, [u64, u32]),
            "orc_shard_count": (u64, [u64, u32, u32]),
            "orc_stats_compute": (i32, [vp, u64, vp]),
            "orc_stats_compute_mode": (i32, [vp, u64, i32, vp]),
            "orc_window_K": (ctypes.c_double, []),
            "orc_window_from_var": (u32, [ctypes.c_double]),
            "orc_code3_chunk_bytes": (u64, [u64, u64]),
            "orc_code3_slot_bytes": (u64, [u64, u32]),
            "orc_code3_encode": (i32, [vp, u64, u32, u32, vp, u64, vp]),
            "orc_code3_encode_chunk": (i32, [vp, u64, u32, u32, u32, vp, u64, vp]),
            "orc_code3_decode": (u32, [vp, vp, u64, u32, vp]),
            "orc_code3_decode_chunk": (u32, [vp, u64, u64, u32, u32, vp]),
            "orc_reuse_bytes": (u64, [u64, u32, u64, i32, u64]),
            "orc_reuse_slot_bytes": (u64, [u64, u32, u32, i32]),
            "orc_reuse_encode": (i32, [vp, u64, u32, u32, vp, i32, i32, vp, vp, u64, vp]),
            "orc_reuse_encode_mode": (i32, [vp, u64, u32, u32, vp, i32, i32, i32, vp, vp, u64, vp]),
            "orc_reuse_encode_hash": (i32, [vp, u64, u32, u32, vp, i32, i32, i32, vp, vp, u64, vp]),
            "orc_splitmix64_next": (u64, [vp]),
            "orc_fp8_stats": (i32, [vp, u64, i32, i32, vp]),
            "orc_fp8_chunk_bytes": (u64, [u64, u64, i32]),
            "orc_fp8_encode": (i32, [vp, u64, u32, i32, u32, vp, u64, vp]),
            "orc_fp8_decode": (u32, [vp, vp, u64, u32, i32, vp]),
            "orc_block_hash": (u64, [vp, u64, u32, u64, i32]),
            "orc_reuse_decode": (u32, [vp, u64, u64, u32, u32, vp, vp]),
            "orc_gather_decode_reuse": (u32, [vp, vp, u64, u32, u32, vp, vp]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def _u16(x) -> np.ndarray:
    """Accept numpy uint16/int16 arrays or torch int16/bfloat16 tensors."""
    if not isinstance(x, np.ndarray):
        import torch
        x = x.detach().cpu().contiguous().view(torch.int16).numpy()
    return np.ascontiguousarray(x).view(np.uint16)


def _map(fn, items, threads: int):
    """fn over items, on `threads` host threads when > 1 (the C calls release
    the GIL; every item touches disjoint parts of the arrays)."""
    items = list(items)
    if threads <= 1 or len(items) <= 1:
        return [fn(i) for i in items]
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=min(threads, len(items))) as ex:
        return list(ex.map(fn, items))


# ----------------------------------------------------------------- geometry

def shard_len(n: int, W: int) -> int:
    return int(lib().orc_shard_len(n, W))


def shard_count(n: int, W: int, r: int) -> int:
    return int(lib().orc_shard_count(n, W, r))


def code3_chunk_bytes(n_c: int, n_esc: int) -> int:
    return int(lib().orc_code3_chunk_bytes(n_c, n_esc))


def code3_slot_bytes(n: int, W: int) -> int:
    return int(lib().orc_code3_slot_bytes(n, W))


def reuse_bytes(n_s: int, B: int, m: int, coded: bool = False, n_esc: int = 0) -> int:
    return int(lib().orc_reuse_bytes(n_s, B, m, int(coded), n_esc))


def reuse_slot_bytes(n: int, W: int, B: int, coded: bool = False) -> int:
    return int(lib().orc_reuse_slot_bytes(n, W, B, int(coded)))


# ----------------------------------------------------------------- stats

def stats(x, window_mode: int = 0) -> dict:
    """window_mode 1: the window from the histogram's densest 7-bin run."""
    x = _u16(x)
    st = _Stats()
    lib().orc_stats_compute_mode(_p(x), x.size, int(window_mode), ctypes.byref(st))
    return _stats_dict(st)


def _stats_dict(st: _Stats) -> dict:
    return {"hist": np.array(st.hist[:], dtype=np.uint64), "n": st.n,
            "n_finite": st.n_finite, "s1": st.s1, "s2": st.s2, "var": st.var,
            "sigma": st.sigma, "K": st.K, "E0": st.E0, "rule": st.rule,
            "n_escape": st.n_escape}


def window_K() -> float:
    return float(lib().orc_window_K())


def window_from_var(var: float) -> int:
    return int(lib().orc_window_from_var(var))


# ----------------------------------------------------------------- code3

def code3_encode(x, W: int, E0: int, threads: int = 1) -> Tuple[np.ndarray, np.ndarray, int]:
    """-> (slots u8[W*slot], sizes u64[W], slot_bytes).  With threads > 1 the
    chunks are encoded by separate single-threaded oracle calls, `threads`
    at a time (same bytes)."""
    x = _u16(x)
    slot = code3_slot_bytes(x.size, W)
    out = np.zeros(W * slot, dtype=np.uint8)
    sizes = np.zeros(W, dtype=np.uint64)
    if threads <= 1:
        rc = lib().orc_code3_encode(_p(x), x.size, W, E0, _p(out), slot, _p(sizes))
        if rc != 0:
            raise ValueError(f"orc_code3_encode failed ({rc})")
        return out, sizes, slot
    n, L = x.size, shard_len(x.size, W)
    buf = x if x.size else np.zeros(1, np.uint16)

    def one(c):
        size = ctypes.c_uint64(0)
        xc = buf[min(c * L, buf.size - 1):]
        rc = lib().orc_code3_encode_chunk(_p(xc), n, W, c, E0, _p(out[c * slot:(c + 1) * slot]),
                                          slot, ctypes.byref(size))
        if rc != 0:
            raise ValueError(f"orc_code3_encode_chunk failed ({rc})")
        sizes[c] = size.value

    _map(one, range(W), threads)
    return out, sizes, slot


def code3_decode(buf: np.ndarray, offsets: np.ndarray, n: int, W: int, threads: int = 1
                 ) -> Tuple[np.ndarray, int]:
    """Decode W chunks laid at offsets (W+1 entries).  With threads > 1 each
    chunk is a separate oracle call, `threads` at a time."""
    buf = np.ascontiguousarray(buf, dtype=np.uint8)
    offsets = np.ascontiguousarray(offsets, dtype=np.uint64)
    out = np.zeros(max(n, 1), dtype=np.uint16)
    if threads <= 1:
        st = lib().orc_code3_decode(_p(buf), _p(offsets), n, W, _p(out))
        return out[:n], int(st)
    L = shard_len(n, W)

    def one(c):
        a, b = int(offsets[c]), int(offsets[c + 1])
        if b < a:
            return BAD_SIZE
        dst = out[min(c * L, out.size - 1):]
        src = buf[min(a, buf.size - 1):]
        return int(lib().orc_code3_decode_chunk(_p(src), b - a, n, W, c, _p(dst)))

    status = 0
    for s in _map(one, range(W), threads):
        status |= s
    return out[:n], status


def code3_decode_chunk(chunk: np.ndarray, n: int, W: int, c: int) -> Tuple[np.ndarray, int]:
    """Chunk c alone (a peer's chunk of an all-to-all), all of its bytes given."""
    chunk = np.ascontiguousarray(chunk, dtype=np.uint8)
    n_c = shard_count(n, W, c)
    out = np.zeros(max(n_c, 1), dtype=np.uint16)
    buf = chunk if chunk.size else np.zeros(1, dtype=np.uint8)
    st = lib().orc_code3_decode_chunk(_p(buf), chunk.size, n, W, c, _p(out))
    return out[:n_c], int(st)


def compact(slots: np.ndarray, sizes: np.ndarray, slot: int
            ) -> Tuple[np.ndarray, np.ndarray]:
    """The receive layout of an allgather of variable-size payloads: payload
    r at the exclusive prefix sum of the sizes."""
    sizes = [int(s) for s in sizes]
    offsets = np.zeros(len(sizes) + 1, dtype=np.uint64)
    offsets[1:] = np.cumsum(sizes)
    recv = np.zeros(max(int(offsets[-1]), 1), dtype=np.uint8)
    for r, s in enumerate(sizes):
        recv[int(offsets[r]):int(offsets[r]) + s] = slots[r * slot:r * slot + s]
    return recv, offsets


# ----------------------------------------------------------------- reuse

def reuse_encode(shard, B: int, shard_index: int, cache: np.ndarray, cold: bool = False,
                 coded: bool = False, window_mode: int = 0) -> Tuple[np.ndarray, Optional[dict]]:
    """Encode one shard; ``cache`` (u8[n_s]) is updated in place."""
    x = _u16(shard)
    assert cache.dtype == np.uint8 and cache.size >= x.size
    nb = -(-x.size // B) if x.size else 0
    cap = reuse_bytes(x.size, B, x.size, coded, x.size if coded else 0)
    out = np.zeros(cap, dtype=np.uint8)
    size = ctypes.c_uint64(0)
    st = _Stats()
    rc = lib().orc_reuse_encode_mode(_p(x), x.size, B, shard_index, _p(cache), int(cold),
                                     int(coded), int(window_mode),
                                     ctypes.byref(st) if coded else None,
                                     _p(out), cap, ctypes.byref(size))
    if rc != 0:
        raise ValueError(f"orc_reuse_encode failed ({rc})")
    del nb
    return out[:size.value].copy(), (_stats_dict(st) if coded else None)


def splitmix64(state: int, count: int) -> list:
    """The first `count` outputs of the SplitMix64 generator from `state`."""
    st = ctypes.c_uint64(state)
    return [int(lib().orc_splitmix64_next(ctypes.byref(st))) for _ in range(count)]


def block_hash(shard, B: int, k: int, s: int) -> int:
    x = _u16(shard)
    buf = x if x.size else np.zeros(1, dtype=np.uint16)
    return int(lib().orc_block_hash(_p(buf), x.size, B, k, s))


def reuse_encode_hash(shard, B: int, shard_index: int, hash_cache: np.ndarray, cold: bool = False,
                      coded: bool = False, window_mode: int = 0) -> Tuple[np.ndarray, Optional[dict]]:
    """Encode one shard with hash-based change detection; ``hash_cache``
    (u64[2 * ceil(n_s / B)]) is updated in place."""
    x = _u16(shard)
    nb = -(-x.size // B) if x.size else 0
    assert hash_cache.dtype == np.uint64 and hash_cache.size >= 2 * nb
    cap = reuse_bytes(x.size, B, x.size, coded, x.size if coded else 0)
    out = np.zeros(cap, dtype=np.uint8)
    size = ctypes.c_uint64(0)
    st = _Stats()
    buf = x if x.size else np.zeros(1, dtype=np.uint16)
    hc = hash_cache if hash_cache.size else np.zeros(2, dtype=np.uint64)
    rc = lib().orc_reuse_encode_hash(_p(buf), x.size, B, shard_index, _p(hc), int(cold), int(coded),
                                     int(window_mode), ctypes.byref(st) if coded else None,
                                     _p(out), cap, ctypes.byref(size))
    if rc != 0:
        raise ValueError(f"orc_reuse_encode_hash failed ({rc})")
    return out[:size.value].copy(), (_stats_dict(st) if coded else None)


def reuse_decode(payload: np.ndarray, n_s: int, B: int, shard_index: int,
                 cache: np.ndarray, avail: Optional[int] = None) -> Tuple[np.ndarray, int]:
    payload = np.ascontiguousarray(payload, dtype=np.uint8)
    if payload.size == 0:
        payload = np.zeros(1, dtype=np.uint8)
        avail = 0
    out = np.zeros(max(n_s, 1), dtype=np.uint16)
    st = lib().orc_reuse_decode(_p(payload), payload.size if avail is None else avail,
                                n_s, B, shard_index, _p(cache), _p(out))
    return out[:n_s], int(st)


def gather_decode_reuse(recv: np.ndarray, offsets: np.ndarray, n: int, W: int, B: int,
                        cache: np.ndarray) -> Tuple[np.ndarray, int]:
    recv = np.ascontiguousarray(recv, dtype=np.uint8)
    offsets = np.ascontiguousarray(offsets, dtype=np.uint64)
    out = np.zeros(max(n, 1), dtype=np.uint16)
    st = lib().orc_gather_decode_reuse(_p(recv), _p(offsets), n, W, B, _p(cache), _p(out))
    return out[:n], int(st)


def reuse_encode_all(x, W: int, B: int, cache: np.ndarray, cold: bool = False,
                     coded: bool = False, window_mode: int = 0, threads: int = 1):
    """Encode all W shards of x (cache u8[n] holds every shard's sender cache),
    one independent single-threaded oracle call per shard, `threads` shards at
    a time.  -> (slots u8[W*slot], sizes u64[W], slot, [stats per shard or None])"""
    x = _u16(x)
    n = x.size
    L = shard_len(n, W)
    slot = reuse_slot_bytes(n, W, B, coded)
    slots = np.zeros(W * slot, dtype=np.uint8)
    sizes = np.zeros(W, dtype=np.uint64)

    def one(r):
        a = min(r * L, n)
        b = min(a + L, n) if a < n else n
        cc = cache[a:b] if b > a else np.zeros(0, np.uint8)
        pay, st = reuse_encode(x[a:b], B, r, cc, cold, coded, window_mode)
        slots[r * slot:r * slot + pay.size] = pay
        sizes[r] = pay.size
        return st

    sts = _map(one, range(W), threads)
    return slots, sizes, slot, sts


def reuse_decode_all(slots: np.ndarray, sizes, slot: int, n: int, W: int, B: int,
                     cache: np.ndarray, threads: int = 1) -> Tuple[np.ndarray, int]:
    """Decode payload r (at slots[r*slot], sizes[r] bytes) of every shard into
    the full tensor against the receiver cache u8[n] (updated in place), one
    oracle call per shard, `threads` shards at a time.  -> (values, OR of the
    shards' status words)"""
    L = shard_len(n, W)
    out = np.zeros(n, dtype=np.uint16)

    def one(r):
        a = min(r * L, n)
        b = min(a + L, n) if a < n else n
        size = int(sizes[r])
        pay = slots[r * slot:r * slot + size]
        cc = cache[a:b] if b > a else np.zeros(0, np.uint8)
        vals, st = reuse_decode(pay, b - a, B, r, cc if cc.size else np.zeros(1, np.uint8))
        out[a:b] = vals
        return st

    sts = _map(one, range(W), threads)
    status = 0
    for s in sts:
        status |= s
    return out, status


# ----------------------------------------------------------------- FP8

def fp8_stats(x, fmt: int, window_mode: int = 0) -> dict:
    """Statistics and window of FP8 values (uint8 bit patterns)."""
    x = np.ascontiguousarray(x, dtype=np.uint8)
    st = _Fp8Stats()
    buf = x if x.size else np.zeros(1, dtype=np.uint8)
    rc = lib().orc_fp8_stats(_p(buf), x.size, fmt, window_mode, ctypes.byref(st))
    if rc != 0:
        raise ValueError("bad FP8 format")
    nb = 32 if fmt == FP8_E5M2 else 16
    return {"hist": np.array(st.hist[:nb], dtype=np.uint64), "n": st.n, "n_finite": st.n_finite,
            "s1": st.s1, "s2": st.s2, "var": st.var, "sigma": st.sigma, "K": st.K, "E0": st.E0,
            "rule": st.rule, "n_escape": st.n_escape}


def fp8_chunk_bytes(n_c: int, n_esc: int, fmt: int) -> int:
    return int(lib().orc_fp8_chunk_bytes(n_c, n_esc, fmt))


def fp8_encode(x, W: int, fmt: int, E0: int) -> Tuple[np.ndarray, np.ndarray, int]:
    """-> (slots u8[W*slot], sizes u64[W], slot_bytes); slot = worst case of one chunk."""
    x = np.ascontiguousarray(x, dtype=np.uint8)
    L = shard_len(x.size, W)
    slot = fp8_chunk_bytes(L, L, fmt)
    out = np.zeros(W * slot, dtype=np.uint8)
    sizes = np.zeros(W, dtype=np.uint64)
    buf = x if x.size else np.zeros(1, dtype=np.uint8)
    rc = lib().orc_fp8_encode(_p(buf), x.size, W, fmt, E0, _p(out), slot, _p(sizes))
    if rc != 0:
        raise ValueError(f"orc_fp8_encode failed ({rc})")
    return out, sizes, slot


def fp8_decode(buf: np.ndarray, offsets: np.ndarray, n: int, W: int, fmt: int) -> Tuple[np.ndarray, int]:
    buf = np.ascontiguousarray(buf, dtype=np.uint8)
    offsets = np.ascontiguousarray(offsets, dtype=np.uint64)
    out = np.zeros(max(n, 1), dtype=np.uint8)
    st = lib().orc_fp8_decode(_p(buf if buf.size else np.zeros(1, np.uint8)), _p(offsets), n, W, fmt,
                              _p(out))
    return out[:n], int(st)
