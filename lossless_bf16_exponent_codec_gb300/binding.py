"""ctypes binding of libexpzip's C ABI (include/expzip.h).

Argument marshalling only: every function here forwards to the C entry point
of the same name.  Device buffers are torch CUDA tensors (their data_ptr is
passed); the stream defaults to torch's current stream.  A missing library
is an error, never a fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libexpzip.so")

EZ_OK, EZ_ERR_ARG, EZ_ERR_CUDA, EZ_ERR_CAPACITY = 0, 1, 2, 3
EZ_ERR_CORRUPT, EZ_ERR_TIMEOUT, EZ_ERR_UNSUPPORTED = 4, 5, 6
EZ_CODEC_CODE3, EZ_CODEC_REUSE, EZ_CODEC_REUSE_CODE3 = 1, 2, 3
EZ_CODEC_FP8_E5M2, EZ_CODEC_FP8_E4M3 = 4, 5
DSTAT_BAD_HEADER, DSTAT_BAD_SIZE, DSTAT_BAD_COUNT = 1, 2, 4
DSTAT_TIMEOUT, DSTAT_MISALIGNED, DSTAT_BAD_STATS = 8, 16, 32
STATS_BYTES = 2120          # sizeof(ez_stats_t)
FP8_STATS_BYTES = 328       # sizeof(ez_fp8_stats_t)
EZ_FLAG_WINDOW_HIST = 1     # plan flag: window from the histogram's densest 7-bin run
EZ_FLAG_HASH_CACHE = 2      # plan flag: sender cache of block hash pairs (reuse codecs, any block size)
NOALLOC_SCRATCH_BYTES = 4 << 20   # EZ_NOALLOC_SCRATCH_BYTES

ENTRY_POINTS = ("ez_plan_create", "ez_plan_destroy", "ez_plan_sizes", "ez_stats",
                "ez_encode_code3", "ez_decode_code3", "ez_encode_reuse", "ez_decode_reuse",
                "ez_gather_decode", "ez_encode_code3_noalloc", "ez_accumulate_bf16",
                "ez_decode_code3_accumulate", "ez_fp8_stats", "ez_fp8_encode", "ez_fp8_decode",
                "ez_status_str", "ez_version")


class EzError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status} ({status_str(status)})")
        self.status = status


class PlanDesc(ctypes.Structure):
    _fields_ = [("n", ctypes.c_uint64), ("W", ctypes.c_uint32), ("B", ctypes.c_uint32),
                ("codec", ctypes.c_uint32), ("flags", ctypes.c_uint32)]


class Sizes(ctypes.Structure):
    _fields_ = [("shard_len", ctypes.c_uint64), ("slot_bytes", ctypes.c_uint64),
                ("workspace_bytes", ctypes.c_uint64), ("cache_bytes", ctypes.c_uint64),
                ("tile_values", ctypes.c_uint64), ("send_cache_bytes", ctypes.c_uint64)]


_lib = None


def lib():
    """Load libexpzip.so; raise if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libexpzip.so is missing ({LIB_PATH}); run build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, u64, u32, i32 = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int
        sig = {
            "ez_plan_create": [ctypes.POINTER(vp), ctypes.POINTER(PlanDesc)],
            "ez_plan_destroy": [vp],
            "ez_plan_sizes": [vp, ctypes.POINTER(Sizes)],
            "ez_stats": [vp, vp, u64, vp, vp, u64, vp],
            "ez_encode_code3": [vp, vp, u32, u32, vp, vp, u64, vp, vp, vp, u64, vp],
            "ez_decode_code3": [vp, vp, vp, u32, u32, vp, vp, vp, u64, vp],
            "ez_encode_reuse": [vp, vp, u32, u32, vp, i32, vp, u64, vp, vp, vp, vp, u64, vp],
            "ez_decode_reuse": [vp, vp, u64, u32, vp, vp, vp, vp, u64, vp],
            "ez_gather_decode": [vp, vp, vp, vp, vp, vp, vp, u64, vp],
            "ez_encode_code3_noalloc": [vp, vp, u32, u32, vp, vp, u64, vp, vp, vp],
            "ez_accumulate_bf16": [vp, vp, u64, i32, vp],
            "ez_decode_code3_accumulate": [vp, vp, vp, u32, u32, vp, i32, vp, vp, u64, vp],
            "ez_fp8_stats": [vp, vp, u64, vp, vp, u64, vp],
            "ez_fp8_encode": [vp, vp, u32, u32, vp, vp, u64, vp, vp, vp, u64, vp],
            "ez_fp8_decode": [vp, vp, vp, u32, u32, vp, vp, vp, u64, vp],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        L.ez_status_str.argtypes = [ctypes.c_int]
        L.ez_status_str.restype = ctypes.c_char_p
        L.ez_version.argtypes = []
        L.ez_version.restype = ctypes.c_uint32
        _lib = L
    return _lib


def status_str(s: int) -> str:
    return lib().ez_status_str(s).decode()


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, rc: int):
    if rc != EZ_OK:
        raise EzError(fn, rc)


# ------------------------------------------------------------------- calls

def ez_plan_create(n: int, W: int, B: int = 0, codec: int = EZ_CODEC_CODE3, flags: int = 0):
    h = ctypes.c_void_p()
    d = PlanDesc(n, W, B, codec, flags)
    _check("ez_plan_create", lib().ez_plan_create(ctypes.byref(h), ctypes.byref(d)))
    return h


def ez_plan_destroy(plan) -> None:
    _check("ez_plan_destroy", lib().ez_plan_destroy(plan))


def ez_plan_sizes(plan) -> dict:
    s = Sizes()
    _check("ez_plan_sizes", lib().ez_plan_sizes(plan, ctypes.byref(s)))
    return {k: int(getattr(s, k)) for k, _ in Sizes._fields_}


def ez_stats(plan, x, n_values: int, stats, ws, ws_bytes: int, stream=None) -> None:
    _check("ez_stats", lib().ez_stats(plan, _ptr(x), n_values, _ptr(stats), _ptr(ws), ws_bytes,
                                      _stream(stream)))


def ez_encode_code3(plan, x, first: int, count: int, stats, out, out_bytes: int, sizes, status,
                    ws, ws_bytes: int, stream=None) -> None:
    _check("ez_encode_code3", lib().ez_encode_code3(plan, _ptr(x), first, count, _ptr(stats),
                                                    _ptr(out), out_bytes, _ptr(sizes),
                                                    _ptr(status), _ptr(ws), ws_bytes,
                                                    _stream(stream)))


def ez_decode_code3(plan, inp, offsets, first: int, count: int, out, status, ws, ws_bytes: int,
                    stream=None) -> None:
    _check("ez_decode_code3", lib().ez_decode_code3(plan, _ptr(inp), _ptr(offsets), first, count,
                                                    _ptr(out), _ptr(status), _ptr(ws), ws_bytes,
                                                    _stream(stream)))


def ez_encode_reuse(plan, x, first: int, count: int, send_cache, cold: bool, out, out_bytes: int,
                    sizes, stats, status, ws, ws_bytes: int, stream=None) -> None:
    _check("ez_encode_reuse", lib().ez_encode_reuse(plan, _ptr(x), first, count, _ptr(send_cache),
                                                    int(bool(cold)), _ptr(out), out_bytes,
                                                    _ptr(sizes), _ptr(stats), _ptr(status),
                                                    _ptr(ws), ws_bytes, _stream(stream)))


def ez_decode_reuse(plan, payload, payload_bytes: int, shard: int, recv_cache, out, status, ws,
                    ws_bytes: int, stream=None) -> None:
    _check("ez_decode_reuse", lib().ez_decode_reuse(plan, _ptr(payload), payload_bytes, shard,
                                                    _ptr(recv_cache), _ptr(out), _ptr(status),
                                                    _ptr(ws), ws_bytes, _stream(stream)))


def ez_gather_decode(plan, recv, offsets, recv_cache, full_out, status, ws, ws_bytes: int,
                     stream=None) -> None:
    _check("ez_gather_decode", lib().ez_gather_decode(plan, _ptr(recv), _ptr(offsets),
                                                      _ptr(recv_cache), _ptr(full_out),
                                                      _ptr(status), _ptr(ws), ws_bytes,
                                                      _stream(stream)))


def ez_encode_code3_noalloc(plan, x, first: int, count: int, stats, out, out_bytes: int, sizes,
                            status, stream=None) -> None:
    _check("ez_encode_code3_noalloc",
           lib().ez_encode_code3_noalloc(plan, _ptr(x), first, count, _ptr(stats), _ptr(out),
                                         out_bytes, _ptr(sizes), _ptr(status), _stream(stream)))


def ez_accumulate_bf16(acc, x, n: int, first: bool, stream=None) -> None:
    _check("ez_accumulate_bf16", lib().ez_accumulate_bf16(_ptr(acc), _ptr(x), n, 1 if first else 0,
                                                          _stream(stream)))


def ez_decode_code3_accumulate(plan, inp, offsets, first: int, count: int, acc, first_source: bool,
                               status, ws, ws_bytes: int, stream=None) -> None:
    _check("ez_decode_code3_accumulate",
           lib().ez_decode_code3_accumulate(plan, _ptr(inp), _ptr(offsets), first, count, _ptr(acc),
                                            1 if first_source else 0, _ptr(status), _ptr(ws), ws_bytes,
                                            _stream(stream)))


def ez_fp8_stats(plan, x, n_values: int, stats, ws, ws_bytes: int, stream=None) -> None:
    _check("ez_fp8_stats", lib().ez_fp8_stats(plan, _ptr(x), n_values, _ptr(stats), _ptr(ws), ws_bytes,
                                              _stream(stream)))


def ez_fp8_encode(plan, x, first: int, count: int, stats, out, out_bytes: int, sizes, status,
                  ws, ws_bytes: int, stream=None) -> None:
    _check("ez_fp8_encode", lib().ez_fp8_encode(plan, _ptr(x), first, count, _ptr(stats), _ptr(out),
                                                out_bytes, _ptr(sizes), _ptr(status), _ptr(ws), ws_bytes,
                                                _stream(stream)))


def ez_fp8_decode(plan, inp, offsets, first: int, count: int, out, status, ws, ws_bytes: int,
                  stream=None) -> None:
    _check("ez_fp8_decode", lib().ez_fp8_decode(plan, _ptr(inp), _ptr(offsets), first, count, _ptr(out),
                                                _ptr(status), _ptr(ws), ws_bytes, _stream(stream)))


def ez_version() -> int:
    return int(lib().ez_version())


# ------------------------------------------------------------ host helpers

def parse_stats(raw) -> dict:
    """Decode an ez_stats_t record (bytes / uint8 numpy / uint8 tensor)."""
    if not isinstance(raw, np.ndarray):
        try:
            raw = raw.detach().cpu().numpy()
        except AttributeError:
            raw = np.frombuffer(bytes(raw), dtype=np.uint8)
    b = np.ascontiguousarray(np.ascontiguousarray(raw, dtype=np.uint8)[:STATS_BYTES])
    hist = b[:2048].view(np.uint64).copy()
    q = b[2048:2104].view(np.uint64)
    d = b[2064:2104].view(np.float64)
    u32 = b[2104:2112].view(np.uint32)
    return {"hist": hist, "n": int(q[0]), "n_finite": int(q[1]), "s1": float(d[0]),
            "s2": float(d[1]), "var": float(d[2]), "sigma": float(d[3]), "K": float(d[4]),
            "E0": int(u32[0]), "rule": int(u32[1]),
            "n_escape": int(b[2112:2120].view(np.uint64)[0])}


def parse_fp8_stats(raw) -> dict:
    """Decode an ez_fp8_stats_t record (bytes / uint8 numpy / uint8 tensor)."""
    if not isinstance(raw, np.ndarray):
        try:
            raw = raw.detach().cpu().numpy()
        except AttributeError:
            raw = np.frombuffer(bytes(raw), dtype=np.uint8)
    b = np.ascontiguousarray(np.ascontiguousarray(raw, dtype=np.uint8)[:FP8_STATS_BYTES])
    q = b[256:272].view(np.uint64)
    d = b[272:312].view(np.float64)
    u32 = b[312:320].view(np.uint32)
    return {"hist": b[:256].view(np.uint64).copy(), "n": int(q[0]), "n_finite": int(q[1]),
            "s1": float(d[0]), "s2": float(d[1]), "var": float(d[2]), "sigma": float(d[3]),
            "K": float(d[4]), "E0": int(u32[0]), "rule": int(u32[1]),
            "n_escape": int(b[320:328].view(np.uint64)[0])}
