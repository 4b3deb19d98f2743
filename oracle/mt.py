"""The CPU oracle's steps over several host threads -- TEST AND BASELINE INFRASTRUCTURE.

``huff_oracle_mt.c`` runs the same per-chunk steps as the sequential oracle
(bit counts, a prefix sum, bit-at-a-time packing; bit-at-a-time canonical
decoding) over contiguous ranges of chunks on POSIX threads, so the oracle
can be timed on all of a host's cores beside the 16-core CPU figures of
"Lossless Compression for LLM Tensor Incremental Snapshots" (English
abstract, experiment highlights).  Its payload equals the sequential
oracle's byte for byte.  Only the tests and the benchmark's CPU baseline use
it; the GPU library never does.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from . import OracleError, _ptr, _u8, code_lengths, canonical_codes

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "huff_oracle_mt.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_mt.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``huff_oracle_mt.c`` into ``liboracle_mt.so`` (plain gcc, -O2, POSIX threads)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=gnu99", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u8p = ctypes.POINTER(ctypes.c_uint8)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        u32p = ctypes.POINTER(ctypes.c_uint32)
        u64p = ctypes.POINTER(ctypes.c_uint64)
        u64, i = ctypes.c_uint64, ctypes.c_int
        lib.mt_histogram.argtypes = [u8p, u64, u64p, i]
        lib.mt_histogram.restype = i
        lib.mt_delta_split.argtypes = [u16p, u16p, u64, u8p, u8p, i]
        lib.mt_delta_split.restype = None
        lib.mt_merge_xor.argtypes = [u8p, u8p, u16p, u64, u16p, i]
        lib.mt_merge_xor.restype = None
        lib.mt_encode.argtypes = [u8p, u64, u8p, u32p, u64, u8p, u64, u64p, i]
        lib.mt_encode.restype = i
        lib.mt_decode.argtypes = [u8p, u64, u64p, u64, u64, u8p, u8p, i]
        lib.mt_decode.restype = i
        _lib = lib
    return _lib


def histogram(data, threads: int) -> np.ndarray:
    buf = _u8(data)
    h = np.zeros(256, dtype=np.uint64)
    if buf.size:
        _load().mt_histogram(_ptr(buf, ctypes.c_uint8), buf.size, _ptr(h, ctypes.c_uint64), threads)
    return h


def delta_split(a, b, threads: int):
    """(hi, lo) planes of a (XOR b when b is not None); a, b uint16 arrays."""
    a16 = np.ascontiguousarray(np.asarray(a).view(np.uint16).reshape(-1))
    n = a16.size
    hi = np.empty(max(n, 1), dtype=np.uint8)
    lo = np.empty(max(n, 1), dtype=np.uint8)
    if n:
        bp = None
        if b is not None:
            b16 = np.ascontiguousarray(np.asarray(b).view(np.uint16).reshape(-1))
            assert b16.size == n
            bp = _ptr(b16, ctypes.c_uint16)
        _load().mt_delta_split(_ptr(a16, ctypes.c_uint16), bp, n, _ptr(hi, ctypes.c_uint8), _ptr(lo, ctypes.c_uint8),
                               threads)
    return hi[:n], lo[:n]


def merge_xor(hi, lo, b, threads: int) -> np.ndarray:
    h, l = _u8(hi), _u8(lo)
    n = h.size
    w = np.empty(max(n, 1), dtype=np.uint16)
    if n:
        bp = None
        if b is not None:
            b16 = np.ascontiguousarray(np.asarray(b).view(np.uint16).reshape(-1))
            bp = _ptr(b16, ctypes.c_uint16)
        _load().mt_merge_xor(_ptr(h, ctypes.c_uint8), _ptr(l, ctypes.c_uint8), bp, n, _ptr(w, ctypes.c_uint16),
                             threads)
    return w[:n]


def encode(data, lengths, codes, chunk_bytes: int, threads: int):
    """Returns (payload uint8[ceil(T/8)], offsets uint64[n_chunks + 1]), as oracle.encode."""
    buf = _u8(data)
    n = buf.size
    ln = _u8(lengths)
    cd = np.ascontiguousarray(np.asarray(codes, dtype=np.uint32))
    cap = max((n * int(ln.max(initial=0)) + 7) // 8 + 1, 1)
    payload = np.empty(cap, dtype=np.uint8)
    off = np.zeros((n + chunk_bytes - 1) // chunk_bytes + 1, dtype=np.uint64)
    src = buf if n else np.zeros(1, np.uint8)
    st = _load().mt_encode(_ptr(src, ctypes.c_uint8), n, _ptr(ln, ctypes.c_uint8), _ptr(cd, ctypes.c_uint32),
                           chunk_bytes, _ptr(payload, ctypes.c_uint8), cap, _ptr(off, ctypes.c_uint64), threads)
    if st != 0:
        raise OracleError("mt_encode", st)
    return payload[: (int(off[-1]) + 7) // 8], off


def decode(payload, offsets, n: int, chunk_bytes: int, lengths, threads: int) -> np.ndarray:
    pl = _u8(payload)
    pbytes = pl.size
    if pl.size == 0:
        pl = np.zeros(1, dtype=np.uint8)
    off = np.ascontiguousarray(np.asarray(offsets, dtype=np.uint64))
    ln = _u8(lengths)
    out = np.empty(max(n, 1), dtype=np.uint8)
    st = _load().mt_decode(_ptr(pl, ctypes.c_uint8), pbytes, _ptr(off, ctypes.c_uint64), n, chunk_bytes,
                           _ptr(ln, ctypes.c_uint8), _ptr(out, ctypes.c_uint8), threads)
    if st != 0:
        raise OracleError("mt_decode", st)
    return out[:n]


def snapshot_round_trip(x0, x1, chunk_bytes: int, threads: int):
    """The whole snapshot path on host threads: delta + planes, histograms, codebooks (the sequential
    oracle's), encode, decode, merge + delta.  Returns (compressed bytes, seconds to compress, seconds
    to decompress); raises if the round trip is not exact."""
    import time
    t0 = time.perf_counter()
    hi, lo = delta_split(x1, x0, threads)
    streams = []
    for p in (hi, lo):
        ln = code_lengths(histogram(p, threads))
        pay, off = encode(p, ln, canonical_codes(ln), chunk_bytes, threads)
        streams.append((pay, off, ln))
    t1 = time.perf_counter()
    planes = [decode(pay, off, hi.size, chunk_bytes, ln, threads) for pay, off, ln in streams]
    back = merge_xor(planes[0], planes[1], x0, threads)
    t2 = time.perf_counter()
    if not np.array_equal(back, np.asarray(x1).view(np.uint16).reshape(-1)):
        raise RuntimeError("multi-threaded oracle round trip differs")
    return sum(p.size for p, _, _ in streams), t1 - t0, t2 - t1
