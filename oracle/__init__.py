"""CPU oracle for canonical Huffman coding of tensor bytes -- TEST INFRASTRUCTURE.

This package is the independent yardstick for the GPU library.  Only the test
suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import it; the product path never does.  It shares no code with the CUDA
library: ``huff_oracle.c`` is a plain sequential C restatement of the method,
``tiny.py`` a second, pure-Python one for small inputs.

Sources followed (page title and section):
  * "Single-stage Huffman encoder for ML compression" (arXiv 2601.10673),
    Methodology steps 1-4 (histogram, averaged distribution, one-time codebook,
    single-stage encode).
  * "Lossless Compression for LLM Tensor Incremental Snapshots" (arXiv
    2505.09810), Method details / technical framework and English abstract
    (byte grouping, per-group statistics and Huffman coding, decompression in
    reverse, incremental delta).
  * RFC 1951 section 3.2.2 (canonical codes) and ITU-T T.81 Annex K.3
    (Adjust_BITS length limiting) for the steps the pages leave open.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "huff_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

REF_OK = 0
REF_ERR_INVALID_ARG = -1
REF_ERR_BUFFER_TOO_SMALL = -2
REF_ERR_SYMBOL_NOT_IN_CODEBOOK = -3
REF_ERR_CORRUPT_STREAM = -4
REF_COVER_ALL = 1


class OracleError(RuntimeError):
    """A non-zero status from an oracle routine."""

    def __init__(self, name: str, status: int):
        super().__init__(f"oracle {name} returned {status}")
        self.status = status


def build(force: bool = False) -> str:
    """Compile ``huff_oracle.c`` into ``liboracle.so`` (plain gcc, -O2)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    from . import mt
    mt.build(force)
    return _LIB_PATH


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u8p = ctypes.POINTER(ctypes.c_uint8)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        u32p = ctypes.POINTER(ctypes.c_uint32)
        u64p = ctypes.POINTER(ctypes.c_uint64)
        u64 = ctypes.c_uint64
        lib.ref_histogram.argtypes = [u8p, u64, u64, u64p]
        lib.ref_histogram.restype = None
        lib.ref_code_lengths.argtypes = [u64p, ctypes.c_int, ctypes.c_uint, u8p]
        lib.ref_code_lengths.restype = ctypes.c_int
        lib.ref_canonical_codes.argtypes = [u8p, u32p]
        lib.ref_canonical_codes.restype = ctypes.c_int
        lib.ref_encode.argtypes = [u8p, u64, u8p, u32p, u64, u8p, u64, u64p]
        lib.ref_encode.restype = ctypes.c_int
        lib.ref_decode.argtypes = [u8p, u64, u64p, u64, u64, u8p, u8p]
        lib.ref_decode.restype = ctypes.c_int
        lib.ref_bytegroup_split.argtypes = [u16p, u64, u8p, u8p]
        lib.ref_bytegroup_split.restype = None
        lib.ref_bytegroup_merge.argtypes = [u8p, u8p, u64, u16p]
        lib.ref_bytegroup_merge.restype = None
        lib.ref_delta_xor.argtypes = [u16p, u16p, u64, u16p]
        lib.ref_delta_xor.restype = None
        lib.ref_entropy.argtypes = [u64p]
        lib.ref_entropy.restype = ctypes.c_double
        lib.ref_total_bits.argtypes = [u64p, u8p]
        lib.ref_total_bits.restype = ctypes.c_uint64
        _lib = lib
    return _lib


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"], "oracle wants contiguous arrays"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _u8(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.uint8:
        a = a.view(np.uint8) if a.dtype == np.int8 else a.astype(np.uint8)
    return np.ascontiguousarray(a).reshape(-1)


def histogram(data, stride: int = 1, n: int | None = None) -> np.ndarray:
    """C1: 256-bin byte histogram of ``data[0], data[stride], ...`` (n elements)."""
    buf = _u8(data)
    if n is None:
        n = (buf.size + stride - 1) // stride if buf.size else 0
    assert n == 0 or (n - 1) * stride < buf.size
    hist = np.zeros(256, dtype=np.uint64)
    _load().ref_histogram(_ptr(buf, ctypes.c_uint8), n, stride, _ptr(hist, ctypes.c_uint64))
    return hist


def code_lengths(hist, max_len: int = 24, flags: int = 0) -> np.ndarray:
    """C3-C5: Huffman lengths with the (count, id) tie-break, limited to max_len."""
    h = np.ascontiguousarray(np.asarray(hist, dtype=np.uint64).reshape(256))
    out = np.zeros(256, dtype=np.uint8)
    st = _load().ref_code_lengths(_ptr(h, ctypes.c_uint64), max_len, flags, _ptr(out, ctypes.c_uint8))
    if st != REF_OK:
        raise OracleError("code_lengths", st)
    return out


def canonical_codes(lengths) -> np.ndarray:
    """C6: canonical (RFC 1951 3.2.2) right-aligned codes for 256 lengths."""
    ln = _u8(lengths)
    assert ln.size == 256
    code = np.zeros(256, dtype=np.uint32)
    st = _load().ref_canonical_codes(_ptr(ln, ctypes.c_uint8), _ptr(code, ctypes.c_uint32))
    if st != REF_OK:
        raise OracleError("canonical_codes", st)
    return code


def encode(data, lengths, codes, chunk_bytes: int, cap: int | None = None):
    """C7: returns (payload uint8[ceil(T/8)], offsets uint64[n_chunks + 1])."""
    buf = _u8(data)
    n = buf.size
    ln = _u8(lengths)
    cd = np.ascontiguousarray(np.asarray(codes, dtype=np.uint32))
    if cap is None:
        cap = (n * int(ln.max(initial=0)) + 7) // 8 + 1
    payload = np.zeros(max(cap, 1), dtype=np.uint8)
    n_chunks = (n + chunk_bytes - 1) // chunk_bytes
    off = np.zeros(n_chunks + 1, dtype=np.uint64)
    st = _load().ref_encode(_ptr(buf, ctypes.c_uint8), n, _ptr(ln, ctypes.c_uint8),
                            _ptr(cd, ctypes.c_uint32), chunk_bytes, _ptr(payload, ctypes.c_uint8),
                            cap, _ptr(off, ctypes.c_uint64))
    if st != REF_OK:
        raise OracleError("encode", st)
    total = int(off[-1])
    return payload[: (total + 7) // 8].copy(), off


def decode(payload, offsets, n: int, chunk_bytes: int, lengths) -> np.ndarray:
    """C8: decode n symbols chunk by chunk; raises on a corrupt stream."""
    pl = _u8(payload)
    if pl.size == 0:
        pl = np.zeros(1, dtype=np.uint8)
        pbytes = 0
    else:
        pbytes = pl.size
    off = np.ascontiguousarray(np.asarray(offsets, dtype=np.uint64))
    ln = _u8(lengths)
    out = np.zeros(max(n, 1), dtype=np.uint8)
    st = _load().ref_decode(_ptr(pl, ctypes.c_uint8), pbytes, _ptr(off, ctypes.c_uint64), n,
                            chunk_bytes, _ptr(ln, ctypes.c_uint8), _ptr(out, ctypes.c_uint8))
    if st != REF_OK:
        raise OracleError("decode", st)
    return out[:n]


def bytegroup_split(w):
    """C9: (hi, lo) byte planes of a little-endian 16-bit array."""
    w16 = np.ascontiguousarray(np.asarray(w).view(np.uint16).reshape(-1))
    n = w16.size
    hi = np.zeros(max(n, 1), dtype=np.uint8)
    lo = np.zeros(max(n, 1), dtype=np.uint8)
    _load().ref_bytegroup_split(_ptr(w16, ctypes.c_uint16) if n else _ptr(np.zeros(1, np.uint16), ctypes.c_uint16),
                                n, _ptr(hi, ctypes.c_uint8), _ptr(lo, ctypes.c_uint8))
    return hi[:n], lo[:n]


def bytegroup_merge(hi, lo) -> np.ndarray:
    """C9: 16-bit words from (hi, lo) byte planes."""
    h = _u8(hi)
    l = _u8(lo)
    assert h.size == l.size
    n = h.size
    w = np.zeros(max(n, 1), dtype=np.uint16)
    if n:
        _load().ref_bytegroup_merge(_ptr(h, ctypes.c_uint8), _ptr(l, ctypes.c_uint8), n, _ptr(w, ctypes.c_uint16))
    return w[:n]


def drift_gap(hist, lengths) -> float:
    """Drift of a shard against a codebook (P1 Limitations: distribution drift under a fixed codebook):
    T = sum h * len bits under the codebook, bound B = n * max(H, 1) with H the shard's own entropy
    (at least one bit per symbol for a Huffman code of bytes); gap = (T - B) / B, infinite when a
    present symbol has no code, 0 for an empty shard."""
    h = np.asarray(hist, dtype=np.uint64)
    ln = np.asarray(lengths, dtype=np.uint64)
    if np.any((h > 0) & (ln == 0)):
        return float("inf")
    n = int(h.sum())
    if n == 0:
        return 0.0
    T = sum(int(a) * int(b) for a, b in zip(h, ln))
    H = 0.0
    for c in h:
        if c:
            p = float(c) / n
            H -= p * np.log2(p)
    B = n * max(H, 1.0)
    return (T - B) / B


def bytegroup_split_w(data, width: int) -> list:
    """Byte planes of width-byte little-endian words (P2 byte grouping for other
    element widths): plane p is byte width-1-p of every word, most significant first."""
    b = np.ascontiguousarray(np.asarray(data).view(np.uint8).reshape(-1))
    assert b.size % width == 0
    words = b.reshape(-1, width)
    return [np.ascontiguousarray(words[:, width - 1 - p]) for p in range(width)]


def bytegroup_merge_w(planes) -> np.ndarray:
    """The words' bytes (little endian) from their byte planes, most significant plane first."""
    width = len(planes)
    n = np.asarray(planes[0]).size
    out = np.empty((n, width), dtype=np.uint8)
    for p in range(width):
        out[:, width - 1 - p] = np.asarray(planes[p], dtype=np.uint8)
    return out.reshape(-1)


def delta_xor(a, b) -> np.ndarray:
    """C9: bitwise XOR of two 16-bit snapshots."""
    a16 = np.ascontiguousarray(np.asarray(a).view(np.uint16).reshape(-1))
    b16 = np.ascontiguousarray(np.asarray(b).view(np.uint16).reshape(-1))
    assert a16.size == b16.size
    n = a16.size
    out = np.zeros(max(n, 1), dtype=np.uint16)
    if n:
        _load().ref_delta_xor(_ptr(a16, ctypes.c_uint16), _ptr(b16, ctypes.c_uint16), n, _ptr(out, ctypes.c_uint16))
    return out[:n]


def entropy(hist) -> float:
    """C10: Shannon entropy, bits per symbol, in double."""
    h = np.ascontiguousarray(np.asarray(hist, dtype=np.uint64).reshape(256))
    return float(_load().ref_entropy(_ptr(h, ctypes.c_uint64)))


def total_bits(hist, lengths) -> int:
    """Closed form T = sum_s hist[s] * len[s]."""
    h = np.ascontiguousarray(np.asarray(hist, dtype=np.uint64).reshape(256))
    ln = _u8(lengths)
    return int(_load().ref_total_bits(_ptr(h, ctypes.c_uint64), _ptr(ln, ctypes.c_uint8)))


def compress_plane(data, chunk_bytes: int, max_len: int = 24, flags: int = 0, hist=None):
    """Per-shard pipeline on one byte stream: histogram -> lengths -> codes -> encode."""
    if hist is None:
        hist = histogram(data)
    ln = code_lengths(hist, max_len, flags)
    cd = canonical_codes(ln)
    payload, off = encode(data, ln, cd, chunk_bytes)
    return ln, cd, payload, off
