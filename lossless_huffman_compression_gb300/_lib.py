"""ctypes binding of libhuff (include/huff.h) -- argument marshalling only.

Every function here has the name of the C entry point it calls.  Device
buffers are torch CUDA tensors (contiguous); the work is enqueued on the
current torch CUDA stream unless a stream is passed.  A non-zero synchronous
status raises HuffError.  Asynchronous device errors land in the caller's
``status`` tensor (int32, device), as in the C ABI.

There is no CPU fallback: when libhuff.so is missing or cannot be loaded,
every call raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libhuff.so")

HUFF_OK = 0
HUFF_ERR_INVALID_ARG = -1
HUFF_ERR_BUFFER_TOO_SMALL = -2
HUFF_ERR_SYMBOL_NOT_IN_CODEBOOK = -3
HUFF_ERR_CORRUPT_STREAM = -4
HUFF_ERR_TIMEOUT = -5
HUFF_ERR_CUDA = -6
HUFF_ERR_INVALID_CODEBOOK = -7
HUFF_MAX_LEN = 24
HUFF_COVER_ALL = 1
HUFF_CHUNK_ALIGN = 32
HUFF_CODEBOOK_MAGIC = 0x48554642
HUFF_NOALLOC_MAX_SYMBOLS = 1 << 30
HUFF_COUNT_SEGMENT = 131072
CODEBOOK_LEN_OFFSET = 16  # byte offset of len[256] inside huff_codebook
HUFF_CONTAINER_MAGIC = 0x43465548
HUFF_CONTAINER_HEADER = 48
HUFF_CONTAINER_LENGTHS = 1

EXPORTS = (
    "huff_version", "huff_status_string", "huff_codebook_size", "huff_encode_bound", "huff_workspace_size",
    "huff_num_chunks", "huff_histogram", "huff_build_codebook", "huff_codebook_from_lengths", "huff_encode",
    "huff_decode", "huff_encode_noalloc", "lmc_bytegroup_split", "lmc_bytegroup_merge", "lmc_delta_xor", "lmc_histogram_bf16",
    "lmc_workspace_size", "lmc_encode_bf16", "lmc_decode_bf16", "huff_code_stats", "lmc_segment_counts_size",
    "lmc_count_segment", "lmc_counted_workspace_size", "lmc_histogram_bf16_counted", "lmc_encode_bf16_counted", "lmc_bytegroup_split_w",
    "lmc_bytegroup_merge_w", "huff_drift_check", "huff_build_codebook_if", "huff_build_codebooks",
    "huff_stream_copy", "huff_container_size", "huff_container_write", "huff_container_parse", "huff_debug_wait",
    "huff_pick_chunk",
)


class HuffError(RuntimeError):
    def __init__(self, name: str, status: int):
        super().__init__(f"{name}: {status_string(status)} ({status})")
        self.status = status


class HuffStats(ctypes.Structure):
    _fields_ = [("n", ctypes.c_uint64), ("total_bits", ctypes.c_uint64), ("entropy_bits", ctypes.c_double),
                ("mean_len", ctypes.c_double), ("shannon_gap", ctypes.c_double)]


class HuffContainerView(ctypes.Structure):
    _fields_ = [("n", ctypes.c_uint64), ("chunk_bytes", ctypes.c_uint64), ("n_chunks", ctypes.c_uint64),
                ("total_bits", ctypes.c_uint64), ("max_len", ctypes.c_int32), ("has_lengths", ctypes.c_int32),
                ("len", ctypes.c_void_p), ("off", ctypes.c_void_p), ("payload", ctypes.c_void_p),
                ("payload_bytes", ctypes.c_uint64)]


_lib = None


def load(path: str = LIB_PATH):
    """Load libhuff.so (built by __graft_entry__.build()); raises if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libhuff.so not found at {path}: build it first "
                           "(python -m lossless_huffman_compression_gb300.build)")
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    S = ctypes.c_size_t
    I = ctypes.c_int
    sig = {
        "huff_version": (ctypes.c_uint32, []),
        "huff_status_string": (ctypes.c_char_p, [I]),
        "huff_codebook_size": (S, []),
        "huff_encode_bound": (S, [S, I]),
        "huff_workspace_size": (S, [S, S]),
        "lmc_workspace_size": (S, [S, S]),
        "huff_num_chunks": (S, [S, S]),
        "huff_histogram": (I, [P, S, S, P, I, P]),
        "huff_build_codebook": (I, [P, I, ctypes.c_uint, P, P, P]),
        "huff_build_codebooks": (I, [P, S, I, ctypes.c_uint, P, P, P]),
        "huff_stream_copy": (I, [P, S, P, S, P, S, P, P, P]),
        "huff_codebook_from_lengths": (I, [P, I, P, P, P]),
        "huff_encode": (I, [P, S, P, S, P, S, P, P, S, P, P]),
        "huff_decode": (I, [P, S, P, S, S, P, P, P, P]),
        "huff_encode_noalloc": (I, [P, S, P, S, P, S, P, P, P]),
        "lmc_bytegroup_split": (I, [P, S, P, P, P]),
        "lmc_bytegroup_merge": (I, [P, P, S, P, P]),
        "lmc_delta_xor": (I, [P, P, S, P, P]),
        "lmc_histogram_bf16": (I, [P, P, S, P, P, I, P]),
        "lmc_encode_bf16": (I, [P, P, S, P, P, S, P, S, P, P, S, P, P, S, P, P]),
        "lmc_decode_bf16": (I, [P, S, P, P, S, P, S, S, P, P, P, P, P, P]),
        "huff_code_stats": (I, [P, P, ctypes.POINTER(HuffStats)]),
        "huff_container_size": (S, [S, S, ctypes.c_uint64, I]),
        "huff_container_write": (I, [P, S, S, S, I, P, P, P, ctypes.POINTER(S)]),
        "huff_container_parse": (I, [P, S, ctypes.POINTER(HuffContainerView)]),
        "lmc_segment_counts_size": (S, [S]),
        "lmc_count_segment": (S, [S]),
        "huff_drift_check": (I, [P, P, ctypes.c_double, P, P, P]),
        "huff_build_codebook_if": (I, [P, P, I, ctypes.c_uint, P, P, P]),
        "lmc_bytegroup_split_w": (I, [P, S, I, P, S, P]),
        "lmc_bytegroup_merge_w": (I, [P, S, I, S, P, P]),
        "lmc_counted_workspace_size": (S, [S]),
        "lmc_histogram_bf16_counted": (I, [P, P, S, P, P, P, S, P]),
        "lmc_encode_bf16_counted": (I, [P, P, S, P, P, S, P, S, P, S, P, P, S, P, P, S, P, P]),
        "huff_debug_wait": (I, [I, P, S, ctypes.c_uint32, ctypes.c_uint32, P, P, P]),
        "huff_pick_chunk": (S, [S, I]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load().huff_status_string(int(status)).decode()
    except Exception:  # library not loadable: still give a message
        return f"status {status}"


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor | None, name: str):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _check(name: str, st: int):
    if st != HUFF_OK:
        raise HuffError(name, st)


# ---------------------------------------------------------------- queries
def huff_version() -> int:
    return int(load().huff_version())


def huff_status_string(status: int) -> str:
    return status_string(status)


def huff_codebook_size() -> int:
    return int(load().huff_codebook_size())


def huff_encode_bound(n: int, max_len: int = HUFF_MAX_LEN) -> int:
    return int(load().huff_encode_bound(n, max_len))


def huff_workspace_size(n: int, chunk_bytes: int) -> int:
    return int(load().huff_workspace_size(n, chunk_bytes))


def huff_pick_chunk(n: int, delta: bool = False) -> int:
    """The smallest chunk size that gives the decode one wave of full blocks on every SM; delta: the
    stream is decoded with an XOR delta (see include/huff.h)."""
    c = int(load().huff_pick_chunk(n, 1 if delta else 0))
    if c == 0:
        raise HuffError("huff_pick_chunk", HUFF_ERR_CUDA)
    return c


def lmc_workspace_size(n: int, chunk_bytes: int) -> int:
    return int(load().lmc_workspace_size(n, chunk_bytes))


def lmc_count_segment(n: int) -> int:
    """Elements per counted segment for n elements on the current device (see include/huff.h)."""
    return int(load().lmc_count_segment(n))


def lmc_segment_counts_size(n: int) -> int:
    return int(load().lmc_segment_counts_size(n))


def lmc_counted_workspace_size(n: int) -> int:
    return int(load().lmc_counted_workspace_size(n))


def huff_num_chunks(n: int, chunk_bytes: int) -> int:
    return int(load().huff_num_chunks(n, chunk_bytes))


# ---------------------------------------------------------------- device calls
def huff_histogram(inp: torch.Tensor, hist: torch.Tensor, n: int | None = None, stride: int = 1,
                   accumulate: bool = False, offset: int = 0, stream=None) -> torch.Tensor:
    """256-bin histogram of n symbols at byte `offset` of inp with the given stride."""
    if n is None:
        n = (inp.numel() * inp.element_size() - offset + stride - 1) // stride
    base = _dev(inp, "inp") + offset
    _check("huff_histogram", load().huff_histogram(base, n, stride, _dev(hist, "hist"), int(bool(accumulate)),
                                                   _stream(stream)))
    return hist


def huff_build_codebook(hist: torch.Tensor, cb: torch.Tensor, status: torch.Tensor, max_len: int = HUFF_MAX_LEN,
                        flags: int = 0, stream=None) -> torch.Tensor:
    _check("huff_build_codebook", load().huff_build_codebook(_dev(hist, "hist"), max_len, flags, _dev(cb, "cb"),
                                                             _dev(status, "status"), _stream(stream)))
    return cb


def huff_build_codebooks(hists: torch.Tensor, cbs: torch.Tensor, status: torch.Tensor, max_len: int = HUFF_MAX_LEN,
                         flags: int = 0, stream=None) -> torch.Tensor:
    """hists: int64 [count, 256]; cbs: uint8 [count, huff_codebook_size()], contiguous."""
    count = hists.numel() // 256
    if hists.numel() != 256 * count or cbs.numel() != count * huff_codebook_size():
        raise ValueError("hists must be [count, 256] and cbs [count, codebook size]")
    _check("huff_build_codebooks", load().huff_build_codebooks(_dev(hists, "hists"), count, max_len, flags,
                                                               _dev(cbs, "cbs"), _dev(status, "status"),
                                                               _stream(stream)))
    return cbs


def huff_stream_copy(payload: torch.Tensor, off: torch.Tensor, dst_payload: torch.Tensor, dst_off: torch.Tensor,
                     status: torch.Tensor, stream=None) -> None:
    """Copy a stream (payload bytes up to its device-side size, and its offsets) to dst buffers."""
    n_chunks = off.numel() - 1
    if n_chunks < 0 or dst_off.numel() != off.numel():
        raise ValueError("dst_off must have as many entries as off")
    _check("huff_stream_copy", load().huff_stream_copy(_dev(payload, "payload"),
                                                       payload.numel() * payload.element_size(), _dev(off, "off"),
                                                       n_chunks,
                                                       _dev(dst_payload, "dst_payload"),
                                                       dst_payload.numel() * dst_payload.element_size(),
                                                       _dev(dst_off, "dst_off"), _dev(status, "status"),
                                                       _stream(stream)))


def huff_codebook_from_lengths(lengths, cb: torch.Tensor, status: torch.Tensor, max_len: int = HUFF_MAX_LEN,
                               stream=None) -> torch.Tensor:
    h = np.ascontiguousarray(np.asarray(lengths, dtype=np.uint8).reshape(256))
    _check("huff_codebook_from_lengths",
           load().huff_codebook_from_lengths(h.ctypes.data, max_len, _dev(cb, "cb"), _dev(status, "status"),
                                             _stream(stream)))
    return cb


def huff_encode(inp: torch.Tensor, cb: torch.Tensor, chunk_bytes: int, payload: torch.Tensor, off: torch.Tensor,
                ws: torch.Tensor, status: torch.Tensor, n: int | None = None, stream=None):
    if n is None:
        n = inp.numel() * inp.element_size()
    _check("huff_encode", load().huff_encode(
        _dev(inp, "inp"), n, _dev(cb, "cb"), chunk_bytes, _dev(payload, "payload"),
        payload.numel() * payload.element_size(), _dev(off, "off"), _dev(ws, "ws"),
        ws.numel() * ws.element_size(), _dev(status, "status"), _stream(stream)))


def huff_encode_noalloc(inp: torch.Tensor, cb: torch.Tensor, chunk_bytes: int, payload: torch.Tensor,
                        off: torch.Tensor, status: torch.Tensor, n: int | None = None, stream=None):
    """huff_encode without a workspace argument (the library's built-in scratch is used)."""
    if n is None:
        n = inp.numel() * inp.element_size()
    _check("huff_encode_noalloc", load().huff_encode_noalloc(
        _dev(inp, "inp"), n, _dev(cb, "cb"), chunk_bytes, _dev(payload, "payload"),
        payload.numel() * payload.element_size(), _dev(off, "off"), _dev(status, "status"), _stream(stream)))


def huff_debug_wait(kind: int, desc, seg: int, limit: int, out: torch.Tensor, status: torch.Tensor, stream=None):
    """Test hook: one bounded device wait run on its own (kind 0: lookback over desc, kind 1: an mbarrier)."""
    _check("huff_debug_wait", load().huff_debug_wait(
        kind, None if desc is None else _dev(desc, "desc"), 0 if desc is None else desc.numel(), seg, limit,
        _dev(out, "out"), _dev(status, "status"), _stream(stream)))


def huff_decode(payload: torch.Tensor, off: torch.Tensor, n: int, chunk_bytes: int, cb: torch.Tensor,
                out: torch.Tensor, status: torch.Tensor, payload_bytes: int | None = None, stream=None):
    if payload_bytes is None:
        payload_bytes = payload.numel() * payload.element_size()
    _check("huff_decode", load().huff_decode(
        _dev(payload, "payload"), payload_bytes, _dev(off, "off"), n, chunk_bytes, _dev(cb, "cb"),
        _dev(out, "out"), _dev(status, "status"), _stream(stream)))


def lmc_bytegroup_split(w: torch.Tensor, hi: torch.Tensor, lo: torch.Tensor, stream=None):
    _check("lmc_bytegroup_split", load().lmc_bytegroup_split(_dev(w, "w"), w.numel(), _dev(hi, "hi"),
                                                             _dev(lo, "lo"), _stream(stream)))


def lmc_bytegroup_merge(hi: torch.Tensor, lo: torch.Tensor, w: torch.Tensor, stream=None):
    _check("lmc_bytegroup_merge", load().lmc_bytegroup_merge(_dev(hi, "hi"), _dev(lo, "lo"), w.numel(),
                                                             _dev(w, "w"), _stream(stream)))


def lmc_delta_xor(a: torch.Tensor, b: torch.Tensor, out: torch.Tensor, stream=None):
    _check("lmc_delta_xor", load().lmc_delta_xor(_dev(a, "a"), _dev(b, "b"), a.numel(), _dev(out, "out"),
                                                 _stream(stream)))


def lmc_histogram_bf16(w: torch.Tensor, x0: torch.Tensor | None, hist_hi: torch.Tensor, hist_lo: torch.Tensor,
                       accumulate: bool = False, stream=None):
    _check("lmc_histogram_bf16", load().lmc_histogram_bf16(
        _dev(w, "w"), _dev(x0, "x0"), w.numel(), _dev(hist_hi, "hist_hi"), _dev(hist_lo, "hist_lo"),
        int(bool(accumulate)), _stream(stream)))


def lmc_encode_bf16(w: torch.Tensor, x0: torch.Tensor | None, cb_hi: torch.Tensor, cb_lo: torch.Tensor,
                    chunk_bytes: int, payload_hi: torch.Tensor, off_hi: torch.Tensor, payload_lo: torch.Tensor,
                    off_lo: torch.Tensor, ws: torch.Tensor, status: torch.Tensor, stream=None):
    _check("lmc_encode_bf16", load().lmc_encode_bf16(
        _dev(w, "w"), _dev(x0, "x0"), w.numel(), _dev(cb_hi, "cb_hi"), _dev(cb_lo, "cb_lo"), chunk_bytes,
        _dev(payload_hi, "payload_hi"), payload_hi.numel() * payload_hi.element_size(), _dev(off_hi, "off_hi"),
        _dev(payload_lo, "payload_lo"), payload_lo.numel() * payload_lo.element_size(), _dev(off_lo, "off_lo"),
        _dev(ws, "ws"), ws.numel() * ws.element_size(), _dev(status, "status"), _stream(stream)))


def huff_drift_check(hist: torch.Tensor, cb: torch.Tensor, threshold: float, flag: torch.Tensor,
                     gap: torch.Tensor | None = None, stream=None):
    _check("huff_drift_check", load().huff_drift_check(_dev(hist, "hist"), _dev(cb, "cb"), float(threshold),
                                                       _dev(flag, "flag"), _dev(gap, "gap"), _stream(stream)))


def huff_build_codebook_if(hist: torch.Tensor, flag: torch.Tensor, cb: torch.Tensor, status: torch.Tensor,
                           max_len: int = HUFF_MAX_LEN, flags: int = 0, stream=None):
    _check("huff_build_codebook_if", load().huff_build_codebook_if(
        _dev(hist, "hist"), _dev(flag, "flag"), max_len, flags, _dev(cb, "cb"), _dev(status, "status"),
        _stream(stream)))


def lmc_bytegroup_split_w(x: torch.Tensor, width: int, planes: torch.Tensor, plane_stride: int, stream=None):
    """Plane p (byte width-1-p of each width-byte word of x) at planes[p * plane_stride:]."""
    nbytes = x.numel() * x.element_size()
    if nbytes % width:
        raise ValueError("tensor size is not a whole number of words")
    _check("lmc_bytegroup_split_w", load().lmc_bytegroup_split_w(_dev(x, "x"), nbytes // width, width,
                                                                 _dev(planes, "planes"), plane_stride,
                                                                 _stream(stream)))


def lmc_bytegroup_merge_w(planes: torch.Tensor, width: int, plane_stride: int, out: torch.Tensor, stream=None):
    nbytes = out.numel() * out.element_size()
    if nbytes % width:
        raise ValueError("tensor size is not a whole number of words")
    _check("lmc_bytegroup_merge_w", load().lmc_bytegroup_merge_w(_dev(planes, "planes"), nbytes // width, width,
                                                                 plane_stride, _dev(out, "out"), _stream(stream)))


def lmc_histogram_bf16_counted(w: torch.Tensor, x0: torch.Tensor | None, hist_hi: torch.Tensor,
                               hist_lo: torch.Tensor, seg_counts: torch.Tensor, stream=None):
    _check("lmc_histogram_bf16_counted", load().lmc_histogram_bf16_counted(
        _dev(w, "w"), _dev(x0, "x0"), w.numel(), _dev(hist_hi, "hist_hi"), _dev(hist_lo, "hist_lo"),
        _dev(seg_counts, "seg_counts"), seg_counts.numel() * seg_counts.element_size(), _stream(stream)))


def lmc_encode_bf16_counted(w: torch.Tensor, x0: torch.Tensor | None, cb_hi: torch.Tensor, cb_lo: torch.Tensor,
                            chunk_bytes: int, seg_counts: torch.Tensor, payload_hi: torch.Tensor,
                            off_hi: torch.Tensor, payload_lo: torch.Tensor, off_lo: torch.Tensor, ws: torch.Tensor,
                            status: torch.Tensor, stream=None):
    _check("lmc_encode_bf16_counted", load().lmc_encode_bf16_counted(
        _dev(w, "w"), _dev(x0, "x0"), w.numel(), _dev(cb_hi, "cb_hi"), _dev(cb_lo, "cb_lo"), chunk_bytes,
        _dev(seg_counts, "seg_counts"), seg_counts.numel() * seg_counts.element_size(),
        _dev(payload_hi, "payload_hi"), payload_hi.numel() * payload_hi.element_size(), _dev(off_hi, "off_hi"),
        _dev(payload_lo, "payload_lo"), payload_lo.numel() * payload_lo.element_size(), _dev(off_lo, "off_lo"),
        _dev(ws, "ws"), ws.numel() * ws.element_size(), _dev(status, "status"), _stream(stream)))


def lmc_decode_bf16(payload_hi: torch.Tensor, off_hi: torch.Tensor, payload_lo: torch.Tensor, off_lo: torch.Tensor,
                    n: int, chunk_bytes: int, cb_hi: torch.Tensor, cb_lo: torch.Tensor, x0: torch.Tensor | None,
                    out: torch.Tensor, status: torch.Tensor, bytes_hi: int | None = None,
                    bytes_lo: int | None = None, stream=None):
    if bytes_hi is None:
        bytes_hi = payload_hi.numel() * payload_hi.element_size()
    if bytes_lo is None:
        bytes_lo = payload_lo.numel() * payload_lo.element_size()
    _check("lmc_decode_bf16", load().lmc_decode_bf16(
        _dev(payload_hi, "payload_hi"), bytes_hi, _dev(off_hi, "off_hi"), _dev(payload_lo, "payload_lo"), bytes_lo,
        _dev(off_lo, "off_lo"), n, chunk_bytes, _dev(cb_hi, "cb_hi"), _dev(cb_lo, "cb_lo"), _dev(x0, "x0"),
        _dev(out, "out"), _dev(status, "status"), _stream(stream)))


def huff_code_stats(hist, lengths) -> dict:
    """Host helper: entropy, total bits, mean length and Shannon gap of one stream."""
    h = np.ascontiguousarray(np.asarray(hist, dtype=np.uint64).reshape(256))
    ln = np.ascontiguousarray(np.asarray(lengths, dtype=np.uint8).reshape(256))
    out = HuffStats()
    st = load().huff_code_stats(h.ctypes.data, ln.ctypes.data, ctypes.byref(out))
    _check("huff_code_stats", st)
    return {"n": int(out.n), "total_bits": int(out.total_bits), "entropy_bits": out.entropy_bits,
            "mean_len": out.mean_len, "shannon_gap": out.shannon_gap}


def huff_container_size(n: int, chunk_bytes: int, total_bits: int, with_lengths: bool) -> int:
    return int(load().huff_container_size(n, chunk_bytes, total_bits, 1 if with_lengths else 0))


def huff_container_write(n: int, chunk_bytes: int, max_len: int, lengths, off, payload) -> bytes:
    """Host helper: the container bytes of a stream (lengths None for a fixed codebook)."""
    o = np.ascontiguousarray(np.asarray(off, dtype=np.uint64))
    pay = np.ascontiguousarray(np.asarray(payload, dtype=np.uint8))
    ln = None if lengths is None else np.ascontiguousarray(np.asarray(lengths, dtype=np.uint8).reshape(256))
    T = int(o[-1]) if o.size else 0
    size = huff_container_size(n, chunk_bytes, T, ln is not None)
    dst = np.empty(size, dtype=np.uint8)
    written = ctypes.c_size_t(0)
    st = load().huff_container_write(dst.ctypes.data, size, n, chunk_bytes, max_len,
                                     None if ln is None else ln.ctypes.data, o.ctypes.data, pay.ctypes.data,
                                     ctypes.byref(written))
    _check("huff_container_write", st)
    return dst[: written.value].tobytes()


def huff_container_parse(buf) -> dict:
    """Host helper: the fields of a container, with copies of its lengths, offsets and payload."""
    src = np.frombuffer(buf, dtype=np.uint8)
    v = HuffContainerView()
    st = load().huff_container_parse(src.ctypes.data, src.size, ctypes.byref(v))
    _check("huff_container_parse", st)
    base = src.ctypes.data

    def view(ptr, count):
        return src[ptr - base: ptr - base + count]

    off = view(v.off, 8 * (v.n_chunks + 1)).copy().view("<u8").astype(np.uint64)
    return {"n": int(v.n), "chunk_bytes": int(v.chunk_bytes), "n_chunks": int(v.n_chunks),
            "total_bits": int(v.total_bits), "max_len": int(v.max_len),
            "lengths": view(v.len, 256).copy() if v.has_lengths else None,
            "off": off, "payload": view(v.payload, int(v.payload_bytes)).copy()}
