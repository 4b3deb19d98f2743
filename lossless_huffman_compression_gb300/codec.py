"""Convenience layer over the binding: buffers sized and allocated by torch,
work done by libhuff's kernels.  Nothing here computes on the host except
buffer sizes.

    cb = build_codebook(histogram(x))          # per-shard codebook
    s = encode(x, cb)                          # Stream(payload, off, n, chunk_bytes)
    y = decode(s, cb)                          # == x

    streams = compress_bf16(x1, x0)            # LMC: XOR delta, byte planes, per-plane codebooks
    x1_back = decompress_bf16(streams, x0)
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import _lib
from ._lib import HuffError

DEFAULT_CHUNK = 16384


class Codebook:
    """A device-resident huff_codebook."""

    def __init__(self, device=None, buf: torch.Tensor | None = None):
        if buf is not None:  # a row of a [count, size] block built by build_codebooks
            self.buf = buf
            return
        device = torch.device("cuda") if device is None else torch.device(device)
        self.buf = torch.zeros(_lib.huff_codebook_size(), dtype=torch.uint8, device=device)

    @property
    def device(self):
        return self.buf.device

    def lengths(self) -> np.ndarray:
        """The 256 code lengths: the transmitted form of the codebook."""
        o = _lib.CODEBOOK_LEN_OFFSET
        return self.buf[o:o + 256].cpu().numpy().copy()

    def codes(self) -> np.ndarray:
        o = _lib.CODEBOOK_LEN_OFFSET + 256
        return self.buf[o:o + 1024].cpu().numpy().view(np.uint32).copy()


@dataclass
class Stream:
    payload: torch.Tensor  # uint8, capacity >= ceil(T/32)*4
    off: torch.Tensor      # int64[n_chunks + 1], bit offsets (uint64 in the C ABI)
    n: int
    chunk_bytes: int

    def total_bits(self) -> int:
        return int(self.off[-1].item())

    def nbytes(self) -> int:
        return (self.total_bits() + 7) // 8

    def n_chunks(self) -> int:
        return self.off.numel() - 1


def new_status(device=None) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def raise_on_status(status: torch.Tensor, what: str) -> None:
    st = int(status.item())
    if st != 0:
        raise HuffError(what, st)


def histogram(x: torch.Tensor, hist: torch.Tensor | None = None, accumulate: bool = False) -> torch.Tensor:
    if hist is None:
        hist = torch.zeros(256, dtype=torch.int64, device=x.device)
    _lib.huff_histogram(x.reshape(-1), hist, accumulate=accumulate)
    return hist


def build_codebook(hist: torch.Tensor, max_len: int = 24, flags: int = 0, cb: Codebook | None = None,
                   status: torch.Tensor | None = None) -> Codebook:
    cb = cb or Codebook(hist.device)
    st = status if status is not None else new_status(hist.device)
    _lib.huff_build_codebook(hist, cb.buf, st, max_len, flags)
    if status is None:
        raise_on_status(st, "huff_build_codebook")
    return cb


def build_codebooks(hists: torch.Tensor, max_len: int = 24, flags: int = 0,
                    status: torch.Tensor | None = None) -> list[Codebook]:
    """One codebook per row of hists ([count, 256]), built in one launch."""
    count = hists.shape[0]
    bufs = torch.zeros((count, _lib.huff_codebook_size()), dtype=torch.uint8, device=hists.device)
    st = status if status is not None else new_status(hists.device)
    _lib.huff_build_codebooks(hists, bufs, st, max_len, flags)
    if status is None:
        raise_on_status(st, "huff_build_codebooks")
    return [Codebook(buf=bufs[k]) for k in range(count)]


def stream_copy(s: Stream, dst_payload: torch.Tensor | None = None, dst_off: torch.Tensor | None = None,
                status: torch.Tensor | None = None) -> Stream:
    """The stream in other device buffers (the loopback link of one GPU): payload bytes up to the
    stream's size, read on the device, and the offsets."""
    if dst_payload is None:
        dst_payload = torch.empty_like(s.payload)
    if dst_off is None:
        dst_off = torch.empty_like(s.off)
    st = status if status is not None else new_status(s.payload.device)
    _lib.huff_stream_copy(s.payload, s.off, dst_payload, dst_off, st)
    if status is None:
        raise_on_status(st, "huff_stream_copy")
    return Stream(dst_payload, dst_off, s.n, s.chunk_bytes)


class CodebookBank:
    """One fixed codebook per tensor type ("Single-stage Huffman encoder for ML
    compression", Methodology 1-3: symbol statistics are recorded per tensor
    type -- activations, gradients, weights -- over warm-up batches, and one
    codebook is built from each type's averaged distribution; a tensor is then
    encoded with its type's codebook).  observe() counts a warm-up tensor into
    its type's histogram on the device; build() makes every type's codebook in
    one launch (every symbol gets a code, so later tensors never miss one);
    encode/decode pick the codebook by type."""

    def __init__(self, types, device=None, max_len: int = 24):
        self.types = list(types)
        if len(set(self.types)) != len(self.types) or not self.types:
            raise ValueError("tensor types must be distinct and at least one")
        self._index = {t: i for i, t in enumerate(self.types)}
        device = torch.device("cuda") if device is None else torch.device(device)
        self.max_len = max_len
        self.hists = torch.zeros((len(self.types), 256), dtype=torch.int64, device=device)
        self.codebooks: list[Codebook] | None = None

    def observe(self, kind, x: torch.Tensor) -> None:
        histogram(x.reshape(-1).view(torch.uint8), self.hists[self._index[kind]], accumulate=True)

    def build(self) -> list[Codebook]:
        self.codebooks = build_codebooks(self.hists, self.max_len, _lib.HUFF_COVER_ALL)
        return self.codebooks

    def codebook(self, kind) -> Codebook:
        if self.codebooks is None:
            raise RuntimeError("CodebookBank.build() has not run")
        return self.codebooks[self._index[kind]]

    def encode(self, kind, x: torch.Tensor, chunk_bytes: int = DEFAULT_CHUNK) -> Stream:
        return encode(x, self.codebook(kind), chunk_bytes, self.max_len)

    def decode(self, kind, s: Stream, out: torch.Tensor | None = None) -> torch.Tensor:
        return decode(s, self.codebook(kind), out=out)


def codebook_from_lengths(lengths, max_len: int = 24, device=None) -> Codebook:
    cb = Codebook(device)
    st = new_status(cb.device)
    _lib.huff_codebook_from_lengths(lengths, cb.buf, st, max_len)
    raise_on_status(st, "huff_codebook_from_lengths")
    return cb


def encode(x: torch.Tensor, cb: Codebook, chunk_bytes: int | None = DEFAULT_CHUNK, max_len: int = 24,
           status: torch.Tensor | None = None) -> Stream:
    """Encode x's bytes with a given codebook; chunk_bytes=None picks the size (huff_pick_chunk)."""
    flat = x.reshape(-1)
    n = flat.numel() * flat.element_size()
    if chunk_bytes is None:
        chunk_bytes = _lib.huff_pick_chunk(n)
    payload = torch.empty(_lib.huff_encode_bound(n, max_len), dtype=torch.uint8, device=x.device)
    off = torch.empty(_lib.huff_num_chunks(n, chunk_bytes) + 1, dtype=torch.int64, device=x.device)
    ws = torch.empty(max(_lib.huff_workspace_size(n, chunk_bytes), 16) // 8, dtype=torch.int64, device=x.device)
    st = status if status is not None else new_status(x.device)
    _lib.huff_encode(flat, cb.buf, chunk_bytes, payload, off, ws, st, n=n)
    if status is None:
        raise_on_status(st, "huff_encode")
    return Stream(payload, off, n, chunk_bytes)


def decode(s: Stream, cb: Codebook, out: torch.Tensor | None = None,
           status: torch.Tensor | None = None) -> torch.Tensor:
    if out is None:
        out = torch.empty(max(s.n, 1), dtype=torch.uint8, device=s.payload.device)[: s.n]
    st = status if status is not None else new_status(s.payload.device)
    _lib.huff_decode(s.payload, s.off, s.n, s.chunk_bytes, cb.buf, out, st)
    if status is None:
        raise_on_status(st, "huff_decode")
    return out


def compress(x: torch.Tensor, chunk_bytes: int = DEFAULT_CHUNK, max_len: int = 24, flags: int = 0,
             status: torch.Tensor | None = None):
    """Per-shard Huffman: histogram, codebook and encode of one byte stream.  The three launches share
    one status, read once at the end (a failed build leaves a codebook the encode rejects)."""
    st = status if status is not None else new_status(x.device)
    cb = build_codebook(histogram(x), max_len, flags, status=st)
    s = encode(x, cb, chunk_bytes, max_len, status=st)
    if status is None:
        raise_on_status(st, "compress")
    return cb, s


def to_container(s: Stream, cb: Codebook | None = None, max_len: int = 24) -> bytes:
    """The stream as container bytes (huff_container_write).  With cb (per-shard mode) the container
    carries cb's 256 code lengths; without (a fixed codebook the receiver holds) it does not."""
    T = s.total_bits()
    off = s.off.cpu().numpy().astype(np.uint64)
    payload = s.payload[: (T + 7) // 8].cpu().numpy()
    return _lib.huff_container_write(s.n, s.chunk_bytes, max_len, None if cb is None else cb.lengths(), off,
                                     payload)


def from_container(buf, cb: Codebook | None = None, device=None) -> tuple[Stream, Codebook]:
    """A container's stream on the device and its codebook: imported from the carried lengths, or the
    fixed codebook cb the caller holds."""
    f = _lib.huff_container_parse(buf)
    device = torch.device("cuda") if device is None else torch.device(device)
    pb = f["payload"].size
    payload = torch.zeros(((pb + 15) // 16) * 16 + 16, dtype=torch.uint8, device=device)
    payload[:pb] = torch.from_numpy(f["payload"]).to(device)
    off = torch.from_numpy(f["off"].astype(np.int64)).to(device)
    if f["lengths"] is not None:
        cb = codebook_from_lengths(f["lengths"], f["max_len"], device)
    elif cb is None:
        raise ValueError("a fixed-codebook container carries no lengths: pass the codebook")
    return Stream(payload, off, f["n"], f["chunk_bytes"]), cb


@dataclass
class Bf16Streams:
    cb_hi: Codebook
    cb_lo: Codebook
    hi: Stream
    lo: Stream
    n: int


def compress_bf16(w: torch.Tensor, x0: torch.Tensor | None = None, chunk_bytes: int | None = DEFAULT_CHUNK,
                  max_len: int = 24, flags: int = 0, cb_hi: Codebook | None = None,
                  cb_lo: Codebook | None = None) -> Bf16Streams:
    """LMC snapshot compress: optional XOR delta, byte planes, one codebook per plane.
    chunk_bytes=None picks the chunk size for the device and for whether a delta is decoded (huff_pick_chunk)."""
    w16 = w.reshape(-1).view(torch.int16)
    x16 = None if x0 is None else x0.reshape(-1).view(torch.int16)
    n = w16.numel()
    if chunk_bytes is None:
        chunk_bytes = _lib.huff_pick_chunk(n, delta=x0 is not None)
    dev = w.device
    cap = _lib.huff_encode_bound(n, max_len)
    p_hi = torch.empty(cap, dtype=torch.uint8, device=dev)
    p_lo = torch.empty(cap, dtype=torch.uint8, device=dev)
    nc = _lib.huff_num_chunks(n, chunk_bytes)
    o_hi = torch.empty(nc + 1, dtype=torch.int64, device=dev)
    o_lo = torch.empty(nc + 1, dtype=torch.int64, device=dev)
    if cb_hi is None or cb_lo is None:
        # per-shard: the histogram pass records per-segment counts, so the encode makes one pass
        hists = torch.empty((2, 256), dtype=torch.int64, device=dev)
        h_hi, h_lo = hists[0], hists[1]
        seg = torch.empty(max(_lib.lmc_segment_counts_size(n), 4) // 4, dtype=torch.int32, device=dev)
        _lib.lmc_histogram_bf16_counted(w16, x16, h_hi, h_lo, seg)
        st = new_status(dev)
        cb_hi, cb_lo = build_codebooks(hists, max_len, flags, status=st)
        raise_on_status(st, "huff_build_codebooks")
        ws = torch.empty(max(_lib.lmc_counted_workspace_size(n), 16) // 8, dtype=torch.int64, device=dev)
        st = new_status(dev)
        _lib.lmc_encode_bf16_counted(w16, x16, cb_hi.buf, cb_lo.buf, chunk_bytes, seg, p_hi, o_hi, p_lo, o_lo, ws,
                                     st)
        raise_on_status(st, "lmc_encode_bf16_counted")
    else:
        # given codebooks: a counting pass over the input, then the one-pass encode
        ws = torch.empty(max(_lib.lmc_workspace_size(n, chunk_bytes), 16) // 8, dtype=torch.int64, device=dev)
        st = new_status(dev)
        _lib.lmc_encode_bf16(w16, x16, cb_hi.buf, cb_lo.buf, chunk_bytes, p_hi, o_hi, p_lo, o_lo, ws, st)
        raise_on_status(st, "lmc_encode_bf16")
    return Bf16Streams(cb_hi, cb_lo, Stream(p_hi, o_hi, n, chunk_bytes), Stream(p_lo, o_lo, n, chunk_bytes), n)


def decompress_bf16(s: Bf16Streams, x0: torch.Tensor | None = None, out: torch.Tensor | None = None) -> torch.Tensor:
    dev = s.hi.payload.device
    if out is None:
        out = torch.empty(max(s.n, 1), dtype=torch.bfloat16, device=dev)[: s.n]
    x16 = None if x0 is None else x0.reshape(-1).view(torch.int16)
    st = new_status(dev)
    _lib.lmc_decode_bf16(s.hi.payload, s.hi.off, s.lo.payload, s.lo.off, s.n, s.hi.chunk_bytes, s.cb_hi.buf,
                         s.cb_lo.buf, x16, out.view(torch.int16), st)
    raise_on_status(st, "lmc_decode_bf16")
    return out


@dataclass
class PlaneStreams:
    """A tensor of width-byte words as byte planes (most significant first), one stream each."""
    width: int
    n: int                 # words
    dtype: torch.dtype
    shape: tuple
    planes: list           # [(Codebook, Stream)] for plane 0 .. width-1


def _plane_stride(n: int) -> int:
    return max(16, (n + 15) // 16 * 16)


def _xor_words(a: torch.Tensor, b: torch.Tensor, out: torch.Tensor) -> None:
    """out = a ^ b on the tensors' bit patterns (lmc_delta_xor on their 16-bit view)."""
    if (a.numel() * a.element_size()) % 2:
        raise ValueError("the XOR delta needs an even number of bytes")
    _lib.lmc_delta_xor(a.reshape(-1).view(torch.int16), b.reshape(-1).view(torch.int16),
                       out.reshape(-1).view(torch.int16))


def compress_planes(x: torch.Tensor, x0: torch.Tensor | None = None, chunk_bytes: int = DEFAULT_CHUNK,
                    max_len: int = 24, flags: int = 0, codebooks: list | None = None) -> PlaneStreams:
    """Byte grouping for any element width (fp32: 4 planes, fp16/bf16: 2, fp8: 1, fp64: 8), optionally of the
    XOR delta against x0, then one canonical Huffman stream per plane (per-plane codebooks, or the given ones)."""
    width = x.element_size()
    flat = x.reshape(-1)
    n = flat.numel()
    src = flat
    if x0 is not None:
        src = torch.empty_like(flat)
        _xor_words(flat, x0, src)
    ps = _plane_stride(n)
    planes = torch.empty(width * ps, dtype=torch.uint8, device=x.device)
    _lib.lmc_bytegroup_split_w(src, width, planes, ps)
    out = []
    for p in range(width):
        pl = planes[p * ps: p * ps + n]
        cb = codebooks[p] if codebooks is not None else build_codebook(histogram(pl), max_len, flags)
        out.append((cb, encode(pl, cb, chunk_bytes, max_len)))
    return PlaneStreams(width, n, x.dtype, tuple(x.shape), out)


def decompress_planes(s: PlaneStreams, x0: torch.Tensor | None = None) -> torch.Tensor:
    dev = s.planes[0][1].payload.device
    ps = _plane_stride(s.n)
    planes = torch.empty(s.width * ps, dtype=torch.uint8, device=dev)
    for p, (cb, st) in enumerate(s.planes):
        decode(st, cb, out=planes[p * ps: p * ps + s.n])
    out = torch.empty(s.shape, dtype=s.dtype, device=dev)
    _lib.lmc_bytegroup_merge_w(planes, s.width, ps, out.reshape(-1))
    if x0 is not None:
        _xor_words(out, x0, out)
    return out


class DriftAdaptiveCodebook:
    """A fixed codebook that is rebuilt from a shard's own histogram when the shard drifts too far from it
    (huff_drift_check + huff_build_codebook_if; no host round trip).  The flag of the last check stays on
    the device in `refreshed`; read it (one sync) to know whether the transmitted lengths changed."""

    def __init__(self, cb: Codebook, threshold: float = 0.02, max_len: int = 24, flags: int = _lib.HUFF_COVER_ALL):
        self.cb = cb
        self.threshold = threshold
        self.max_len = max_len
        self.flags = flags
        dev = cb.device
        self.refreshed = torch.zeros(1, dtype=torch.int32, device=dev)
        self.gap = torch.zeros(1, dtype=torch.float64, device=dev)
        self.status = new_status(dev)
        self.hist = torch.zeros(256, dtype=torch.int64, device=dev)

    def encode(self, x: torch.Tensor, chunk_bytes: int = DEFAULT_CHUNK) -> Stream:
        histogram(x, self.hist)
        _lib.huff_drift_check(self.hist, self.cb.buf, self.threshold, self.refreshed, self.gap)
        _lib.huff_build_codebook_if(self.hist, self.refreshed, self.cb.buf, self.status, self.max_len, self.flags)
        return encode(x, self.cb, chunk_bytes, self.max_len)

