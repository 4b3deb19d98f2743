"""The byte-stream decode with a warp per chunk, bit-exact.

huff_decode takes this path between 12 and 768 chunks per SM: a warp decodes a
chunk in rounds of 32 slices, one walk per slice from the slice's first bit,
with the start of each slice's first codes noted so that the previous slice's
exit tells whether the walk fell onto the true boundaries (otherwise the slice
is walked again from that exit).  Inputs here are sized into that range and
give it the cases that make it work hardest: codes of one length, codes that
resynchronise rarely, a single 1-bit code, long codes on data the codebook was
not built for, chunks whose slices hold more symbols than a staging area
(half runs of a 1-bit code, half wide data), ragged last chunks, the oracle's
own payload, and corrupt offsets, sizes and counts.
"""
import numpy as np
import pytest
import torch

import oracle
from lossless_huffman_compression_gb300 import _lib, codec
from gpu_util import dev_u8, host_u8, oracle_codebook

pytestmark = pytest.mark.gpu

RNG = np.random.default_rng(4242)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    _lib.load()
    assert torch.cuda.is_available()


def _sms() -> int:
    return torch.cuda.get_device_properties(0).multi_processor_count


def _n(per_sm: float, chunk: int, tail: int = 77) -> int:
    """Symbols for about per_sm chunks per SM (inside the warp path's 12 to 768) and a ragged tail."""
    assert 12 < per_sm < 700
    return int(per_sm * _sms()) * chunk + tail


def _gauss(n, sigma, rng=RNG):
    return np.clip(np.round(rng.normal(0, sigma, n)), -128, 127).astype(np.int8).view(np.uint8)


def _round_trip(x: np.ndarray, cb: codec.Codebook, chunk: int) -> None:
    d = dev_u8(x)
    s = codec.encode(d, cb, chunk)
    out = codec.decode(s, cb)
    np.testing.assert_array_equal(host_u8(out), x)


@pytest.mark.parametrize("chunk,per_sm", [(256, 20), (1024, 13.5), (4096, 16), (32, 600)])
def test_warp_path_gauss(chunk, per_sm):
    x = _gauss(_n(per_sm, chunk), 8)
    _round_trip(x, codec.build_codebook(codec.histogram(dev_u8(x))), chunk)


def test_warp_path_decodes_oracle_payload():
    """The oracle's payload (not the GPU encoder's), a ragged last chunk of 5 symbols."""
    chunk = 1024
    n = _n(14, chunk, tail=5)
    x = _gauss(n, 8)
    ln, cd = oracle_codebook(oracle.histogram(x))
    pay, off = oracle.encode(x, ln, cd, chunk)
    cb = codec.codebook_from_lengths(ln)
    pd = torch.from_numpy(np.concatenate([pay, np.zeros(16, np.uint8)])).cuda()
    s = codec.Stream(pd, torch.from_numpy(off.astype(np.int64)).cuda(), n, chunk)
    out = torch.empty(n, dtype=torch.uint8, device="cuda")
    st = codec.new_status()
    _lib.huff_decode(pd, s.off, n, chunk, cb.buf, out, st, payload_bytes=pay.size)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    np.testing.assert_array_equal(host_u8(out), x)


def test_warp_path_codes_of_one_length():
    """256 codes of 8 bits: slices start on multiples of 8 bits from the chunk's start."""
    cb = codec.build_codebook(torch.full((256,), 1000, dtype=torch.int64, device="cuda"))
    assert (host_u8(cb.buf)[16:16 + 256] == 8).all()
    x = RNG.integers(0, 256, _n(16, 2048), dtype=np.uint8)
    _round_trip(x, cb, 2048)


def test_warp_path_slow_resynchronisation():
    """Lengths 7, 8 and 9 on data of the 8-bit codes only: most first walks stay off the byte grid,
    so slices are walked again from their predecessor's exit, pass after pass."""
    h = torch.full((256,), 1000, dtype=torch.int64, device="cuda")
    h[0], h[254], h[255] = 2000, 1, 1
    cb = codec.build_codebook(h)
    ln = host_u8(cb.buf)[16:16 + 256]
    assert sorted(set(ln.tolist())) == [7, 8, 9]
    eight = np.flatnonzero(ln == 8).astype(np.uint8)
    x = RNG.choice(eight, _n(14, 4096))
    _round_trip(x, cb, 4096)


def test_warp_path_single_code_and_two_codes():
    chunk = 4096
    x = np.full(_n(14, chunk), 9, np.uint8)
    _round_trip(x, codec.build_codebook(codec.histogram(dev_u8(x))), chunk)
    y = RNG.choice(np.array([3, 200], dtype=np.uint8), _n(14, chunk), p=[0.5, 0.5])
    _round_trip(y, codec.build_codebook(codec.histogram(dev_u8(y))), chunk)


def test_warp_path_long_codes():
    """A floor-at-1 codebook from narrow data, used on wide data: most codes are 17 to 24 bits."""
    warm = _gauss(1 << 20, 4)
    cb = codec.build_codebook(codec.histogram(dev_u8(warm)), flags=_lib.HUFF_COVER_ALL)
    assert int(host_u8(cb.buf)[16:16 + 256].max()) >= 17
    x = RNG.integers(0, 256, _n(14, 8192), dtype=np.uint8)
    _round_trip(x, cb, 8192)


def test_warp_path_slices_past_the_staging_area():
    """Each chunk: a run of the 1-bit code's symbol, then wide data.  Slices are sized from the
    chunk's mean code length, so those in the run hold hundreds of symbols and take the path that
    writes them straight to the output."""
    chunk = 8192
    n = _n(14, chunk)
    x = RNG.integers(0, 256, n, dtype=np.uint8)
    x.reshape(-1)[: (n // chunk) * chunk].reshape(-1, chunk)[:, : chunk // 2] = 0
    h = torch.full((256,), 1, dtype=torch.int64, device="cuda")
    h[0] = 1 << 20
    cb = codec.build_codebook(h)
    assert int(host_u8(cb.buf)[16]) == 1
    _round_trip(x, cb, chunk)


def test_warp_path_mixed_distributions():
    """Segments of different widths under one fixed codebook (the chunk-size sweep's shape, small)."""
    chunk = 1 << 10
    seg = 3 * _sms() * chunk
    parts = [_gauss(seg, 4), _gauss(seg, 16), _gauss(seg, 48),
             np.clip(np.round(RNG.laplace(0, 8, seg)), -128, 127).astype(np.int8).view(np.uint8),
             RNG.integers(0, 256, seg, dtype=np.uint8)]
    x = np.concatenate(parts + [_gauss(999, 4)])
    assert 12 * _sms() <= -(-x.size // chunk) < 768 * _sms()
    cb = codec.build_codebook(codec.histogram(dev_u8(parts[0])), flags=_lib.HUFF_COVER_ALL)
    _round_trip(x, cb, chunk)


def test_warp_path_corrupt_streams_detected():
    chunk = 2048
    n = _n(14, chunk)
    x = _gauss(n, 8)
    d = dev_u8(x)
    cb = codec.build_codebook(codec.histogram(d))
    s = codec.encode(d, cb, chunk)
    out = torch.empty(n, dtype=torch.uint8, device="cuda")
    for at, bump in ((2, 1), (2, -1), (700, 8), (-2, -3)):
        off = s.off.clone()
        off[at] += bump
        st = codec.new_status()
        _lib.huff_decode(s.payload, off, n, chunk, cb.buf, out, st, payload_bytes=s.nbytes())
        torch.cuda.synchronize()
        assert int(st.item()) == _lib.HUFF_ERR_CORRUPT_STREAM, (at, bump)
    st = codec.new_status()
    _lib.huff_decode(s.payload, s.off, n, chunk, cb.buf, out, st, payload_bytes=s.nbytes() - 1)
    torch.cuda.synchronize()
    assert int(st.item()) == _lib.HUFF_ERR_CORRUPT_STREAM
    st = codec.new_status()
    _lib.huff_decode(s.payload, s.off, n + 5, chunk, cb.buf, torch.empty(n + 5, dtype=torch.uint8, device="cuda"),
                     st, payload_bytes=s.nbytes())
    torch.cuda.synchronize()
    assert int(st.item()) == _lib.HUFF_ERR_CORRUPT_STREAM
