"""The byte-stream decode's one-lane path and its few-chunk cases, bit-exact.

huff_decode gives every chunk one lane when there are enough chunks to fill
the GPU (at least 768 per SM); in one wave of blocks a block's warps spread
over the input, in more waves block b takes the range with the b-th most
bits.  With fewer, a team of warps takes each chunk
(a whole CTA of 28 warps when chunks are as few as here; every team size is
tested in test_gpu_decode_warp.py) and each thread a slice of its bits, whose
code boundaries are found by self-synchronisation: one walk per slice from
its first bit, then from its end until the next slice's walk is met.  These
tests size inputs on both ends and give the few-chunk cases the codes that
make them work hardest:
- codes of one length (slices start on the lengths' common divisor), and
  codes that resynchronise only rarely;
- a single 1-bit code;
- long codes on data the codebook was not built for;
- ragged last chunks;
- corrupt offsets and payloads.
"""
import numpy as np
import pytest
import torch

import oracle
from lossless_huffman_compression_gb300 import _lib, codec
from gpu_util import dev_u8, host_u8, oracle_codebook

pytestmark = pytest.mark.gpu

RNG = np.random.default_rng(77)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    _lib.load()
    assert torch.cuda.is_available()


def _gauss(n, sigma, rng=RNG):
    return np.clip(np.round(rng.normal(0, sigma, n)), -128, 127).astype(np.int8).view(np.uint8)


def _round_trip(x: np.ndarray, cb: codec.Codebook, chunk: int) -> None:
    d = dev_u8(x)
    s = codec.encode(d, cb, chunk)
    out = codec.decode(s, cb)
    np.testing.assert_array_equal(host_u8(out), x)


def _lanes_threshold() -> int:
    # a chunk count above the one from which every chunk gets one lane (768 per SM)
    return torch.cuda.get_device_properties(0).multi_processor_count * 1024


@pytest.mark.parametrize("kind", ["gauss", "skew"])
def test_one_lane_per_chunk_path(kind):
    """Enough chunks for one lane each (not the team path), ragged tail."""
    chunk = 256
    n = _lanes_threshold() * chunk + 77
    if kind == "gauss":
        x = _gauss(n, 8)
    else:
        x = RNG.choice(np.array([0, 1, 2, 255], dtype=np.uint8), n, p=[0.95, 0.03, 0.019, 0.001])
    cb = codec.build_codebook(codec.histogram(dev_u8(x)))
    _round_trip(x, cb, chunk)


@pytest.mark.parametrize("waves", [1.0, 2.3])
def test_one_lane_spread_and_ranked_blocks(waves):
    """One lane per chunk in one wave of 896-lane blocks (the warps of a block spread over the input)
    and in 2.3 waves of chunks of 4096 symbols (block b takes the range with the b-th most bits).
    Regions of three widths under one codebook make the ranges' bit counts differ; ragged tail."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    chunk = 4096
    n = int(waves * sms * 896) * chunk + 77
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    x = torch.empty(n, dtype=torch.uint8, device="cuda")
    step = 64 << 20
    for k, a in enumerate(range(0, n, step)):
        m = min(step, n - a)
        v = torch.randn(m, device="cuda", generator=g) * (4.0, 16.0, 48.0)[k % 3]
        x[a:a + m] = torch.clamp(torch.round(v), -128, 127).to(torch.int8).view(torch.uint8)
    cb = codec.build_codebook(codec.histogram(x[: 64 << 20]), flags=_lib.HUFF_COVER_ALL)
    s = codec.encode(x, cb, chunk)
    out = codec.decode(s, cb)
    assert torch.equal(out, x)


@pytest.mark.parametrize("n,chunk", [(1, 256), (1000, 256), (1000, 32), (100_003, 96), (65_536, 65_536), (65_537, 65_536),
                                     (1_000_003, 1 << 20), (3_000_001, 1 << 22), (200_017, 16_384),
                                     (2_000_001, 1 << 30)])  # the largest chunk the ABI accepts
def test_few_chunks_matches_oracle_payload(n, chunk):
    """The oracle's payload (not the GPU encoder's) decoded with few chunks."""
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


@pytest.mark.parametrize("n", [1_000_003, 777_777])
def test_few_chunks_codes_of_one_length(n):
    """256 codes of 8 bits: a walk that starts off the byte grid never meets it, so slices start on
    multiples of the lengths' common divisor (and the chunk is not a multiple of the slice count)."""
    cb = codec.build_codebook(torch.full((256,), 1000, dtype=torch.int64, device="cuda"))
    assert (host_u8(cb.buf)[16:16 + 256] == 8).all()  # len[] follows the four 32-bit header fields
    x = RNG.integers(0, 256, n, dtype=np.uint8)
    _round_trip(x, cb, 1 << 20)


@pytest.mark.parametrize("n", [1_000_003, 300_001])
def test_few_chunks_slow_resynchronisation(n):
    """Lengths 7, 8 and 9 (common divisor 1) on data of the 8-bit codes only: a walk off the byte
    grid moves onto it only when it happens to read the 7- or 9-bit code, about once in a hundred
    codes, so many walks do not meet the next slice's noted steps and slices are walked again from
    the previous exit."""
    h = torch.full((256,), 1000, dtype=torch.int64, device="cuda")
    h[0], h[254], h[255] = 2000, 1, 1
    cb = codec.build_codebook(h)
    ln = host_u8(cb.buf)[16:16 + 256]
    assert sorted(set(ln.tolist())) == [7, 8, 9]
    eight = np.flatnonzero(ln == 8).astype(np.uint8)
    x = RNG.choice(eight, n)
    _round_trip(x, cb, 1 << 20)


def test_few_chunks_single_code_and_two_codes():
    n = 2_000_001
    x = np.full(n, 9, np.uint8)
    _round_trip(x, codec.build_codebook(codec.histogram(dev_u8(x))), 1 << 20)
    y = RNG.choice(np.array([3, 200], dtype=np.uint8), n, p=[0.5, 0.5])
    _round_trip(y, codec.build_codebook(codec.histogram(dev_u8(y))), 1 << 20)


def test_few_chunks_long_codes():
    """A floor-at-1 codebook from narrow data, used on wide data: most codes are 17 to 24 bits."""
    warm = _gauss(1 << 20, 4)
    cb = codec.build_codebook(codec.histogram(dev_u8(warm)), flags=_lib.HUFF_COVER_ALL)
    x = RNG.integers(0, 256, 1_500_007, dtype=np.uint8)
    _round_trip(x, cb, 1 << 18)


@pytest.mark.parametrize("n,chunk", [(600_000, 1 << 17), (3_000_000, 1 << 19)])  # the split decode; teams of 28 warps
def test_few_chunks_corrupt_streams_detected(n, chunk):
    x = _gauss(n, 8)
    d = dev_u8(x)
    cb = codec.build_codebook(codec.histogram(d))
    s = codec.encode(d, cb, chunk)
    out = torch.empty(n, dtype=torch.uint8, device="cuda")
    for bump in (1, -1, 8):
        off = s.off.clone()
        off[2] += bump
        st = codec.new_status()
        _lib.huff_decode(s.payload, off, n, chunk, cb.buf, out, st, payload_bytes=s.nbytes())
        torch.cuda.synchronize()
        assert int(st.item()) == _lib.HUFF_ERR_CORRUPT_STREAM
    st = codec.new_status()
    _lib.huff_decode(s.payload, s.off, n, chunk, cb.buf, out, st, payload_bytes=s.nbytes() - 1)
    torch.cuda.synchronize()
    assert int(st.item()) == _lib.HUFF_ERR_CORRUPT_STREAM
    # a count that is not the stream's: more symbols than the last chunk holds
    st = codec.new_status()
    _lib.huff_decode(s.payload, s.off, n + 5, chunk, cb.buf, torch.empty(n + 5, dtype=torch.uint8, device="cuda"),
                     st, payload_bytes=s.nbytes())
    torch.cuda.synchronize()
    assert int(st.item()) == _lib.HUFF_ERR_CORRUPT_STREAM


def test_largest_chunk_gpu_round_trip():
    """Encode and decode on the GPU with one chunk of the largest accepted size."""
    x = _gauss(3_000_017, 8)
    cb = codec.build_codebook(codec.histogram(dev_u8(x)))
    _round_trip(x, cb, 1 << 30)
