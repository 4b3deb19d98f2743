"""The byte-stream decode with a warp (or a team of warps) per chunk, bit-exact.

huff_decode takes this path below 768 chunks per SM when a chunk is at least
four rounds of the team: a team of 1, 2, 4, 7, 14 or 28 warps (the fewest
that leave at most a tenth of the teams without a chunk) decodes a chunk in
rounds of one slice per thread (about 56 symbols each), one walk per slice
from the slice's first bit, noting where its first steps start; each thread
then decodes past its slice's end until it meets a noted step of the next
slice's walk (otherwise that slice is walked again from this slice's exit).
Inputs here are sized
into every team size and give the path the cases that make it work hardest:
codes of one length, codes that resynchronise rarely, a single 1-bit code,
long codes on data the codebook was not built for, chunks whose slices hold
more symbols than a staging area (half runs of a 1-bit code, half wide
data), ragged last chunks, the oracle's own payload, and corrupt offsets,
sizes and counts.
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
    """Symbols for about per_sm chunks per SM (below the warp path's 768) and a ragged tail."""
    assert 0 < per_sm < 700
    return int(per_sm * _sms()) * chunk + tail


def _gauss(n, sigma, rng=RNG):
    return np.clip(np.round(rng.normal(0, sigma, n)), -128, 127).astype(np.int8).view(np.uint8)


def _round_trip(x: np.ndarray, cb: codec.Codebook, chunk: int) -> None:
    d = dev_u8(x)
    s = codec.encode(d, cb, chunk)
    out = codec.decode(s, cb)
    np.testing.assert_array_equal(host_u8(out), x)


def _mode(n_chunks: int, chunk: int) -> int:
    """huff_decode's choice: TW warps per chunk, 0 one lane per chunk, -1 the split decode."""
    sms = _sms()
    if n_chunks >= 768 * sms:
        return 0
    tw = 28
    for d in (1, 2, 4, 7, 14):
        if 10 * sms * (28 // d) <= 11 * n_chunks:
            tw = d
            break
    if chunk >= 4 * tw * 32 * 56:
        return tw
    return 0 if n_chunks >= 256 * sms else -1


# the default case of the tests below: a warp per chunk (30 chunks per SM, chunks of 9 rounds)
CHUNK, PER_SM = 16384, 30


@pytest.mark.parametrize("tw,per_sm,chunk", [(28, 0.05, 1 << 18), (28, 1, 1 << 18), (14, 2, 1 << 17), (7, 4, 1 << 16),
                                             (4, 8, 1 << 15), (2, 15, 1 << 14), (1, 30, 1 << 13)])
def test_every_team_size_mixed_data(tw, per_sm, chunk):
    """Gaussian segments of three widths and uniform data under one fixed codebook, at chunk counts
    and sizes that select each team size."""
    n = _n(per_sm, chunk)
    assert _mode(-(-n // chunk), chunk) == tw
    q = n // 4
    x = np.concatenate([_gauss(q, 4), _gauss(q, 16), _gauss(q, 48), RNG.integers(0, 256, n - 3 * q, dtype=np.uint8)])
    cb = codec.build_codebook(codec.histogram(dev_u8(x[:q])), flags=_lib.HUFF_COVER_ALL)
    _round_trip(x, cb, chunk)


@pytest.mark.parametrize("chunk,per_sm,mode", [(CHUNK, PER_SM, 1), (1 << 18, 3, 14), (8192, 100, 1), (256, 20, -1),
                                                (32, 600, 0)])
def test_warp_path_gauss(chunk, per_sm, mode):
    x = _gauss(_n(per_sm, chunk), 8)
    assert _mode(-(-x.size // chunk), chunk) == mode
    _round_trip(x, codec.build_codebook(codec.histogram(dev_u8(x))), chunk)


def test_warp_path_decodes_oracle_payload():
    """The oracle's payload (not the GPU encoder's), a ragged last chunk of 5 symbols."""
    chunk = CHUNK
    n = _n(PER_SM, chunk, tail=5)
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
    x = RNG.integers(0, 256, _n(PER_SM, CHUNK), dtype=np.uint8)
    _round_trip(x, cb, CHUNK)


@pytest.mark.parametrize("tw,per_sm,chunk", [(1, PER_SM, CHUNK), (7, 4, 1 << 16), (28, 0.05, 1 << 18)])
def test_warp_path_slow_resynchronisation(tw, per_sm, chunk):
    """Lengths 7, 8 and 9 on data of the 8-bit codes only: most first walks stay off the byte grid,
    so slices are walked again from their predecessor's exit, pass after pass."""
    h = torch.full((256,), 1000, dtype=torch.int64, device="cuda")
    h[0], h[254], h[255] = 2000, 1, 1
    cb = codec.build_codebook(h)
    ln = host_u8(cb.buf)[16:16 + 256]
    assert sorted(set(ln.tolist())) == [7, 8, 9]
    eight = np.flatnonzero(ln == 8).astype(np.uint8)
    x = RNG.choice(eight, _n(per_sm, chunk))
    assert _mode(-(-x.size // chunk), chunk) == tw
    _round_trip(x, cb, chunk)


def test_warp_path_single_code_and_two_codes():
    chunk = CHUNK
    x = np.full(_n(PER_SM, chunk), 9, np.uint8)
    _round_trip(x, codec.build_codebook(codec.histogram(dev_u8(x))), chunk)
    y = RNG.choice(np.array([3, 200], dtype=np.uint8), _n(PER_SM, chunk), p=[0.5, 0.5])
    _round_trip(y, codec.build_codebook(codec.histogram(dev_u8(y))), chunk)


def test_warp_path_long_codes():
    """A floor-at-1 codebook from narrow data, used on wide data: most codes are 17 to 24 bits."""
    warm = _gauss(1 << 20, 4)
    cb = codec.build_codebook(codec.histogram(dev_u8(warm)), flags=_lib.HUFF_COVER_ALL)
    assert int(host_u8(cb.buf)[16:16 + 256].max()) >= 17
    x = RNG.integers(0, 256, _n(PER_SM, CHUNK), dtype=np.uint8)
    _round_trip(x, cb, CHUNK)


@pytest.mark.parametrize("tw,per_sm,chunk", [(1, PER_SM, CHUNK), (4, 8, 1 << 15), (28, 1, 1 << 18)])
def test_warp_path_slices_past_the_staging_area(tw, per_sm, chunk):
    """Each chunk: a run of the 1-bit code's symbol, then wide data.  Slices are sized from the
    chunk's mean code length, so those in the run hold hundreds of symbols and take the path that
    writes them straight to the output (a warp per chunk, and teams of 4 and 28 warps)."""
    n = _n(per_sm, chunk)
    assert _mode(-(-n // chunk), chunk) == tw
    x = RNG.integers(0, 256, n, dtype=np.uint8)
    x.reshape(-1)[: (n // chunk) * chunk].reshape(-1, chunk)[:, : chunk // 2] = 0
    h = torch.full((256,), 1, dtype=torch.int64, device="cuda")
    h[0] = 1 << 20
    cb = codec.build_codebook(h)
    assert int(host_u8(cb.buf)[16]) == 1
    _round_trip(x, cb, chunk)


def test_warp_path_mixed_distributions():
    """Segments of different widths under one fixed codebook (the chunk-size sweep's shape, small)."""
    chunk = CHUNK
    seg = 7 * _sms() * chunk
    parts = [_gauss(seg, 4), _gauss(seg, 16), _gauss(seg, 48),
             np.clip(np.round(RNG.laplace(0, 8, seg)), -128, 127).astype(np.int8).view(np.uint8),
             RNG.integers(0, 256, seg, dtype=np.uint8)]
    x = np.concatenate(parts + [_gauss(999, 4)])
    assert _mode(-(-x.size // chunk), chunk) == 1
    cb = codec.build_codebook(codec.histogram(dev_u8(parts[0])), flags=_lib.HUFF_COVER_ALL)
    _round_trip(x, cb, chunk)


@pytest.mark.parametrize("tw,per_sm,chunk", [(1, PER_SM, CHUNK), (28, 1, 1 << 18)])
def test_warp_path_corrupt_streams_detected(tw, per_sm, chunk):
    n = _n(per_sm, chunk)
    n_chunks = -(-n // chunk)
    assert _mode(n_chunks, chunk) == tw
    x = _gauss(n, 8)
    d = dev_u8(x)
    cb = codec.build_codebook(codec.histogram(d))
    s = codec.encode(d, cb, chunk)
    out = torch.empty(n, dtype=torch.uint8, device="cuda")
    for at, bump in ((2, 1), (2, -1), (n_chunks // 2, 8), (-2, -3)):
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
