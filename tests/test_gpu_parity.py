"""GPU path vs the CPU oracle, element by element, through the C ABI.

Integer and byte work: every comparison is exact.  Sizes span several encode
tiles (8192 symbols; 4096 bf16 elements) with ragged tails, several chunk
sizes, odd alignments and the degenerate codebooks (empty, one symbol,
length-limited).
"""
import numpy as np
import pytest
import torch

import oracle
from lossless_huffman_compression_gb300 import _lib, codec
from gpu_util import (assert_stream_equal, bits_of, dev_u8, host, host_u8, oracle_codebook)

pytestmark = pytest.mark.gpu

RNG = np.random.default_rng(2024)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    _lib.load()
    assert torch.cuda.is_available()


def _data(kind: str, n: int, rng=RNG) -> np.ndarray:
    if kind == "gauss":
        return np.clip(np.round(rng.normal(0, 8, n)), -128, 127).astype(np.int8).view(np.uint8)
    if kind == "wide":
        return np.clip(np.round(rng.normal(0, 48, n)), -128, 127).astype(np.int8).view(np.uint8)
    if kind == "uniform":
        return rng.integers(0, 256, n, dtype=np.uint8)
    if kind == "single":
        return np.full(n, 7, dtype=np.uint8)
    if kind == "two":
        return rng.choice(np.array([3, 200], dtype=np.uint8), n, p=[0.97, 0.03])
    if kind == "skew":
        return rng.choice(np.array([0, 1, 2, 255], dtype=np.uint8), n, p=[0.95, 0.03, 0.019, 0.001])
    raise ValueError(kind)


# ------------------------------------------------------------------ histogram
@pytest.mark.parametrize("n", [0, 1, 15, 16, 17, 255, 4097, 100_003, 1 << 20])
@pytest.mark.parametrize("kind", ["gauss", "uniform", "single"])
def test_histogram(n, kind):
    x = _data(kind, n)
    hist = torch.zeros(256, dtype=torch.int64, device="cuda")
    _lib.huff_histogram(dev_u8(x), hist, n=n)
    np.testing.assert_array_equal(host(hist).astype(np.uint64), oracle.histogram(x))


@pytest.mark.parametrize("offset", [1, 3, 7, 13])
def test_histogram_misaligned_and_accumulate(offset):
    x = _data("gauss", 50_001)
    d = dev_u8(x)
    hist = torch.zeros(256, dtype=torch.int64, device="cuda")
    _lib.huff_histogram(d, hist, n=x.size - offset, offset=offset)
    _lib.huff_histogram(d, hist, n=x.size - offset, offset=offset, accumulate=True)
    np.testing.assert_array_equal(host(hist).astype(np.uint64), 2 * oracle.histogram(x[offset:]))


@pytest.mark.parametrize("n", [1, 2, 9, 17, 4096, 77_777])
def test_histogram_plane_view_stride2(n):
    w = RNG.integers(0, 1 << 16, n, dtype=np.uint16)
    d = dev_u8(w.view(np.uint8))
    lo = torch.zeros(256, dtype=torch.int64, device="cuda")
    hi = torch.zeros(256, dtype=torch.int64, device="cuda")
    _lib.huff_histogram(d, lo, n=n, stride=2, offset=0)
    _lib.huff_histogram(d, hi, n=n, stride=2, offset=1)
    b = w.view(np.uint8)
    np.testing.assert_array_equal(host(lo).astype(np.uint64), oracle.histogram(b, stride=2, n=n))
    np.testing.assert_array_equal(host(hi).astype(np.uint64), oracle.histogram(b[1:], stride=2, n=n))


# ------------------------------------------------------------------ codebook
def _adversarial_hists():
    out = []
    h = np.zeros(256, np.uint64); out.append(h)                          # empty
    h = np.zeros(256, np.uint64); h[9] = 5; out.append(h)                # one symbol
    h = np.zeros(256, np.uint64); h[0] = 1; h[255] = 10 ** 12; out.append(h)
    out.append(np.full(256, 3, np.uint64))                               # all equal
    fib = [1, 1]
    while len(fib) < 40:
        fib.append(fib[-1] + fib[-2])
    h = np.zeros(256, np.uint64); h[:40] = fib; out.append(h)            # depth 39 before the limit
    h = np.zeros(256, np.uint64); h[100:140] = fib; out.append(h)
    h = np.array([2 ** min(i, 54) for i in range(256)], dtype=np.uint64); out.append(h)  # total just below 2^63
    h = np.zeros(256, np.uint64); h[::2] = 1; out.append(h)
    return out


def _build_many(hists, max_len, flags):
    k = len(hists)
    H = torch.from_numpy(np.stack(hists).astype(np.int64)).cuda()
    sz = _lib.huff_codebook_size()
    cbs = torch.zeros(k, sz, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for i in range(k):
        _lib.huff_build_codebook(H[i], cbs[i], st, max_len, flags)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return host(cbs)


@pytest.mark.parametrize("max_len,flags", [(24, 0), (24, 1), (12, 0), (9, 1), (8, 1)])
def test_codebooks_match_oracle(max_len, flags):
    hists = _adversarial_hists()
    for _ in range(300):
        m = int(RNG.integers(1, 257))
        h = np.zeros(256, np.uint64)
        syms = RNG.choice(256, m, replace=False)
        mode = RNG.integers(0, 4)
        if mode == 0:
            h[syms] = RNG.integers(1, 1000, m)
        elif mode == 1:
            h[syms] = RNG.integers(1, 4, m)                                  # many ties
        elif mode == 2:
            h[syms] = (1e9 * np.exp(-RNG.uniform(0, 30, m))).astype(np.uint64) + 1
        else:
            h[syms] = RNG.integers(1, 10 ** 12, m)
        hists.append(h)
    cbs = _build_many(hists, max_len, flags)
    o = _lib.CODEBOOK_LEN_OFFSET
    for h, cb in zip(hists, cbs):
        ln, cd = oracle_codebook(h, max_len, flags)
        got_len = cb[o:o + 256]
        got_code = cb[o + 256:o + 256 + 1024].view(np.uint32)
        np.testing.assert_array_equal(got_len, ln)
        np.testing.assert_array_equal(got_code, cd)
        magic = int(cb[:4].view(np.uint32)[0])
        assert magic == _lib.HUFF_CODEBOOK_MAGIC


def test_counts_summing_to_2_63_are_rejected():
    h = np.zeros(256, np.uint64)
    h[0] = 1 << 62
    h[1] = 1 << 62
    with pytest.raises(oracle.OracleError):
        oracle.code_lengths(h)
    with pytest.raises(_lib.HuffError) as e:
        codec.build_codebook(torch.from_numpy(h.astype(np.int64)).cuda())
    assert e.value.status == _lib.HUFF_ERR_INVALID_CODEBOOK


def test_codebook_from_lengths_round_trip_and_rejects_oversubscription():
    h = oracle.histogram(_data("gauss", 10_000))
    ln, cd = oracle_codebook(h)
    cb = codec.codebook_from_lengths(ln)
    np.testing.assert_array_equal(cb.lengths(), ln)
    np.testing.assert_array_equal(cb.codes(), cd)
    bad = np.zeros(256, np.uint8)
    bad[:3] = 1
    with pytest.raises(_lib.HuffError) as e:
        codec.codebook_from_lengths(bad)
    assert e.value.status == _lib.HUFF_ERR_INVALID_CODEBOOK


# ------------------------------------------------------------------ encode / decode
SIZES = [1, 2, 100, 8191, 8192, 8193, 3 * 8192 + 123, 65536 + 4096 + 17, 300_001]


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("kind", ["gauss", "uniform", "single", "skew"])
@pytest.mark.parametrize("chunk", [32, 96, 256, 4064, 4096, 16384])  # multiples of 32, some not of 64
def test_encode_decode_bit_exact(n, kind, chunk):
    x = _data(kind, n)
    h = oracle.histogram(x)
    ln, cd = oracle_codebook(h)
    ref_pay, ref_off = oracle.encode(x, ln, cd, chunk)
    d = dev_u8(x)
    cb = codec.build_codebook(codec.histogram(d))
    np.testing.assert_array_equal(cb.lengths(), ln)
    s = codec.encode(d, cb, chunk)
    assert_stream_equal(s, ref_pay, ref_off)
    np.testing.assert_array_equal(host(codec.decode(s, cb)), x)


def test_encode_empty():
    cb = codec.build_codebook(codec.histogram(dev_u8(np.arange(256, dtype=np.uint8))))
    s = codec.encode(torch.empty(0, dtype=torch.uint8, device="cuda"), cb, 4096)
    assert host(s.off).tolist() == [0]
    out = codec.decode(s, cb)
    assert out.numel() == 0


def test_length_limited_codebook_end_to_end():
    # Fibonacci-like frequencies force the 24-bit limit; encode every symbol, long codes included
    fib = [1, 1]
    while len(fib) < 34:
        fib.append(fib[-1] + fib[-2])
    x = np.repeat(np.arange(34, dtype=np.uint8), [min(f, 5000) for f in fib])
    RNG.shuffle(x)
    h = np.zeros(256, np.uint64)
    h[:34] = fib
    ln, cd = oracle_codebook(h)
    assert int(ln.max()) == 24
    Hd = torch.from_numpy(h.astype(np.int64)).cuda()
    cb = codec.build_codebook(Hd)
    np.testing.assert_array_equal(cb.lengths(), ln)
    ref_pay, ref_off = oracle.encode(x, ln, cd, 1024)
    s = codec.encode(dev_u8(x), cb, 1024)
    assert_stream_equal(s, ref_pay, ref_off)
    np.testing.assert_array_equal(host(codec.decode(s, cb)), x)


@pytest.mark.parametrize("chunk", [256, 16384])
def test_gpu_decodes_oracle_payload(chunk):
    x = _data("wide", 123_457)
    ln, cd = oracle_codebook(oracle.histogram(x))
    pay, off = oracle.encode(x, ln, cd, chunk)
    cb = codec.codebook_from_lengths(ln)
    pd = torch.zeros(((pay.size + 15) // 16) * 16, dtype=torch.uint8, device="cuda")
    pd[: pay.size] = dev_u8(pay)
    s = codec.Stream(pd, torch.from_numpy(off.astype(np.int64)).cuda(), x.size, chunk)
    out = torch.empty(x.size, dtype=torch.uint8, device="cuda")
    st = codec.new_status()
    _lib.huff_decode(pd, s.off, x.size, chunk, cb.buf, out, st, payload_bytes=pay.size)
    codec.raise_on_status(st, "decode")
    np.testing.assert_array_equal(host(out), x)


# ------------------------------------------------------------------ device-side errors (made on the host)
def test_symbol_not_in_codebook_sets_status():
    x = _data("gauss", 20_000)
    cb = codec.build_codebook(codec.histogram(dev_u8(x[:1000])))
    ln = cb.lengths()
    y = x.copy()
    missing = np.flatnonzero(ln == 0)
    y[5000] = missing[0]
    with pytest.raises(_lib.HuffError) as e:
        codec.encode(dev_u8(y), cb, 4096)
    assert e.value.status == _lib.HUFF_ERR_SYMBOL_NOT_IN_CODEBOOK


def test_payload_too_small_sets_status():
    x = _data("uniform", 50_000)
    d = dev_u8(x)
    cb = codec.build_codebook(codec.histogram(d))
    payload = torch.empty(1024, dtype=torch.uint8, device="cuda")
    off = torch.empty(_lib.huff_num_chunks(x.size, 4096) + 1, dtype=torch.int64, device="cuda")
    ws = torch.empty(_lib.huff_workspace_size(x.size, 4096) // 8 + 2, dtype=torch.int64, device="cuda")
    st = codec.new_status()
    _lib.huff_encode(d, cb.buf, 4096, payload, off, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == _lib.HUFF_ERR_BUFFER_TOO_SMALL


def test_corrupt_offsets_and_truncation_detected():
    x = _data("gauss", 40_000)
    d = dev_u8(x)
    cb = codec.build_codebook(codec.histogram(d))
    s = codec.encode(d, cb, 4096)
    bad = codec.Stream(s.payload, s.off.clone(), s.n, s.chunk_bytes)
    bad.off[3] += 1
    with pytest.raises(_lib.HuffError) as e:
        codec.decode(bad, cb)
    assert e.value.status == _lib.HUFF_ERR_CORRUPT_STREAM
    out = torch.empty(x.size, dtype=torch.uint8, device="cuda")
    st = codec.new_status()
    _lib.huff_decode(s.payload, s.off, s.n, 4096, cb.buf, out, st, payload_bytes=s.nbytes() - 64)
    torch.cuda.synchronize()
    assert int(st.item()) == _lib.HUFF_ERR_CORRUPT_STREAM


def test_chunk_bit_counts_out_of_range_and_empty_payload_are_corrupt():
    """Codes are 1 to 24 bits long, so a chunk of c symbols spans c to 24 c bits; the decoder
    rejects any other chunk before it reads anything, which also covers an empty payload."""
    x = _data("gauss", 40_000)
    d = dev_u8(x)
    cb = codec.build_codebook(codec.histogram(d))
    s = codec.encode(d, cb, 4096)
    out = torch.empty(x.size, dtype=torch.uint8, device="cuda")
    for span in (4095, 24 * 4096 + 1):  # chunk 1: 4096 symbols in fewer than 1 or more than 24 bits each
        off = s.off.clone()
        off[2] = off[1] + span
        assert int(off[2]) <= 8 * s.nbytes()
        st = codec.new_status()
        _lib.huff_decode(s.payload, off, s.n, 4096, cb.buf, out, st, payload_bytes=s.nbytes())
        torch.cuda.synchronize()
        assert int(st.item()) == _lib.HUFF_ERR_CORRUPT_STREAM
    zero = torch.zeros_like(s.off)
    st = codec.new_status()
    _lib.huff_decode(s.payload, zero, s.n, 4096, cb.buf, out, st, payload_bytes=0)
    torch.cuda.synchronize()
    assert int(st.item()) == _lib.HUFF_ERR_CORRUPT_STREAM


@pytest.mark.parametrize("fixed", [False, True])
def test_container_round_trip(fixed):
    """Encode on the GPU, serialise to host bytes, parse, upload and decode: per-shard mode carries
    the lengths (the codebook is imported from them), fixed mode relies on the receiver's codebook."""
    x = _data("gauss", 300_001)
    d = dev_u8(x)
    cb = codec.build_codebook(codec.histogram(d), flags=_lib.HUFF_COVER_ALL if fixed else 0)
    s = codec.encode(d, cb, 16384)
    buf = codec.to_container(s, None if fixed else cb)
    s2, cb2 = codec.from_container(buf, cb if fixed else None)
    if not fixed:
        np.testing.assert_array_equal(cb2.lengths(), cb.lengths())
    assert torch.equal(s2.off, s.off)
    np.testing.assert_array_equal(host_u8(codec.decode(s2, cb2)), x)
    with pytest.raises(ValueError):
        codec.from_container(codec.to_container(s, None))


def test_unbuilt_codebook_is_rejected():
    cb = codec.Codebook()
    with pytest.raises(_lib.HuffError) as e:
        codec.encode(dev_u8(_data("gauss", 1000)), cb, 256)
    assert e.value.status in (_lib.HUFF_ERR_INVALID_CODEBOOK, _lib.HUFF_ERR_SYMBOL_NOT_IN_CODEBOOK)


def test_host_side_argument_errors():
    cb = codec.build_codebook(codec.histogram(dev_u8(np.arange(256, dtype=np.uint8))))
    x = dev_u8(np.zeros(4096, np.uint8))
    with pytest.raises(_lib.HuffError) as e:
        codec.encode(x, cb, 1000)          # chunk not a multiple of 32
    assert e.value.status == _lib.HUFF_ERR_INVALID_ARG
    with pytest.raises(_lib.HuffError):
        codec.encode(x[1:], cb, 4096)      # misaligned input
    h = torch.zeros(256, dtype=torch.int64, device="cuda")
    with pytest.raises(_lib.HuffError):
        _lib.huff_build_codebook(h, cb.buf, codec.new_status(), max_len=25)


# ------------------------------------------------------------------ byte grouping and delta
def test_split_merge_xor_exhaustive():
    w = np.arange(1 << 16, dtype=np.uint16)
    b = RNG.permutation(w)
    dw = torch.from_numpy(w.view(np.int16)).cuda()
    db = torch.from_numpy(b.view(np.int16)).cuda()
    hi = torch.empty(w.size, dtype=torch.uint8, device="cuda")
    lo = torch.empty_like(hi)
    _lib.lmc_bytegroup_split(dw, hi, lo)
    rh, rl = oracle.bytegroup_split(w)
    np.testing.assert_array_equal(host(hi), rh)
    np.testing.assert_array_equal(host(lo), rl)
    back = torch.empty_like(dw)
    _lib.lmc_bytegroup_merge(hi, lo, back)
    np.testing.assert_array_equal(host_u8(back).view(np.uint16), w)
    d = torch.empty_like(dw)
    _lib.lmc_delta_xor(dw, db, d)
    np.testing.assert_array_equal(host_u8(d).view(np.uint16), oracle.delta_xor(w, b))
    _lib.lmc_delta_xor(d, db, d)  # in place, self-inverse
    np.testing.assert_array_equal(host_u8(d).view(np.uint16), w)


@pytest.mark.parametrize("n", [1, 7, 15, 17, 33, 1001])
def test_split_merge_odd_sizes_and_offsets(n):
    w = RNG.integers(0, 1 << 16, n + 3, dtype=np.uint16)
    dw = torch.from_numpy(w.view(np.int16)).cuda()
    hi = torch.empty(n + 3, dtype=torch.uint8, device="cuda")
    lo = torch.empty_like(hi)
    _lib.lmc_bytegroup_split(dw[1:n + 1], hi[2:n + 2], lo[1:n + 1])  # unaligned views take the scalar path
    rh, rl = oracle.bytegroup_split(w[1:n + 1])
    np.testing.assert_array_equal(host(hi[2:n + 2]), rh)
    np.testing.assert_array_equal(host(lo[1:n + 1]), rl)


# ------------------------------------------------------------------ fused bf16 paths
def _bf16_pair(n, rng):
    x0 = torch.from_numpy((rng.normal(0, 0.02, n)).astype(np.float32)).to(torch.bfloat16)
    x1 = (x0.float() + torch.from_numpy(rng.normal(0, 1e-4, n).astype(np.float32))).to(torch.bfloat16)
    return x0, x1


@pytest.mark.parametrize("n", [1, 8, 4095, 4096, 4097, 3 * 4096 + 77, 100_001])
@pytest.mark.parametrize("delta", [False, True])
@pytest.mark.parametrize("chunk", [96, 256, 14688, 16384])  # 96 and 14 688 are multiples of 32, not of 256
def test_fused_bf16_matches_split_then_encode(n, delta, chunk):
    rng = np.random.default_rng(n + delta)
    x0, x1 = _bf16_pair(n, rng)
    w = x1.view(torch.int16).numpy().view(np.uint16)
    if delta:
        w = oracle.delta_xor(w, x0.view(torch.int16).numpy().view(np.uint16))
    hi, lo = oracle.bytegroup_split(w)
    refs = []
    for plane in (hi, lo):
        ln, cd = oracle_codebook(oracle.histogram(plane))
        refs.append((ln, cd) + oracle.encode(plane, ln, cd, chunk))
    dx1, dx0 = x1.cuda(), x0.cuda()
    # fused histogram
    hh = torch.empty(256, dtype=torch.int64, device="cuda")
    hl = torch.empty(256, dtype=torch.int64, device="cuda")
    _lib.lmc_histogram_bf16(dx1.view(torch.int16), dx0.view(torch.int16) if delta else None, hh, hl)
    np.testing.assert_array_equal(host(hh).astype(np.uint64), oracle.histogram(hi))
    np.testing.assert_array_equal(host(hl).astype(np.uint64), oracle.histogram(lo))
    s = codec.compress_bf16(dx1, dx0 if delta else None, chunk)
    for (ln, cd, pay, off), cb, st in ((refs[0], s.cb_hi, s.hi), (refs[1], s.cb_lo, s.lo)):
        np.testing.assert_array_equal(cb.lengths(), ln)
        assert_stream_equal(st, pay, off)
    back = codec.decompress_bf16(s, dx0 if delta else None)
    assert torch.equal(back.view(torch.int16).cpu(), x1.view(torch.int16))


def test_fused_bf16_specials_round_trip():
    vals = torch.tensor([0.0, -0.0, float("inf"), float("-inf"), float("nan"), 1e-40, -3.5, 65504.0] * 1000,
                        dtype=torch.bfloat16)
    x0 = torch.zeros_like(vals)
    s = codec.compress_bf16(vals.cuda(), x0.cuda(), 256)
    back = codec.decompress_bf16(s, x0.cuda())
    assert torch.equal(back.view(torch.int16).cpu(), vals.view(torch.int16))


def test_build_codebooks_batch_equals_single_builds():
    rng = np.random.default_rng(17)
    hists = []
    for k in range(5):
        h = rng.integers(0, 1000, 256).astype(np.int64)
        h[rng.random(256) < 0.3 * k / 4] = 0  # some symbols absent
        hists.append(h)
    hists[3][:] = 0
    hists[3][7] = 5  # one symbol
    hists[4][:] = 0  # empty
    H = torch.from_numpy(np.stack(hists)).cuda()
    cbs = codec.build_codebooks(H, 24, 0)
    for k in range(5):
        one = codec.build_codebook(H[k].clone(), 24, 0)
        assert torch.equal(cbs[k].buf, one.buf)
        np.testing.assert_array_equal(cbs[k].lengths(), oracle.code_lengths(hists[k].astype(np.uint64), 24))


def test_build_codebooks_arguments():
    H = torch.zeros((2, 256), dtype=torch.int64, device="cuda")
    bufs = torch.zeros((2, _lib.huff_codebook_size()), dtype=torch.uint8, device="cuda")
    st = codec.new_status()
    with pytest.raises(_lib.HuffError) as e:
        _lib.huff_build_codebooks(H, bufs, st, 40, 0)  # max_len out of range
    assert e.value.status == _lib.HUFF_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        _lib.huff_build_codebooks(H, bufs[:1], st, 24, 0)
