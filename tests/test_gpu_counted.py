"""The counted per-shard bf16 path (per-segment counts from the histogram
pass, one-pass encode) against the oracle and against the two-pass encode,
element by element, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from lossless_huffman_compression_gb300 import _lib, codec
from gpu_util import assert_offsets_match_lengths, assert_stream_equal, check_sampled_chunks, host, oracle_codebook

pytestmark = pytest.mark.gpu

SEG = _lib.HUFF_COUNT_SEGMENT


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    _lib.load()
    assert torch.cuda.is_available()


def _pair(n, rng, sigma_noise=1e-4):
    x0 = torch.from_numpy(rng.normal(0, 0.02, n).astype(np.float32)).to(torch.bfloat16)
    x1 = (x0.float() + torch.from_numpy(rng.normal(0, sigma_noise, n).astype(np.float32))).to(torch.bfloat16)
    return x0, x1


def _counted(dx1, dx0, chunk, cb_hi=None, cb_lo=None):
    n = dx1.numel()
    w16 = dx1.view(torch.int16)
    x16 = None if dx0 is None else dx0.view(torch.int16)
    hh = torch.empty(256, dtype=torch.int64, device="cuda")
    hl = torch.empty(256, dtype=torch.int64, device="cuda")
    seg = torch.full((max(_lib.lmc_segment_counts_size(n), 4) // 4,), -1, dtype=torch.int32, device="cuda")
    _lib.lmc_histogram_bf16_counted(w16, x16, hh, hl, seg)
    if cb_hi is None:
        cb_hi = codec.build_codebook(hh)
        cb_lo = codec.build_codebook(hl)
    cap = _lib.huff_encode_bound(n, 24)
    nc = _lib.huff_num_chunks(n, chunk)
    p_hi = torch.empty(cap, dtype=torch.uint8, device="cuda")
    p_lo = torch.empty(cap, dtype=torch.uint8, device="cuda")
    o_hi = torch.empty(nc + 1, dtype=torch.int64, device="cuda")
    o_lo = torch.empty(nc + 1, dtype=torch.int64, device="cuda")
    ws = torch.empty(max(_lib.lmc_counted_workspace_size(n), 16) // 8, dtype=torch.int64, device="cuda")
    st = codec.new_status()
    _lib.lmc_encode_bf16_counted(w16, x16, cb_hi.buf, cb_lo.buf, chunk, seg, p_hi, o_hi, p_lo, o_lo, ws, st)
    torch.cuda.synchronize()
    return (hh, hl, seg, cb_hi, cb_lo, codec.Stream(p_hi, o_hi, n, chunk), codec.Stream(p_lo, o_lo, n, chunk),
            int(st.item()))


@pytest.mark.parametrize("n", [1, 8, 4097, SEG - 1, SEG, SEG + 1, 3 * SEG + 4097, 1_000_003])
@pytest.mark.parametrize("delta", [False, True])
@pytest.mark.parametrize("chunk", [96, 256, 16384])
def test_counted_matches_oracle_and_two_pass(n, delta, chunk):
    rng = np.random.default_rng(n * 2 + delta)
    x0, x1 = _pair(n, rng)
    w = x1.view(torch.int16).numpy().view(np.uint16)
    if delta:
        w = oracle.delta_xor(w, x0.view(torch.int16).numpy().view(np.uint16))
    hi, lo = oracle.bytegroup_split(w)
    dx1, dx0 = x1.cuda(), (x0.cuda() if delta else None)
    hh, hl, seg, cb_hi, cb_lo, s_hi, s_lo, st = _counted(dx1, dx0, chunk)
    assert st == 0
    np.testing.assert_array_equal(host(hh).astype(np.uint64), oracle.histogram(hi))
    np.testing.assert_array_equal(host(hl).astype(np.uint64), oracle.histogram(lo))
    counts = host(seg).view(np.uint32)
    S = _lib.lmc_count_segment(n)
    assert S == SEG  # inputs this small keep the least segment size
    n_seg = (n + S - 1) // S
    for s in range(n_seg):
        np.testing.assert_array_equal(counts[s * 512:s * 512 + 256].astype(np.uint64),
                                      oracle.histogram(hi[s * S:(s + 1) * S]))
        np.testing.assert_array_equal(counts[s * 512 + 256:s * 512 + 512].astype(np.uint64),
                                      oracle.histogram(lo[s * S:(s + 1) * S]))
    for plane, cb, stream in ((hi, cb_hi, s_hi), (lo, cb_lo, s_lo)):
        ln, cd = oracle_codebook(oracle.histogram(plane))
        np.testing.assert_array_equal(cb.lengths(), ln)
        pay, off = oracle.encode(plane, ln, cd, chunk)
        assert_stream_equal(stream, pay, off)
    # byte-identical to the two-pass encode with the same codebooks
    two = codec.compress_bf16(dx1, dx0, chunk, cb_hi=cb_hi, cb_lo=cb_lo)
    for a, b in ((two.hi, s_hi), (two.lo, s_lo)):
        assert torch.equal(a.off, b.off)
        nb = (a.total_bits() + 7) // 8
        assert torch.equal(a.payload[:nb], b.payload[:nb])
    back = codec.decompress_bf16(codec.Bf16Streams(cb_hi, cb_lo, s_hi, s_lo, n), dx0)
    assert torch.equal(back.view(torch.int16).cpu(), x1.view(torch.int16))


def _enc_warps():  # the counted encode: one CTA of 20 warps per SM
    return torch.cuda.get_device_properties(0).multi_processor_count * 20


@pytest.mark.parametrize("n", [0, 1, SEG, 398_458_879, 398_458_880, 400_000_003, 2_000_027_648, 1 << 34])
def test_count_segment_gives_every_encode_warp_the_same_rounds(n):
    """lmc_count_segment: SEG while the encode's warps outnumber SEG-element segments; otherwise the
    smallest whole number of 512-element tiles that splits the input into at most warps x rounds
    segments, rounds = floor(tiles / (256 warps))."""
    S = _lib.lmc_count_segment(n)
    warps = _enc_warps()
    tiles = -(-n // 512)
    rounds = tiles // (256 * warps)
    if rounds == 0:
        assert S == SEG
        return
    assert S % 512 == 0 and SEG <= S < 2 * SEG
    st = S // 512
    assert -(-tiles // st) <= warps * rounds < -(-tiles // (st - 1))
    if n == 2_000_027_648 and warps == 152 * 20:
        assert S == 257 * 512 and -(-n // S) == 15200  # exactly 5 rounds of 3040 warps


def test_counted_segments_above_the_least_size():
    """A 400 M-element delta, where segments are longer than SEG: sampled segments' counts equal
    torch.bincount of their bytes, every chunk's offset difference equals its symbols' summed code
    lengths, sampled chunks equal the oracle's encoding, and the decode is exact."""
    n = 400_000_003
    S = _lib.lmc_count_segment(n)
    if S == SEG:
        pytest.skip("this GPU keeps the least segment size at this n")
    g = torch.Generator(device="cuda").manual_seed(11)
    x0 = (torch.randn(n, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    x1 = (x0.float() + torch.randn(n, device="cuda", generator=g) * 1e-4).to(torch.bfloat16)
    chunk = 16384
    hh, hl, seg, cb_hi, cb_lo, s_hi, s_lo, st = _counted(x1, x0, chunk)
    assert st == 0
    d16 = (x1.view(torch.int16) ^ x0.view(torch.int16)).to(torch.int32) & 0xFFFF
    counts = seg.view(torch.int32)
    n_seg = -(-n // S)
    for s in sorted({0, 1, n_seg // 2, n_seg - 1}):
        v = d16[s * S:min(n, (s + 1) * S)]
        for plane, sh in ((0, 8), (1, 0)):
            want = torch.bincount((v >> sh) & 0xFF, minlength=256)
            got = counts[s * 512 + 256 * plane: s * 512 + 256 * plane + 256].to(torch.int64)
            assert torch.equal(got, want), (s, plane)
    for hist, cb, stream, sh in ((hh, cb_hi, s_hi, 8), (hl, cb_lo, s_lo, 0)):
        ln, cd = oracle_codebook(host(hist).astype(np.uint64))
        np.testing.assert_array_equal(cb.lengths(), ln)
        sym = lambda a, b, sh=sh: ((d16[a:b] >> sh) & 0xFF).to(torch.uint8)
        assert_offsets_match_lengths(stream.off, sym, n, ln, chunk)
        offs = host(stream.off).astype(np.uint64)
        nc = stream.n_chunks()
        for c in sorted({0, nc // 3, nc - 1}):
            lo, hi = int(offs[c]), int(offs[c + 1])
            b0, b1 = lo // 8, (hi + 7) // 8
            pay = host(stream.payload[b0:b1 + 1])
            check_sampled_chunks(pay, np.array([lo - 8 * b0, hi - 8 * b0], dtype=np.uint64),
                                 host(sym(c * chunk, min(n, (c + 1) * chunk))), ln, cd, chunk, [0])
    back = codec.decompress_bf16(codec.Bf16Streams(cb_hi, cb_lo, s_hi, s_lo, n), x0)
    assert torch.equal(back.view(torch.int16), x1.view(torch.int16))


def test_counted_compress_bf16_round_trip_wide_noise():
    # larger noise: longer codes and more long (> 12 bit) codes in the low plane
    rng = np.random.default_rng(7)
    x0, x1 = _pair(2 * SEG + 333, rng, sigma_noise=3e-3)
    s = codec.compress_bf16(x1.cuda(), x0.cuda(), 4096)
    back = codec.decompress_bf16(s, x0.cuda())
    assert torch.equal(back.view(torch.int16).cpu(), x1.view(torch.int16))


def test_counted_symbol_without_code_sets_status():
    rng = np.random.default_rng(11)
    x0, x1 = _pair(SEG + 5, rng)
    # codebooks from a histogram that lacks most symbols
    h = torch.zeros(256, dtype=torch.int64, device="cuda")
    h[0] = 10
    h[1] = 3
    cb = codec.build_codebook(h)
    *_, st = _counted(x1.cuda(), x0.cuda(), 4096, cb_hi=cb, cb_lo=cb)
    assert st == _lib.HUFF_ERR_SYMBOL_NOT_IN_CODEBOOK


def test_counted_argument_errors():
    n = 4096
    w = torch.zeros(n + 8, dtype=torch.int16, device="cuda")
    hh = torch.zeros(256, dtype=torch.int64, device="cuda")
    hl = torch.zeros(256, dtype=torch.int64, device="cuda")
    seg = torch.zeros(512, dtype=torch.int32, device="cuda")
    small = torch.zeros(100, dtype=torch.int32, device="cuda")
    with pytest.raises(_lib.HuffError) as e:
        _lib.lmc_histogram_bf16_counted(w[:n], None, hh, hl, small)
    assert e.value.status == _lib.HUFF_ERR_BUFFER_TOO_SMALL
    with pytest.raises(_lib.HuffError) as e:
        _lib.lmc_histogram_bf16_counted(w[1:n + 1], None, hh, hl, seg)  # 2-byte offset: not 16-byte aligned
    assert e.value.status == _lib.HUFF_ERR_INVALID_ARG
    with pytest.raises(_lib.HuffError) as e:
        _lib.lmc_histogram_bf16_counted(w[:n], None, hh, hh, seg)
    assert e.value.status == _lib.HUFF_ERR_INVALID_ARG


def _long_code_plane(n, rng):
    """Bytes with geometric counts (code lengths up to about 19 bits) where the rarest
    symbols sit next to each other, so some pairs of codes are longer than 31 bits."""
    counts = [1 << (18 - k) for k in range(1, 13)]
    vals = np.concatenate([np.full(c, k + 1, np.uint8) for k, c in enumerate(counts)])
    vals = np.concatenate([vals, np.zeros(n - vals.size, np.uint8)])
    rng.shuffle(vals)
    pos = rng.choice(n // 2 - 1, 40, replace=False) * 2
    vals[pos] = rng.integers(14, 20, 40)
    vals[pos + 1] = rng.integers(14, 20, 40)
    return vals


def test_counted_long_code_pairs():
    # pairs of codes longer than 31 bits make warps take the one-code-at-a-time path; ragged last tile
    n = 3 * SEG + 1000
    rng = np.random.default_rng(21)
    hi_b, lo_b = _long_code_plane(n, rng), _long_code_plane(n, rng)
    w = (hi_b.astype(np.uint16) << 8) | lo_b
    x1 = torch.from_numpy(w.view(np.int16).copy()).view(torch.bfloat16)
    hi, lo = oracle.bytegroup_split(w)
    hh, hl, seg, cb_hi, cb_lo, s_hi, s_lo, st = _counted(x1.cuda(), None, 4096)
    assert st == 0
    for plane, cb, stream in ((hi, cb_hi, s_hi), (lo, cb_lo, s_lo)):
        ln, cd = oracle_codebook(oracle.histogram(plane))
        pair_len = ln[plane[: n // 2 * 2]].astype(np.int64).reshape(-1, 2).sum(1)
        assert pair_len.max() > 31  # the case under test is present
        np.testing.assert_array_equal(cb.lengths(), ln)
        pay, off = oracle.encode(plane, ln, cd, 4096)
        assert_stream_equal(stream, pay, off)
    back = codec.decompress_bf16(codec.Bf16Streams(cb_hi, cb_lo, s_hi, s_lo, n), None)
    assert torch.equal(back.view(torch.int16).cpu(), x1.view(torch.int16))


def test_counted_counts_of_other_data_set_status():
    # counts recorded for x, encode of x reversed (same symbols, other per-segment counts)
    n = 4 * SEG
    rng = np.random.default_rng(5)
    x0, x1 = _pair(n, rng, sigma_noise=3e-3)
    dx1 = x1.cuda()
    w16 = dx1.view(torch.int16)
    hh = torch.empty(256, dtype=torch.int64, device="cuda")
    hl = torch.empty(256, dtype=torch.int64, device="cuda")
    seg = torch.empty(_lib.lmc_segment_counts_size(n) // 4, dtype=torch.int32, device="cuda")
    _lib.lmc_histogram_bf16_counted(w16, None, hh, hl, seg)
    cb_hi, cb_lo = codec.build_codebook(hh), codec.build_codebook(hl)
    other = torch.flip(w16, [0]).contiguous()
    cap = _lib.huff_encode_bound(n, 24)
    nc = _lib.huff_num_chunks(n, 4096)
    p_hi = torch.empty(cap, dtype=torch.uint8, device="cuda")
    p_lo = torch.empty(cap, dtype=torch.uint8, device="cuda")
    o_hi = torch.empty(nc + 1, dtype=torch.int64, device="cuda")
    o_lo = torch.empty(nc + 1, dtype=torch.int64, device="cuda")
    ws = torch.empty(_lib.lmc_counted_workspace_size(n) // 8 + 2, dtype=torch.int64, device="cuda")
    st = codec.new_status()
    _lib.lmc_encode_bf16_counted(other, None, cb_hi.buf, cb_lo.buf, 4096, seg, p_hi, o_hi, p_lo, o_lo, ws, st)
    assert int(st.item()) == _lib.HUFF_ERR_INVALID_ARG


@pytest.mark.parametrize("run_byte", [0x00, 0x3C, 0xFF])
def test_runs_of_a_nonzero_one_bit_symbol(run_byte):
    # the high plane is mostly one byte value (a 1-bit code) in runs of every length; decode
    # emits long runs of that code at once, whatever the byte is
    n = 2 * SEG + 777
    rng = np.random.default_rng(run_byte)
    hi_b = np.full(n, run_byte, np.uint8)
    breaks = rng.random(n) < rng.choice([0.01, 0.05, 0.2], n)
    hi_b[breaks] = rng.integers(0, 256, int(breaks.sum()))
    lo_b = rng.integers(0, 256, n).astype(np.uint8)
    w = (hi_b.astype(np.uint16) << 8) | lo_b
    x1 = torch.from_numpy(w.view(np.int16).copy()).view(torch.bfloat16)
    hi, lo = oracle.bytegroup_split(w)
    for chunk in (256, 4096):
        hh, hl, seg, cb_hi, cb_lo, s_hi, s_lo, st = _counted(x1.cuda(), None, chunk)
        assert st == 0
        ln, cd = oracle_codebook(oracle.histogram(hi))
        assert ln[run_byte] == 1
        pay, off = oracle.encode(hi, ln, cd, chunk)
        assert_stream_equal(s_hi, pay, off)
        back = codec.decompress_bf16(codec.Bf16Streams(cb_hi, cb_lo, s_hi, s_lo, n), None)
        assert torch.equal(back.view(torch.int16).cpu(), x1.view(torch.int16))
        # the byte-stream decoder on the high plane alone
        cb, s = codec.compress(torch.from_numpy(hi).cuda(), chunk)
        assert torch.equal(codec.decode(s, cb).cpu(), torch.from_numpy(hi))


def test_counted_more_segments_than_the_scan_holds_in_registers():
    # 16 385 segments: the segment scan's threads take runs longer than they keep in registers
    n = 16385 * SEG + 7
    g = torch.Generator(device="cuda")
    g.manual_seed(12)
    x1 = (torch.randn(n, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    s = codec.compress_bf16(x1, None, 16384)  # counted path
    hh = torch.zeros(256, dtype=torch.int64, device="cuda")
    hl = torch.zeros(256, dtype=torch.int64, device="cuda")
    two = codec.compress_bf16(x1, None, 16384, cb_hi=s.cb_hi, cb_lo=s.cb_lo)  # two-pass, same codebooks
    for a, b in ((two.hi, s.hi), (two.lo, s.lo)):
        assert torch.equal(a.off, b.off)
        nb = (a.total_bits() + 7) // 8
        assert torch.equal(a.payload[:nb], b.payload[:nb])
    del two, hh, hl
    back = codec.decompress_bf16(s, None)
    assert torch.equal(back.view(torch.int16), x1.view(torch.int16))


@pytest.mark.parametrize("chunk,n", [(256, 70_001 * 256 + 77), (256, 152 * 448 * 2 * 256 + 3), (1024, 300_000 * 1024 - 5)])
@pytest.mark.parametrize("delta", [False, True])
def test_decode_more_chunk_pairs_than_one_wave(chunk, n, delta):
    # more chunk pairs than the SMs hold lanes at once: the decode runs in several waves
    g = torch.Generator(device="cuda")
    g.manual_seed(n % 1000 + delta)
    x0 = (torch.randn(n, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    x1 = (x0.float() + torch.randn(n, generator=g, device="cuda") * 3e-4).to(torch.bfloat16)
    s = codec.compress_bf16(x1, x0 if delta else None, chunk)
    back = codec.decompress_bf16(s, x0 if delta else None)
    assert torch.equal(back.view(torch.int16), x1.view(torch.int16))


# ------------------------------------------------------------------ given codebooks (the fixed-codebook mode)
@pytest.mark.parametrize("n", [1, 4097, SEG + 1, 3 * SEG + 4097])
@pytest.mark.parametrize("delta", [False, True])
def test_given_codebooks_match_oracle(n, delta):
    """lmc_encode_bf16 with codebooks fixed in advance (built, every symbol covered, from a warm-up
    pair) encodes another pair exactly as the oracle does with those lengths."""
    rng = np.random.default_rng(1000 + n + delta)
    w0, w1 = _pair(50_000, rng)  # warm-up
    x0, x1 = _pair(n, rng)
    def planes(a, b):
        w = a.view(torch.int16).numpy().view(np.uint16)
        if delta:
            w = oracle.delta_xor(w, b.view(torch.int16).numpy().view(np.uint16))
        return oracle.bytegroup_split(w)
    whi, wlo = planes(w1, w0)
    hi, lo = planes(x1, x0)
    cbs, lens = [], []
    for p in (whi, wlo):
        h = torch.from_numpy(oracle.histogram(p).astype(np.int64)).cuda()
        cbs.append(codec.build_codebook(h, 24, _lib.HUFF_COVER_ALL))
        lens.append(oracle.code_lengths(oracle.histogram(p), 24, oracle.REF_COVER_ALL))
        np.testing.assert_array_equal(cbs[-1].lengths(), lens[-1])
    dx0 = x0.cuda() if delta else None
    s = codec.compress_bf16(x1.cuda(), dx0, 4096, cb_hi=cbs[0], cb_lo=cbs[1])
    for plane, ln, stream in ((hi, lens[0], s.hi), (lo, lens[1], s.lo)):
        pay, off = oracle.encode(plane, ln, oracle.canonical_codes(ln), 4096)
        assert_stream_equal(stream, pay, off)
    back = codec.decompress_bf16(s, dx0)
    assert torch.equal(back.view(torch.int16).cpu(), x1.view(torch.int16))


def test_given_codebook_without_a_symbol_sets_status():
    rng = np.random.default_rng(12)
    x0, x1 = _pair(SEG + 77, rng)
    h = torch.zeros(256, dtype=torch.int64, device="cuda")
    h[0] = 10
    h[1] = 3
    cb = codec.build_codebook(h)
    with pytest.raises(_lib.HuffError) as e:
        codec.compress_bf16(x1.cuda(), x0.cuda(), 4096, cb_hi=cb, cb_lo=cb)
    assert e.value.status == _lib.HUFF_ERR_SYMBOL_NOT_IN_CODEBOOK


def test_given_codebooks_workspace_size_is_checked():
    n = SEG + 1
    w = torch.zeros(n, dtype=torch.int16, device="cuda")
    cb = codec.build_codebook(torch.ones(256, dtype=torch.int64, device="cuda"))
    cap = _lib.huff_encode_bound(n, 24)
    p = torch.empty(cap, dtype=torch.uint8, device="cuda")
    o = torch.empty(_lib.huff_num_chunks(n, 4096) + 1, dtype=torch.int64, device="cuda")
    need = _lib.lmc_workspace_size(n, 4096)
    assert need >= _lib.lmc_segment_counts_size(n) + _lib.lmc_counted_workspace_size(n)
    ws = torch.empty(need // 8 - 1, dtype=torch.int64, device="cuda")
    with pytest.raises(_lib.HuffError) as e:
        _lib.lmc_encode_bf16(w, None, cb.buf, cb.buf, 4096, p, o, p.clone(), o.clone(), ws, codec.new_status())
    assert e.value.status == _lib.HUFF_ERR_BUFFER_TOO_SMALL
