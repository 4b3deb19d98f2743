"""The five workloads at their full sizes, through the C ABI, in the launch
configuration the benchmark uses (16 KiB chunks, 14 688-element chunks for the
snapshot delta; max length 24).

At these sizes the oracle cannot encode whole tensors in seconds, so the
checks are:
- histograms equal torch.bincount of the same bytes (a library routine, no
  code shared with either side), drawn in blocks;
- codebooks equal the oracle's, built from those exact histograms;
- sampled chunks (first, second, middle, last and random ones) equal the
  oracle's encoding of that chunk's symbols alone, bit for bit;
- the total bit count equals sum(hist * len) (true at any size);
- every chunk's offset difference equals the sum of its symbols' code
  lengths, gathered with torch over the whole stream (independent of the
  decoder);
- decode returns the input exactly;
- the small workloads (1 MiB) are compared whole.
"""
import numpy as np
import pytest
import torch

import oracle
from lossless_huffman_compression_gb300 import _lib, codec, workloads
from gpu_util import assert_offsets_match_lengths, assert_stream_equal, check_sampled_chunks, host, host_u8

pytestmark = pytest.mark.gpu

CHUNK = 16384
SNAPSHOT_CHUNK = 14688  # the benchmark's snapshot chunk: 896-lane decode blocks on all 152 SMs
BLOCK = 1 << 27


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    _lib.load()
    assert torch.cuda.is_available()


def _bincount_u8(x: torch.Tensor) -> np.ndarray:
    flat = x.reshape(-1).view(torch.uint8)
    h = torch.zeros(256, dtype=torch.int64, device=flat.device)
    for s in range(0, flat.numel(), BLOCK):
        h += torch.bincount(flat[s:s + BLOCK].to(torch.int32), minlength=256)
    return host(h).astype(np.uint64)


def _bincount_planes(w16: torch.Tensor):
    flat = w16.reshape(-1).view(torch.int16)
    hh = torch.zeros(256, dtype=torch.int64, device=flat.device)
    hl = torch.zeros(256, dtype=torch.int64, device=flat.device)
    for s in range(0, flat.numel(), BLOCK):
        v = flat[s:s + BLOCK].to(torch.int32) & 0xFFFF
        hh += torch.bincount(v >> 8, minlength=256)
        hl += torch.bincount(v & 0xFF, minlength=256)
    return host(hh).astype(np.uint64), host(hl).astype(np.uint64)


def _sample_chunks(n_chunks: int, seed: int, k: int = 6):
    rng = np.random.default_rng(seed)
    fixed = {0, min(1, n_chunks - 1), n_chunks // 2, n_chunks - 1}
    return sorted(fixed | set(int(c) for c in rng.integers(0, n_chunks, k)))


def _chunk_symbols(x_u8: torch.Tensor, chunks, chunk: int) -> dict:
    """Host copies of the sampled chunks' symbols, by chunk index."""
    n = x_u8.numel()
    out = {}
    for c in chunks:
        out[c] = host(x_u8[c * chunk: min(n, (c + 1) * chunk)])
    return out


def _check_stream_samples(payload: torch.Tensor, off: torch.Tensor, sym_of_chunk: dict, ln, cd, chunk: int):
    offs = host(off).astype(np.uint64)
    for c, s in sym_of_chunk.items():
        lo, hi = int(offs[c]), int(offs[c + 1])
        b0, b1 = lo // 8, (hi + 7) // 8
        pay = host(payload[b0:b1 + 1])
        # re-base the chunk's bits at bit (lo - 8 b0) of the copied bytes
        check_sampled_chunks(pay, np.array([lo - 8 * b0, hi - 8 * b0], dtype=np.uint64), s, ln, cd, chunk, [0])


def _total_bits(hist: np.ndarray, ln: np.ndarray) -> int:
    return int(oracle.total_bits(hist, ln))


# ------------------------------------------------------------------ per-shard int8, 1 MiB: whole comparison
def test_per_shard_int8_whole():
    x = workloads.per_shard_int8(device="cuda")
    xb = host_u8(x)
    ln = oracle.code_lengths(oracle.histogram(xb))
    cd = oracle.canonical_codes(ln)
    ref_pay, ref_off = oracle.encode(xb, ln, cd, CHUNK)
    cb, s = codec.compress(x, CHUNK)
    np.testing.assert_array_equal(cb.lengths(), ln)
    assert_stream_equal(s, ref_pay, ref_off)
    assert torch.equal(codec.decode(s, cb), x.view(torch.uint8))
    # ratio against the entropy: mean length within [H, H + 1)
    H = oracle.entropy(oracle.histogram(xb))
    L = int(ref_off[-1]) / xb.size
    assert H <= L < H + 1


# ------------------------------------------------------------------ fixed codebook: 16 warm-up + 64 test shards
def test_fixed_codebook_shards():
    hist = torch.zeros(256, dtype=torch.int64, device="cuda")
    ref = np.zeros(256, dtype=np.uint64)
    for k in range(workloads.WARMUP_SHARDS):
        w = workloads.fixed_codebook_shard(k, warmup=True, device="cuda")
        codec.histogram(w, hist, accumulate=True)
        ref += oracle.histogram(host_u8(w))
    np.testing.assert_array_equal(host(hist).astype(np.uint64), ref)
    ln = oracle.code_lengths(ref, 24, oracle.REF_COVER_ALL)
    cd = oracle.canonical_codes(ln)
    cb = codec.build_codebook(hist, 24, _lib.HUFF_COVER_ALL)
    np.testing.assert_array_equal(cb.lengths(), ln)
    for k in range(workloads.TEST_SHARDS):
        x = workloads.fixed_codebook_shard(k, warmup=False, device="cuda")
        s = codec.encode(x, cb, CHUNK)
        xb = x.reshape(-1).view(torch.uint8)
        h = _bincount_u8(xb)
        assert s.total_bits() == _total_bits(h, ln)
        if k < 2:  # two shards compared whole
            ref_pay, ref_off = oracle.encode(host(xb), ln, cd, CHUNK)
            assert_stream_equal(s, ref_pay, ref_off)
        else:
            chunks = _sample_chunks(s.n_chunks(), k, 2)
            _check_stream_samples(s.payload, s.off, _chunk_symbols(xb, chunks, CHUNK), ln, cd, CHUNK)
            assert_offsets_match_lengths(s.off, lambda a, b: xb[a:b], xb.numel(), ln, CHUNK)
        assert torch.equal(codec.decode(s, cb), xb)


# ------------------------------------------------------------------ bf16 tensors: weights (1 GiB) and snapshot delta (4 GB)
def _bf16_config(w: torch.Tensor, x0, chunk: int = CHUNK):
    w16 = w.reshape(-1).view(torch.int16)
    d16 = w16 if x0 is None else (w16 ^ x0.reshape(-1).view(torch.int16))
    hh, hl = _bincount_planes(d16)
    s = codec.compress_bf16(w, x0, chunk)
    for hist, cb, st, shift in ((hh, s.cb_hi, s.hi, 8), (hl, s.cb_lo, s.lo, 0)):
        ln = oracle.code_lengths(hist)
        cd = oracle.canonical_codes(ln)
        np.testing.assert_array_equal(cb.lengths(), ln)
        assert st.total_bits() == _total_bits(hist, ln)
        chunks = _sample_chunks(st.n_chunks(), shift + 17)
        plane = {}
        for c in chunks:
            seg = d16[c * chunk: min(s.n, (c + 1) * chunk)].to(torch.int32) & 0xFFFF
            plane[c] = host(((seg >> shift) & 0xFF).to(torch.uint8))
        _check_stream_samples(st.payload, st.off, plane, ln, cd, chunk)
        del plane
        assert_offsets_match_lengths(
            st.off, lambda a, b, sh=shift: ((d16[a:b].to(torch.int32) >> sh) & 0xFF).to(torch.uint8), s.n, ln, chunk)
    back = codec.decompress_bf16(s, x0)
    assert torch.equal(back.view(torch.int16), w16)


def test_bf16_weights_full():
    _bf16_config(workloads.bf16_weights(device="cuda"), None)


def test_snapshot_delta_full():
    x0, x1 = workloads.snapshot_pair(device="cuda")
    _bf16_config(x1, x0, SNAPSHOT_CHUNK)


# ------------------------------------------------------------------ chunk-size sweep: 16 GiB int8, fixed codebook
def test_chunk_size_sweep_16gib():
    seg_bytes = workloads.SWEEP_SEGMENT_BYTES
    n = workloads.SWEEP_SEGMENTS * seg_bytes
    x = torch.empty(n, dtype=torch.int8, device="cuda")
    for k in range(workloads.SWEEP_SEGMENTS):
        x[k * seg_bytes:(k + 1) * seg_bytes] = workloads.sweep_segment(k, device="cuda")
    xb = x.view(torch.uint8)
    head = xb[: 64 << 20]
    hist = codec.histogram(head)
    ref_head = _bincount_u8(head)
    np.testing.assert_array_equal(host(hist).astype(np.uint64), ref_head)
    ln = oracle.code_lengths(ref_head, 24, oracle.REF_COVER_ALL)
    cd = oracle.canonical_codes(ln)
    cb = codec.build_codebook(hist, 24, _lib.HUFF_COVER_ALL)
    np.testing.assert_array_equal(cb.lengths(), ln)
    T = _total_bits(_bincount_u8(xb), ln)
    out = torch.empty_like(xb)
    for chunk in (16 << 10, 64 << 10, 256 << 10, 1 << 20):
        s = codec.encode(xb, cb, chunk)
        assert s.total_bits() == T  # the payload does not depend on the chunk size
        chunks = _sample_chunks(s.n_chunks(), chunk, 3)
        _check_stream_samples(s.payload, s.off, _chunk_symbols(xb, chunks, chunk), ln, cd, chunk)
        assert_offsets_match_lengths(s.off, lambda a, b: xb[a:b], n, ln, chunk)
        codec.decode(s, cb, out=out)
        assert torch.equal(out, xb)
        del s
        torch.cuda.empty_cache()
