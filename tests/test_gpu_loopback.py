"""The one-GPU loopback link: encode with a fixed codebook, copy the stream to
other device buffers with its size read on the device, decode there.  The
copy must move exactly the stream's bytes and offsets, refuse a destination
that is too small, and work inside a captured CUDA graph."""
import numpy as np
import pytest
import torch

import oracle
from lossless_huffman_compression_gb300 import _lib, codec, workloads
from gpu_util import assert_stream_equal, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    _lib.load()
    assert torch.cuda.is_available()


@pytest.fixture(scope="module")
def fixed_cb():
    hist = torch.zeros(256, dtype=torch.int64, device="cuda")
    for k in range(4):
        codec.histogram(workloads.fixed_codebook_shard(k, warmup=True, device="cuda"), hist, accumulate=True)
    return codec.build_codebook(hist, 24, _lib.HUFF_COVER_ALL)


@pytest.mark.parametrize("n", [1, 15, 4096, 65_537, 1 << 20, 3_000_001])
@pytest.mark.parametrize("chunk", [256, 16384])
def test_loopback_round_trip(fixed_cb, n, chunk):
    x = workloads.fixed_codebook_shard(7, warmup=False, device="cuda").reshape(-1)[:n].view(torch.uint8)
    s = codec.encode(x, fixed_cb, chunk)
    marker = torch.full_like(s.payload, 0xA5)
    r = codec.stream_copy(s, dst_payload=marker)
    nw = (s.total_bits() + 31) // 32 * 4  # the stream's words
    assert torch.equal(r.off, s.off)
    assert torch.equal(r.payload[:nw], s.payload[:nw])
    assert bool((r.payload[nw:] == 0xA5).all())  # nothing past the stream's last word
    assert torch.equal(codec.decode(r, fixed_cb), x)
    # the copied stream is the oracle's stream of x under the same code lengths
    if n <= 65_537:
        ln = fixed_cb.lengths()
        pay, ref_off = oracle.encode(host(x), ln, oracle.canonical_codes(ln), chunk)
        assert_stream_equal(r, pay, ref_off)


def test_loopback_empty(fixed_cb):
    x = torch.empty(0, dtype=torch.uint8, device="cuda")
    s = codec.encode(x, fixed_cb, 4096)
    r = codec.stream_copy(s)
    assert int(r.off[0].item()) == 0
    assert codec.decode(r, fixed_cb).numel() == 0


def test_loopback_destination_too_small(fixed_cb):
    x = workloads.fixed_codebook_shard(3, warmup=False, device="cuda").reshape(-1)[:100_000].view(torch.uint8)
    s = codec.encode(x, fixed_cb, 4096)
    small = torch.full(((s.total_bits() + 31) // 32 * 4 - 1,), 0x5A, dtype=torch.uint8, device="cuda")
    off = torch.full_like(s.off, -7)
    st = codec.new_status()
    _lib.huff_stream_copy(s.payload, s.off, small, off, st)
    assert int(st.item()) == _lib.HUFF_ERR_BUFFER_TOO_SMALL
    assert bool((small == 0x5A).all()) and bool((off == -7).all())


def test_loopback_size_past_source_is_corrupt(fixed_cb):
    x = workloads.fixed_codebook_shard(4, warmup=False, device="cuda").reshape(-1)[:50_000].view(torch.uint8)
    s = codec.encode(x, fixed_cb, 4096)
    bad_off = s.off.clone()
    bad_off[-1] = s.payload.numel() * 8 + 1
    dst = torch.zeros_like(s.payload)
    st = codec.new_status()
    _lib.huff_stream_copy(s.payload, bad_off, dst, torch.empty_like(bad_off), st)
    assert int(st.item()) == _lib.HUFF_ERR_CORRUPT_STREAM
    assert bool((dst == 0).all())


def test_loopback_arguments(fixed_cb):
    x = torch.zeros(1000, dtype=torch.uint8, device="cuda")
    s = codec.encode(x, fixed_cb, 256)
    st = codec.new_status()
    with pytest.raises(_lib.HuffError) as e:  # copying onto itself
        _lib.huff_stream_copy(s.payload, s.off, s.payload, torch.empty_like(s.off), st)
    assert e.value.status == _lib.HUFF_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        _lib.huff_stream_copy(s.payload, s.off, torch.empty_like(s.payload), s.off[:-1].clone(), st)


def test_loopback_in_a_cuda_graph(fixed_cb):
    # encode -> copy -> decode captured once and replayed on new data in the same buffers
    n, chunk = 1 << 20, 16384
    x = torch.empty(n, dtype=torch.uint8, device="cuda")
    x.copy_(workloads.fixed_codebook_shard(9, warmup=False, device="cuda").reshape(-1)[:n].view(torch.uint8))
    cap = _lib.huff_encode_bound(n, 24)
    nc = _lib.huff_num_chunks(n, chunk)
    pay = torch.empty(cap, dtype=torch.uint8, device="cuda")
    off = torch.empty(nc + 1, dtype=torch.int64, device="cuda")
    ws = torch.empty(max(_lib.huff_workspace_size(n, chunk), 16) // 8, dtype=torch.int64, device="cuda")
    pay2 = torch.empty_like(pay)
    off2 = torch.empty_like(off)
    out = torch.empty_like(x)
    st = codec.new_status()

    def loop():
        _lib.huff_encode(x, fixed_cb.buf, chunk, pay, off, ws, st)
        _lib.huff_stream_copy(pay, off, pay2, off2, st)
        _lib.huff_decode(pay2, off2, n, chunk, fixed_cb.buf, out, st)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        loop()  # warm-up outside the capture (first-call attributes)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        loop()
    for k in (10, 11):
        x.copy_(workloads.fixed_codebook_shard(k, warmup=False, device="cuda").reshape(-1)[:n].view(torch.uint8))
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert torch.equal(out, x)
