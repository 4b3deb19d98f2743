"""huff_encode_noalloc: the encode entry point for callers that cannot allocate.

Some callers cannot give huff_encode a workspace: their device memory belongs
to a framework's pool, or they run in a loop that must not call cudaMalloc or
cudaFree (both can stall the whole device).  huff_encode_noalloc runs the same
encode with a fixed scratch array inside the library.  Its output must be
byte-for-byte the output of huff_encode with a caller-provided workspace, and
stay so on consecutive calls that reuse the shared scratch.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

from lossless_huffman_compression_gb300 import _lib, codec

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    _lib.load()
    assert torch.cuda.is_available()


def _encode_noalloc(x: torch.Tensor, cb: codec.Codebook, chunk: int):
    n = x.numel()
    payload = torch.zeros(_lib.huff_encode_bound(n, 24), dtype=torch.uint8, device="cuda")
    off = torch.zeros(_lib.huff_num_chunks(n, chunk) + 1, dtype=torch.int64, device="cuda")
    st = codec.new_status()
    _lib.huff_encode_noalloc(x, cb.buf, chunk, payload, off, st)
    codec.raise_on_status(st, "huff_encode_noalloc")
    return payload, off


def test_noalloc_encode_equals_workspace_encode_on_two_calls_in_a_row():
    rng = np.random.default_rng(77)
    cases = [(300_001, 8.0, 4096), ((1 << 20) + 123, 30.0, 16384)]  # several tiles, ragged tails
    for n, sigma, chunk in cases:
        x = torch.from_numpy(np.clip(np.round(rng.normal(0, sigma, n)), -128, 127).astype(np.int8)
                             .view(np.uint8)).cuda()
        cb = codec.build_codebook(codec.histogram(x))
        ref = codec.encode(x, cb, chunk)  # huff_encode with its own workspace
        payload, off = _encode_noalloc(x, cb, chunk)
        assert torch.equal(off, ref.off)
        T = int(ref.off[-1].item())
        used = ((T + 31) // 32) * 4
        assert torch.equal(payload[:used], ref.payload[:used])
        assert torch.equal(codec.decode(codec.Stream(payload, off, n, chunk), cb), x)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    cb = codec.build_codebook(codec.histogram(torch.arange(256, dtype=torch.uint8, device="cuda")))
    x = torch.zeros(16, dtype=torch.uint8, device="cuda")
    payload = torch.zeros(64, dtype=torch.uint8, device="cuda")
    off = torch.zeros(2, dtype=torch.int64, device="cuda")
    with pytest.raises(_lib.HuffError) as e:
        _lib.huff_encode_noalloc(x, cb.buf, 1 << 20, payload, off, codec.new_status(),
                                 n=_lib.HUFF_NOALLOC_MAX_SYMBOLS + 1)
    assert e.value.status == _lib.HUFF_ERR_BUFFER_TOO_SMALL


def test_noalloc_at_its_largest_size_equals_workspace_encode():
    """n at HUFF_NOALLOC_MAX_SYMBOLS (and just below it, ragged), where the byte-stream encode uses the
    most segments of 16 tiles and so the most of the scratch: the same stream as huff_encode."""
    g = torch.Generator(device="cuda")
    g.manual_seed(123)
    top = _lib.HUFF_NOALLOC_MAX_SYMBOLS
    for n, chunk in ((top, 1 << 20), (top - 4097, 16384)):
        x = torch.randn(n, device="cuda", generator=g).mul_(12).round_().clamp_(-128, 127).to(torch.int8)
        x = x.view(torch.uint8)
        cb = codec.build_codebook(codec.histogram(x))
        ref = codec.encode(x, cb, chunk)
        payload, off = _encode_noalloc(x, cb, chunk)
        assert torch.equal(off, ref.off)
        T = int(ref.off[-1].item())
        used = ((T + 31) // 32) * 4
        assert torch.equal(payload[:used], ref.payload[:used])
        del x, ref, payload, off
        torch.cuda.empty_cache()
