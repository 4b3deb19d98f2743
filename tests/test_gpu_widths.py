"""Byte planes of other element widths (fp32: 4, fp16/bf16: 2, fp8: 1,
fp64: 8) on the GPU against the oracle, element by element, and their
per-plane Huffman streams against the oracle's encoding of each plane."""
import numpy as np
import pytest
import torch

import oracle
from lossless_huffman_compression_gb300 import _lib, codec
from gpu_util import assert_stream_equal, host, oracle_codebook

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    _lib.load()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("width", [1, 2, 4, 8])
@pytest.mark.parametrize("n", [1, 15, 16, 17, 4096, 100_003])
@pytest.mark.parametrize("offset", [0, 1])
def test_split_merge_w_match_oracle(width, n, offset):
    rng = np.random.default_rng(width * 1000 + n + offset)
    words = rng.integers(0, 256, (n + offset) * width, dtype=np.uint8)
    dev = torch.from_numpy(words).cuda()
    src = dev[offset * width:]  # offset 1: not 16-byte aligned, the scalar path
    ps = (n + 15) // 16 * 16 + 16 * offset
    planes = torch.full((width * ps,), 0xAB, dtype=torch.uint8, device="cuda")
    _lib.lmc_bytegroup_split_w(src, width, planes, ps)
    want = oracle.bytegroup_split_w(words[offset * width:], width)
    got = host(planes)
    for p in range(width):
        np.testing.assert_array_equal(got[p * ps: p * ps + n], want[p])
    back = torch.empty(n * width, dtype=torch.uint8, device="cuda")
    _lib.lmc_bytegroup_merge_w(planes, width, ps, back)
    np.testing.assert_array_equal(host(back), oracle.bytegroup_merge_w(want))


def test_width2_planes_equal_the_bf16_split():
    rng = np.random.default_rng(3)
    w = torch.from_numpy(rng.integers(-32768, 32767, 50_000, dtype=np.int16)).cuda()
    hi = torch.empty(50_000, dtype=torch.uint8, device="cuda")
    lo = torch.empty(50_000, dtype=torch.uint8, device="cuda")
    _lib.lmc_bytegroup_split(w, hi, lo)
    planes = torch.empty(2 * 50_000, dtype=torch.uint8, device="cuda")
    _lib.lmc_bytegroup_split_w(w, 2, planes, 50_000)
    assert torch.equal(planes[:50_000], hi) and torch.equal(planes[50_000:], lo)


def _tensor(kind: str, shape, rng):
    x = torch.from_numpy(rng.normal(0, 0.02, shape).astype(np.float32))
    if kind == "fp32":
        return x
    if kind == "fp16":
        return x.to(torch.float16)
    if kind == "bf16":
        return x.to(torch.bfloat16)
    if kind == "fp64":
        return x.to(torch.float64)
    if kind == "fp8":
        return (x * 50).to(torch.float8_e4m3fn)
    if kind == "int8":
        return torch.from_numpy(np.clip(np.round(rng.normal(0, 8, shape)), -128, 127).astype(np.int8))
    raise ValueError(kind)


@pytest.mark.parametrize("kind", ["fp32", "fp16", "bf16", "fp64", "fp8", "int8"])
@pytest.mark.parametrize("delta", [False, True])
def test_compress_planes_streams_match_oracle(kind, delta):
    rng = np.random.default_rng(["fp32", "fp16", "bf16", "fp64", "fp8", "int8"].index(kind) * 2 + delta)
    shape = (300, 333)  # an even byte count for every width (the delta works on 16-bit words)
    x = _tensor(kind, shape, rng)
    x0 = _tensor(kind, shape, np.random.default_rng(99)) if delta else None
    width = x.element_size()
    b = x.reshape(-1).view(torch.uint8).numpy()
    if delta:
        b = b ^ x0.reshape(-1).view(torch.uint8).numpy()
    ref_planes = oracle.bytegroup_split_w(b, width)
    s = codec.compress_planes(x.cuda(), x0.cuda() if delta else None, chunk_bytes=4096)
    assert s.width == width and len(s.planes) == width
    for plane, (cb, st) in zip(ref_planes, s.planes):
        ln, cd = oracle_codebook(oracle.histogram(plane))
        np.testing.assert_array_equal(cb.lengths(), ln)
        pay, off = oracle.encode(plane, ln, cd, 4096)
        assert_stream_equal(st, pay, off)
    back = codec.decompress_planes(s, x0.cuda() if delta else None)
    assert back.dtype == x.dtype and tuple(back.shape) == shape
    assert torch.equal(back.cpu().reshape(-1).view(torch.uint8), x.reshape(-1).view(torch.uint8))


def test_bad_width_is_rejected():
    x = torch.zeros(63, dtype=torch.uint8, device="cuda")
    planes = torch.zeros(64 * 3, dtype=torch.uint8, device="cuda")
    with pytest.raises(_lib.HuffError) as e:
        _lib.lmc_bytegroup_split_w(x, 3, planes, 64)
    assert e.value.status == _lib.HUFF_ERR_INVALID_ARG
