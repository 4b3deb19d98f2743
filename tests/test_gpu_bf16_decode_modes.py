"""The fused bf16 decode's kernel cases, each reached on purpose, bit-exact.

With more than 448 chunk pairs per SM the decode runs one lane per chunk pair
with the two planes decoded one after the other.  Three kernels cover that:
the high plane decoded by table lookups (no 1-bit code), the high plane
decoded as runs of its 1-bit code, and the same with x0 staged in shared
memory (when x0 is given and the block's staging area fits, which it does up
to the widest block, 896 lanes, next to the split low-plane table).  These tests
size inputs (256-element chunks) to land in each, with ragged last chunks, a
run symbol other than 0, long high-plane codes, and streams written by the
oracle rather than by the GPU encoder.
"""
import numpy as np
import pytest
import torch

import oracle
from lossless_huffman_compression_gb300 import _lib, codec
from gpu_util import host

pytestmark = pytest.mark.gpu

CHUNK = 256


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    _lib.load()
    assert torch.cuda.is_available()


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _n_for_lanes(lanes_per_sm: int, tail: int) -> int:
    """Elements giving about `lanes_per_sm` chunk pairs per SM, plus a ragged tail."""
    return (_sms() * lanes_per_sm - 1) * CHUNK + tail


def _snapshot_like(n, seed, noise=1e-4):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    x0 = (torch.randn(n, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    x1 = (x0.float() + torch.randn(n, device="cuda", generator=g) * noise).to(torch.bfloat16)
    return x0, x1


def _round_trip(x1, x0):
    s = codec.compress_bf16(x1, x0, CHUNK)
    back = codec.decompress_bf16(s, x0)
    assert torch.equal(back.view(torch.int16), x1.reshape(-1).view(torch.int16))
    return s


@pytest.mark.parametrize("lanes", [480, 832, 900])
@pytest.mark.parametrize("delta", [True, False])
def test_run_decoded_high_plane(lanes, delta):
    """Snapshot delta (high plane with a 1-bit code for 0): the run kernels (staged x0 with a delta)."""
    n = _n_for_lanes(lanes, 77)
    x0, x1 = _snapshot_like(n, lanes)
    if delta:
        s = _round_trip(x1, x0)
    else:  # the delta materialised, decoded without x0
        d = (x1.view(torch.int16) ^ x0.view(torch.int16)).view(torch.bfloat16)
        s = _round_trip(d, None)
    assert s.cb_hi.lengths().astype(int).tolist().count(1) == 1  # the high plane has a 1-bit code


@pytest.mark.parametrize("lanes", [480, 832])
def test_table_decoded_high_plane(lanes):
    """bf16 weights: the high plane has no 1-bit code, so the table kernel decodes it."""
    n = _n_for_lanes(lanes, 13)
    g = torch.Generator(device="cuda")
    g.manual_seed(9)
    w = (torch.randn(n, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    s = _round_trip(w, None)
    assert 1 not in s.cb_hi.lengths().astype(int).tolist()
    x0 = (torch.randn(n, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    _round_trip(w, x0)  # a delta of unrelated tensors: no 1-bit code either


@pytest.mark.parametrize("run_high", [True, False])
def test_low_plane_windows_past_the_split_entry(run_high):
    """A delta whose low plane has 2-bit codes (four symbols of about a quarter each, a thin tail, no
    1-bit code): its 13-bit windows hold up to 6 symbols, more than the 4 a split table entry keeps,
    so the rest go to the step's next lookup.  With a run-decoded high plane (staged x0) and with a
    table-decoded one."""
    n = _n_for_lanes(832, 123)
    g = torch.Generator(device="cuda")
    g.manual_seed(31 + run_high)
    main = torch.randint(0, 4, (n,), device="cuda", generator=g, dtype=torch.int32) * 17
    tail = torch.randint(0, 256, (n,), device="cuda", generator=g, dtype=torch.int32)
    lo = torch.where(torch.rand(n, device="cuda", generator=g) < 0.03, tail, main)
    if run_high:  # 0 for about 98 % of elements: a 1-bit code
        hi = torch.where(torch.rand(n, device="cuda", generator=g) < 0.02,
                         torch.randint(0, 256, (n,), device="cuda", generator=g, dtype=torch.int32), 0)
    else:  # spread over 40 values: no 1-bit code
        hi = torch.randint(0, 40, (n,), device="cuda", generator=g, dtype=torch.int32)
    d = ((hi << 8) | lo).to(torch.int16)
    x0 = torch.randint(-32768, 32767, (n,), device="cuda", generator=g, dtype=torch.int32).to(torch.int16)
    x1 = (d ^ x0).view(torch.bfloat16)
    s = _round_trip(x1, x0.view(torch.bfloat16))
    ln_lo = s.cb_lo.lengths().astype(int).tolist()
    assert 1 not in ln_lo and ln_lo.count(2) >= 3  # the three-lookup steps, with 2-bit codes
    assert (1 in s.cb_hi.lengths().astype(int).tolist()) == run_high


def test_run_symbol_other_than_zero():
    """A high plane whose 1-bit code is 0x3f (the ring is pre-filled with that byte, not 0)."""
    n = _n_for_lanes(832, 201)
    g = torch.Generator(device="cuda")
    g.manual_seed(21)
    lo = torch.randint(0, 256, (n,), device="cuda", generator=g, dtype=torch.int32)
    hi = torch.full((n,), 0x3F, device="cuda", dtype=torch.int32)
    rare = torch.rand(n, device="cuda", generator=g) < 0.02
    hi = torch.where(rare, torch.randint(0, 256, (n,), device="cuda", generator=g, dtype=torch.int32), hi)
    w = ((hi << 8) | lo).to(torch.int16).view(torch.bfloat16)
    s = _round_trip(w, None)
    ln = s.cb_hi.lengths()
    assert int(ln[0x3F]) == 1
    x0 = torch.zeros_like(w)
    _round_trip(w, x0)  # with x0 (all zero): the staged kernel, same planes


def test_decodes_oracle_written_streams():
    """Streams written by the oracle (per plane, from its own histograms) decode to the input, staged x0."""
    n = _n_for_lanes(832, 99)
    x0, x1 = _snapshot_like(n, 5)
    a = host(x1.view(torch.int16)).view(np.uint16)
    b = host(x0.view(torch.int16)).view(np.uint16)
    hi, lo = oracle.bytegroup_split(oracle.delta_xor(a, b))
    streams, cbs = [], []
    for plane in (hi, lo):
        ln = oracle.code_lengths(oracle.histogram(plane))
        pay, off = oracle.encode(plane, ln, oracle.canonical_codes(ln), CHUNK)
        cap = ((int(off[-1]) + 31) // 32) * 4 + 16
        p = torch.zeros(cap, dtype=torch.uint8, device="cuda")
        p[: pay.size] = torch.from_numpy(pay).cuda()
        streams.append(codec.Stream(p, torch.from_numpy(off.astype(np.int64)).cuda(), n, CHUNK))
        cbs.append(codec.codebook_from_lengths(ln))
    assert int(streams[0].off.numel()) == (n + CHUNK - 1) // CHUNK + 1
    back = codec.decompress_bf16(codec.Bf16Streams(cbs[0], cbs[1], streams[0], streams[1], n), x0)
    assert torch.equal(back.view(torch.int16), x1.view(torch.int16))


def test_corrupt_stream_is_reported_by_the_run_kernels():
    n = _n_for_lanes(832, 0)
    x0, x1 = _snapshot_like(n, 6)
    s = codec.compress_bf16(x1, x0, CHUNK)
    s.hi.off[1000] += 3  # chunk 999 of the high plane now ends 3 bits late, chunk 1000 starts there
    st = codec.new_status()
    out = torch.empty(n, dtype=torch.int16, device="cuda")
    _lib.lmc_decode_bf16(s.hi.payload, s.hi.off, s.lo.payload, s.lo.off, n, CHUNK, s.cb_hi.buf, s.cb_lo.buf,
                         x0.view(torch.int16), out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == _lib.HUFF_ERR_CORRUPT_STREAM


@pytest.mark.parametrize("delta", [True, False])
@pytest.mark.parametrize("n", [0, 1, 1 << 20, 1 << 26, 536_870_912, 2_000_027_648, 1 << 36])
def test_pick_chunk_gives_one_wave_of_full_blocks(n, delta):
    """huff_pick_chunk: the smallest multiple of 32, at least 256, that gives at most L chunks per SM, L
    the widest decode block (896 lanes with or without a delta on a GPU with 227 KiB of shared memory per
    block: the x0 staging fits next to the split low-plane table)."""
    c = _lib.huff_pick_chunk(n, delta)
    sms = _sms()
    assert c % 32 == 0 and 256 <= c <= (1 << 30)
    if torch.cuda.get_device_properties(0).shared_memory_per_block_optin != 232448:
        pytest.skip("the lane count per SM is checked on a GPU with 227 KiB of shared memory per block")
    lanes = 896
    assert -(-n // c) <= sms * lanes
    assert c == 256 or -(-n // (c - 32)) > sms * lanes  # the smallest such size
    if sms == 152 and (n, delta) in ((2_000_027_648, True), (536_870_912, False)):
        # the snapshot delta: 136 168 chunk pairs; the 1 GiB bf16 weights: 135 301; both in 896-lane blocks on
        # all 152 SMs
        assert c == (14688 if delta else 3968)
        nc = -(-n // c)
        block = -(-(-(-nc // sms)) // 32) * 32
        assert (block, -(-nc // block)) == (896, 152)
