"""The multi-threaded driver of the oracle's steps equals the sequential oracle.

Its payload and offsets must be byte-identical to oracle.encode's for any
thread count (the pack writes bytes shared by two chunks with an atomic OR),
its decode must invert them and reject a moved offset, and its histogram,
delta and plane helpers must equal the sequential ones."""
import numpy as np
import pytest

import oracle
from oracle import mt


@pytest.mark.parametrize("n,chunk", [(0, 256), (1, 256), (255, 256), (257, 256), (100_003, 256),
                                     (300_001, 4096), (65_536, 65_536)])
@pytest.mark.parametrize("threads", [1, 2, 7, 64])
def test_mt_encode_decode_equal_sequential(n, chunk, threads):
    rng = np.random.default_rng(n + threads)
    x = np.clip(np.round(rng.normal(0, 5 + (n % 7), n)), -128, 127).astype(np.int8).view(np.uint8)
    h = oracle.histogram(x) if n else np.ones(256, dtype=np.uint64)
    ln = oracle.code_lengths(h)
    cd = oracle.canonical_codes(ln)
    p1, o1 = oracle.encode(x, ln, cd, chunk)
    p2, o2 = mt.encode(x, ln, cd, chunk, threads)
    np.testing.assert_array_equal(o2, o1)
    np.testing.assert_array_equal(p2, p1)
    np.testing.assert_array_equal(mt.decode(p2, o2, n, chunk, ln, threads), x)
    np.testing.assert_array_equal(mt.histogram(x, threads), oracle.histogram(x))


def test_mt_decode_rejects_a_moved_offset_and_encode_a_missing_code():
    rng = np.random.default_rng(3)
    x = rng.integers(0, 40, 50_000, dtype=np.uint8)
    ln = oracle.code_lengths(oracle.histogram(x))
    pay, off = mt.encode(x, ln, oracle.canonical_codes(ln), 1024, 4)
    bad = off.copy()
    bad[7] += 1
    with pytest.raises(oracle.OracleError):
        mt.decode(pay, bad, x.size, 1024, ln, 4)
    y = x.copy()
    y[123] = 200  # no code for 200
    with pytest.raises(oracle.OracleError):
        mt.encode(y, ln, oracle.canonical_codes(ln), 1024, 4)


@pytest.mark.parametrize("threads", [1, 5])
def test_mt_planes_and_delta_equal_sequential(threads):
    rng = np.random.default_rng(threads)
    a = rng.integers(0, 1 << 16, 12_345, dtype=np.uint16)
    b = rng.integers(0, 1 << 16, 12_345, dtype=np.uint16)
    hi, lo = mt.delta_split(a, b, threads)
    rh, rl = oracle.bytegroup_split(oracle.delta_xor(a, b))
    np.testing.assert_array_equal(hi, rh)
    np.testing.assert_array_equal(lo, rl)
    np.testing.assert_array_equal(mt.merge_xor(hi, lo, b, threads), a)
    hi2, lo2 = mt.delta_split(a, None, threads)
    np.testing.assert_array_equal(mt.merge_xor(hi2, lo2, None, threads), a)


def test_mt_snapshot_round_trip():
    rng = np.random.default_rng(11)
    x0 = rng.normal(0, 0.02, 200_000).astype(np.float32)
    x1 = (x0 + rng.normal(0, 1e-4, x0.size)).astype(np.float32)
    # bf16 bit patterns by truncation (any 16-bit patterns do for the round trip)
    b0 = (x0.view(np.uint32) >> 16).astype(np.uint16)
    b1 = (x1.view(np.uint32) >> 16).astype(np.uint16)
    size, tc, td = mt.snapshot_round_trip(b0, b1, 16384, 4)
    assert 0 < size < 2 * b1.size and tc >= 0 and td >= 0
