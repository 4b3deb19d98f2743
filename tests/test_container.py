"""The serialised stream (container): its byte layout as include/huff.h states it,
round trips of oracle streams through the C ABI, and rejection of damaged
containers.  Host code only: runs without a GPU."""
import struct

import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from lossless_huffman_compression_gb300 import _lib
    _lib.load()
    return _lib


def _stream(n, chunk, seed=0):
    rng = np.random.default_rng(seed)
    x = np.clip(np.round(rng.normal(0, 8, n)), -128, 127).astype(np.int8).view(np.uint8)
    ln = oracle.code_lengths(oracle.histogram(x))
    pay, off = oracle.encode(x, ln, oracle.canonical_codes(ln), chunk)
    return x, ln, pay, off


def test_layout_is_the_documented_one(lib):
    n, chunk = 10_000, 4096
    x, ln, pay, off = _stream(n, chunk)
    T = int(off[-1])
    b = lib.huff_container_write(n, chunk, 24, ln, off, pay)
    magic, version, flags, max_len, zero, n_, chunk_, nc, T_ = struct.unpack_from("<IHHIIQQQQ", b, 0)
    assert b[:4] == b"HUFC" and magic == lib.HUFF_CONTAINER_MAGIC
    assert (version, flags, max_len, zero, n_, chunk_, nc, T_) == (1, 1, 24, 0, n, chunk, 3, T)
    assert bytes(b[48:48 + 256]) == ln.astype(np.uint8).tobytes()
    offs = struct.unpack_from("<4Q", b, 48 + 256)
    assert list(offs) == [int(o) for o in off]
    body = b[48 + 256 + 32:]
    assert len(body) == (T + 7) // 8 and body == pay[: (T + 7) // 8].tobytes()
    assert len(b) == lib.huff_container_size(n, chunk, T, True)


@pytest.mark.parametrize("n,chunk,with_lengths", [(0, 256, True), (1, 256, False), (77_777, 1024, True),
                                                  (77_777, 1 << 20, False)])
def test_round_trip(lib, n, chunk, with_lengths):
    x, ln, pay, off = _stream(n, chunk, seed=n)
    b = lib.huff_container_write(n, chunk, 24, ln if with_lengths else None, off, pay)
    f = lib.huff_container_parse(b)
    assert (f["n"], f["chunk_bytes"], f["n_chunks"], f["max_len"]) == (n, chunk, lib.huff_num_chunks(n, chunk), 24)
    np.testing.assert_array_equal(f["off"], off)
    T = int(off[-1])
    assert f["total_bits"] == T
    np.testing.assert_array_equal(f["payload"], pay[: (T + 7) // 8])
    if with_lengths:
        np.testing.assert_array_equal(f["lengths"], ln)
        assert len(b) == 48 + 256 + 8 * (f["n_chunks"] + 1) + (T + 7) // 8
    else:
        assert f["lengths"] is None
        assert len(b) == 48 + 8 * (f["n_chunks"] + 1) + (T + 7) // 8
    if n:
        # the decoded container is the oracle's stream: decoding it gives the input back
        got = oracle.decode(f["payload"], f["off"], n, chunk, ln)
        np.testing.assert_array_equal(got, x)


def test_damaged_containers_are_rejected(lib):
    n, chunk = 20_000, 4096
    _, ln, pay, off = _stream(n, chunk, seed=3)
    good = bytearray(lib.huff_container_write(n, chunk, 24, ln, off, pay))
    lib.huff_container_parse(bytes(good))

    def bad(mutate):
        b = bytearray(good)
        mutate(b)
        with pytest.raises(lib.HuffError) as e:
            lib.huff_container_parse(bytes(b))
        assert e.value.status == lib.HUFF_ERR_CORRUPT_STREAM

    bad(lambda b: b.__setitem__(0, ord("X")))                      # magic
    bad(lambda b: struct.pack_into("<H", b, 4, 2))                 # version
    bad(lambda b: struct.pack_into("<H", b, 6, 3))                 # unknown flag
    bad(lambda b: struct.pack_into("<I", b, 12, 1))                # reserved field
    bad(lambda b: struct.pack_into("<Q", b, 32, 4))                # chunk count
    bad(lambda b: struct.pack_into("<Q", b, 24, 1000))             # chunk size not a multiple of 32
    bad(lambda b: b.__setitem__(48 + 7, 25))                       # a length above max_len
    bad(lambda b: struct.pack_into("<Q", b, 48 + 256 + 8, 1 << 40))  # offsets not rising to T
    bad(lambda b: b.pop())                                         # truncated
    bad(lambda b: b.append(0))                                     # trailing byte
    with pytest.raises(lib.HuffError) as e:
        lib.huff_container_parse(bytes(good[:40]))
    assert e.value.status == lib.HUFF_ERR_CORRUPT_STREAM


def test_write_rejects_bad_streams(lib):
    n, chunk = 5000, 1024
    _, ln, pay, off = _stream(n, chunk, seed=5)
    for args, status in (
        ((n, chunk, 24, ln, off[::-1].copy(), pay), lib.HUFF_ERR_INVALID_ARG),     # offsets falling
        ((n, 1000, 24, ln, off, pay), lib.HUFF_ERR_INVALID_ARG),                    # chunk size
        ((n, chunk, 8, ln, off, pay), lib.HUFF_ERR_INVALID_ARG),                    # lengths above max_len
    ):
        if status == lib.HUFF_ERR_INVALID_ARG and args[2] == 8 and int(np.max(ln)) <= 8:
            continue
        with pytest.raises(lib.HuffError) as e:
            lib.huff_container_write(*args)
        assert e.value.status == status
