"""Pins for the CPU oracle, checked against facts that do not come from the oracle.

Each test ties one step of the oracle to something fixed outside it: a worked
example of a published specification (RFC 1951 3.2.2), hand derivations of the
stated rules (fixtures under tests/golden, each with its derivation), closed
forms (dyadic sources, T = sum count * len), textbook invariants (Kraft
equality, H <= mean length < H + 1, prefix-freeness), brute force over all
prefix codes of tiny alphabets, exhaustive checks over all 2^16 bf16 bit
patterns, and a library routine (numpy.bincount) for the histogram.
"""
import json
import math
from fractions import Fraction
import os

import numpy as np
import pytest

import oracle
from oracle import tiny

RNG = np.random.default_rng(12345)


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def _hist_from(d):
    h = np.zeros(256, dtype=np.uint64)
    for k, v in d.items():
        h[int(k)] = v
    return h


def _bits(code, length):
    return format(int(code), f"0{int(length)}b")


# --------------------------------------------------------------------- C1
def test_histogram_matches_bincount_and_sums_to_n():
    for n in [0, 1, 7, 1000, 65537]:
        x = RNG.integers(0, 256, n, dtype=np.uint8)
        h = oracle.histogram(x)
        np.testing.assert_array_equal(h, np.bincount(x, minlength=256).astype(np.uint64))
        assert int(h.sum()) == n


def test_histogram_strided_plane_view():
    w = RNG.integers(0, 1 << 16, 5001, dtype=np.uint16)
    b = w.view(np.uint8)
    # little-endian: byte 2i is the low byte, byte 2i + 1 the high byte
    lo = oracle.histogram(b, stride=2, n=w.size)
    hi = oracle.histogram(b[1:], stride=2, n=w.size)
    np.testing.assert_array_equal(lo, np.bincount(w & 0xFF, minlength=256).astype(np.uint64))
    np.testing.assert_array_equal(hi, np.bincount(w >> 8, minlength=256).astype(np.uint64))


def test_int8_reads_as_twos_complement_byte():
    x = np.array([-1, -128, 0, 127, -1], dtype=np.int8)
    h = oracle.histogram(x)
    assert h[0xFF] == 2 and h[0x80] == 1 and h[0] == 1 and h[0x7F] == 1


# --------------------------------------------------------------------- C6
def test_canonical_codes_rfc1951_example(golden_dir):
    g = _load(golden_dir, "rfc1951_canonical.json")
    ln = np.zeros(256, dtype=np.uint8)
    for k, v in g["lengths"].items():
        ln[int(k)] = v
    code = oracle.canonical_codes(ln)
    for k, want in g["codes"].items():
        assert _bits(code[int(k)], ln[int(k)]) == want
    tw = tiny.canonical_codes(list(ln))
    for k, want in g["codes"].items():
        assert tw[int(k)] == want


def test_canonical_codes_reject_oversubscribed_lengths():
    ln = np.zeros(256, dtype=np.uint8)
    ln[:3] = 1
    with pytest.raises(oracle.OracleError):
        oracle.canonical_codes(ln)


# --------------------------------------------------------------------- C3-C7 worked by hand
def test_hand_small_example(golden_dir):
    g = _load(golden_dir, "hand_small.json")
    x = np.array(g["input"], dtype=np.uint8)
    h = oracle.histogram(x)
    ln = oracle.code_lengths(h)
    cd = oracle.canonical_codes(ln)
    for k, v in g["lengths"].items():
        assert ln[int(k)] == v
    for k, v in g["codes"].items():
        assert _bits(cd[int(k)], ln[int(k)]) == v
    payload, off = oracle.encode(x, ln, cd, g["chunk_bytes"])
    assert payload.tobytes().hex() == g["payload_hex"]
    assert list(off) == g["offsets"]
    np.testing.assert_array_equal(oracle.decode(payload, off, x.size, g["chunk_bytes"], ln), x)


def test_hand_tie_break_and_reassignment(golden_dir):
    g = _load(golden_dir, "hand_ties.json")
    h = _hist_from(g["counts"])
    depths = tiny.huffman_depths([int(c) for c in h])
    assert {str(k): v for k, v in depths.items()} == g["tree_depths"]
    ln = oracle.code_lengths(h)
    for k, v in g["lengths"].items():
        assert ln[int(k)] == v
    cd = oracle.canonical_codes(ln)
    for k, v in g["codes"].items():
        assert _bits(cd[int(k)], ln[int(k)]) == v
    payload, off = oracle.encode(np.array(g["input"], dtype=np.uint8), ln, cd, 64)
    assert payload.tobytes().hex() == g["payload_hex"]
    assert int(off[-1]) == g["total_bits"]


def test_dyadic_closed_form(golden_dir):
    g = _load(golden_dir, "dyadic.json")
    h = _hist_from(g["counts"])
    ln = oracle.code_lengths(h)
    for k, v in g["lengths"].items():
        assert ln[int(k)] == v
    H = oracle.entropy(h)
    assert H == pytest.approx(g["entropy_bits"], abs=1e-12)
    mean_len = oracle.total_bits(h, ln) / float(h.sum())
    assert mean_len == pytest.approx(H, abs=1e-12)


@pytest.mark.parametrize("k", [2, 5, 9, 17])
def test_dyadic_general(k):
    # counts 2^(k-1), 2^(k-2), ..., 2, 1, 1  ->  lengths 1, 2, ..., k-1, k, k
    counts = [1 << (k - 1 - i) for i in range(k)] + [1]
    h = np.zeros(256, dtype=np.uint64)
    syms = RNG.choice(256, size=len(counts), replace=False)
    for s, c in zip(syms, counts):
        h[s] = c
    ln = oracle.code_lengths(h)
    want = list(range(1, k + 1)) + [k]
    assert [int(ln[s]) for s in syms] == want


# --------------------------------------------------------------------- C5 special cases
def test_special_cases_zero_one_two_symbols():
    h = np.zeros(256, dtype=np.uint64)
    assert int(oracle.code_lengths(h).max()) == 0
    h[77] = 1000
    ln = oracle.code_lengths(h)
    assert ln[77] == 1 and int(ln.sum()) == 1
    assert oracle.canonical_codes(ln)[77] == 0
    h[3] = 1
    ln = oracle.code_lengths(h)
    assert ln[77] == 1 and ln[3] == 1 and int(ln.sum()) == 2


def test_counts_must_sum_below_2_63():
    h = np.zeros(256, dtype=np.uint64)
    h[0] = 1 << 62
    h[1] = (1 << 62) - 1
    assert int(oracle.code_lengths(h).sum()) == 2
    h[1] = 1 << 62
    with pytest.raises(oracle.OracleError):
        oracle.code_lengths(h)
    with pytest.raises(ValueError):
        tiny.code_lengths([int(v) for v in h])


def test_one_symbol_stream_round_trip():
    x = np.full(1000, 42, dtype=np.uint8)
    ln, cd, payload, off = oracle.compress_plane(x, 256)
    assert int(off[-1]) == 1000 and payload.size == 125 and not payload.any()
    np.testing.assert_array_equal(oracle.decode(payload, off, x.size, 256, ln), x)


def test_cover_all_gives_every_symbol_a_code():
    h = np.zeros(256, dtype=np.uint64)
    h[0] = 10 ** 9
    h[1] = 5
    ln = oracle.code_lengths(h, 24, oracle.REF_COVER_ALL)
    assert int((ln > 0).sum()) == 256 and int(ln.max()) <= 24
    _kraft_equal(ln)


def test_symbol_missing_from_codebook_is_an_error():
    h = np.zeros(256, dtype=np.uint64)
    h[1] = 3
    h[2] = 4
    ln = oracle.code_lengths(h)
    cd = oracle.canonical_codes(ln)
    with pytest.raises(oracle.OracleError) as e:
        oracle.encode(np.array([1, 2, 3], dtype=np.uint8), ln, cd, 256)
    assert e.value.status == oracle.REF_ERR_SYMBOL_NOT_IN_CODEBOOK


# --------------------------------------------------------------------- invariants
def _kraft_equal(ln):
    L = [int(v) for v in ln if v > 0]
    top = max(L)
    assert sum(1 << (top - l) for l in L) == (1 << top), "Kraft sum must be exactly 1"


def _random_hist(m, skew):
    h = np.zeros(256, dtype=np.uint64)
    syms = RNG.choice(256, size=m, replace=False)
    if skew == "geom":
        vals = np.floor(1e6 * 0.6 ** np.arange(m)) + 1
    elif skew == "equalish":
        vals = RNG.integers(1000, 1003, m)
    else:
        vals = RNG.integers(1, 10 ** 6, m)
    h[syms] = vals.astype(np.uint64)
    return h


@pytest.mark.parametrize("m", [2, 3, 17, 100, 256])
@pytest.mark.parametrize("skew", ["uniform", "geom", "equalish"])
def test_kraft_equality_and_entropy_bounds(m, skew):
    h = _random_hist(m, skew)
    ln = oracle.code_lengths(h, 24)
    assert int((ln > 0).sum()) == m
    _kraft_equal(ln)
    H = oracle.entropy(h)
    mean_len = oracle.total_bits(h, ln) / float(h.sum())
    if int(ln.max()) < 24:  # no limit triggered: plain Huffman
        assert H - 1e-9 <= mean_len < H + 1


def test_prefix_free():
    for m in [2, 5, 40, 256]:
        h = _random_hist(m, "uniform")
        ln = oracle.code_lengths(h)
        cd = oracle.canonical_codes(ln)
        words = sorted(_bits(cd[s], ln[s]) for s in range(256) if ln[s])
        for a, b in zip(words, words[1:]):
            assert not b.startswith(a)


@pytest.mark.parametrize("m", [2, 3, 4, 5, 6, 7, 8])
def test_brute_force_optimal_unlimited(m):
    for trial in range(25):
        h = np.zeros(256, dtype=np.uint64)
        syms = RNG.choice(256, size=m, replace=False)
        h[syms] = RNG.integers(1, 60, m).astype(np.uint64)
        if trial % 5 == 0:
            h[syms] = np.array([1 << i for i in range(m)], dtype=np.uint64)
        ln = oracle.code_lengths(h, 24)
        cost = oracle.total_bits(h, ln)
        assert cost == tiny.brute_force_min_cost([int(c) for c in h])


@pytest.mark.parametrize("m,max_len", [(5, 3), (6, 3), (8, 3), (7, 4), (8, 4), (4, 2)])
def test_length_limited_is_valid_and_not_below_limited_optimum(m, max_len):
    for _ in range(25):
        h = np.zeros(256, dtype=np.uint64)
        syms = RNG.choice(256, size=m, replace=False)
        h[syms] = np.array([int(1.9 ** i) + int(RNG.integers(0, 3)) for i in range(m)], dtype=np.uint64)
        ln = oracle.code_lengths(h, max_len)
        assert int(ln.max()) <= max_len
        _kraft_equal(ln)
        cost = oracle.total_bits(h, ln)
        assert cost >= tiny.brute_force_min_cost([int(c) for c in h], max_len)


def test_fibonacci_counts_force_the_length_limit():
    fib = [1, 1]
    while len(fib) < 30:
        fib.append(fib[-1] + fib[-2])
    h = np.zeros(256, dtype=np.uint64)
    h[:30] = np.array(fib, dtype=np.uint64)
    unlimited = oracle.code_lengths(h, 63)
    assert int(unlimited.max()) == 29  # the Fibonacci tree is a path
    limited = oracle.code_lengths(h, 24)
    assert int(limited.max()) == 24
    _kraft_equal(limited)
    assert oracle.total_bits(h, limited) >= oracle.total_bits(h, unlimited)
    # the most frequent symbols keep the shortest codes
    order = np.argsort(-h[:30].astype(np.int64), kind="stable")
    assert all(limited[order[i]] <= limited[order[i + 1]] for i in range(29))


def _adjust_bits_cases(golden_dir):
    with open(os.path.join(golden_dir, "adjust_bits.json")) as f:
        return json.load(f)["cases"]


def _case_counts(case) -> np.ndarray:
    h = np.zeros(256, dtype=np.uint64)
    if "counts" in case:
        for k, v in case["counts"].items():
            h[int(k)] = v
    else:
        fib = [1, 1]
        while len(fib) < case["counts_fibonacci_symbols"]:
            fib.append(fib[-1] + fib[-2])
        h[: len(fib)] = fib
    return h


def test_adjust_bits_golden_moves_follow_the_procedure(golden_dir):
    """Each recorded move of the hand derivation is the one T.81 Annex K.3 prescribes (the fixture
    is checked against the rule itself, independently of either oracle)."""
    for case in _adjust_bits_cases(golden_dir):
        if "bits_window" in case:  # BITS(lo..hi) shown; BITS(1..lo-1) stay 1 throughout
            lo = case["bits_window"][0]
            bits = [0] + [1] * (lo - 1) + case["bits_before_window"]
            moves = [(i, j, [1] * (lo - 1) + b) for i, j, b in case["moves_window"]]
        else:
            bits = [0] + case["bits_before"]
            moves = case["moves"]
        L = case["max_len"]
        for i, j, after in moves:
            over = [k for k in range(L + 1, len(bits)) if bits[k] > 0]
            assert i == max(over), case["name"]
            jj = i - 2
            while bits[jj] == 0:
                jj -= 1
            assert j == jj, case["name"]
            bits[i] -= 2
            bits[i - 1] += 1
            bits[j + 1] += 2
            bits[j] -= 1
            assert bits[1:] == after, (case["name"], i, j)
            assert sum(Fraction(b, 2 ** k) for k, b in enumerate(bits) if k) == 1
        assert not any(bits[L + 1:]), case["name"]
        if "bits_after" in case:
            assert bits[1:] == case["bits_after"]


def test_adjust_bits_golden_lengths(golden_dir):
    """Both oracles end at the hand-derived lengths; their unlimited depths are the derivation's start."""
    for case in _adjust_bits_cases(golden_dir):
        h = _case_counts(case)
        L = case["max_len"]
        if "lengths" in case:
            want = np.zeros(256, dtype=np.uint8)
            for k, v in case["lengths"].items():
                want[int(k)] = v
            start = case["bits_before"]
        else:
            want = np.zeros(256, dtype=np.uint8)
            want[: len(case["lengths_by_symbol"])] = case["lengths_by_symbol"]
            lo = case["bits_window"][0]
            start = [1] * (lo - 1) + case["bits_before_window"]
        unlimited = oracle.code_lengths(h, 63)
        bl = np.bincount(unlimited[unlimited > 0], minlength=len(start) + 1)[1:]
        assert list(bl[: len(start)]) == start[: len(bl)] and not bl[len(start):].any(), case["name"]
        got = oracle.code_lengths(h, L)
        np.testing.assert_array_equal(got, want, err_msg=case["name"])
        assert tiny.code_lengths([int(v) for v in h], L) == [int(v) for v in want], case["name"]


@pytest.mark.parametrize("max_len", [8, 9, 10, 12])
def test_c_and_python_oracles_agree_when_the_limit_triggers(max_len):
    """Skewed histograms whose Huffman depths exceed max_len: the two restatements of the repair agree."""
    rng = np.random.default_rng(100 + max_len)
    hit = 0
    for trial in range(40):
        m = int(rng.integers(max_len + 2, 257))
        h = np.zeros(256, dtype=np.uint64)
        syms = rng.choice(256, size=m, replace=False)
        ratio = 1.3 + rng.random() * 0.9  # geometric counts give deep trees
        h[syms] = np.maximum(1, (ratio ** rng.uniform(0, 40, m)).astype(np.uint64))
        unlimited = oracle.code_lengths(h, 63)
        ln = oracle.code_lengths(h, max_len)
        if int(unlimited.max()) > max_len:
            hit += 1
        assert int(ln.max()) <= max_len
        _kraft_equal(ln)
        assert [int(v) for v in ln] == tiny.code_lengths([int(v) for v in h], max_len)
    assert hit >= 20  # the repair ran in most trials


# --------------------------------------------------------------------- C6 + C7 closed forms
def test_equal_counts_give_identity_payload():
    h = np.full(256, 7, dtype=np.uint64)
    ln = oracle.code_lengths(h)
    assert (ln == 8).all()
    cd = oracle.canonical_codes(ln)
    np.testing.assert_array_equal(cd, np.arange(256, dtype=np.uint32))
    x = RNG.integers(0, 256, 10_000, dtype=np.uint8)
    payload, off = oracle.encode(x, ln, cd, 1024)
    np.testing.assert_array_equal(payload, x)
    np.testing.assert_array_equal(off, np.arange(0, 10_000 + 1024, 1024).clip(max=10_000) * 8)


def test_total_bits_offsets_and_chunk_independence():
    x = oracle_input = (np.clip(np.round(RNG.normal(0, 8, 50_000)), -128, 127)).astype(np.int8).view(np.uint8)
    h = oracle.histogram(x)
    ln = oracle.code_lengths(h)
    cd = oracle.canonical_codes(ln)
    ref_payload = None
    for cb in [256, 1024, 4096, 65536]:
        payload, off = oracle.encode(oracle_input, ln, cd, cb)
        assert int(off[-1]) == oracle.total_bits(h, ln)
        per_chunk = [int(ln[x[c:c + cb]].astype(np.int64).sum()) for c in range(0, x.size, cb)]
        np.testing.assert_array_equal(np.diff(off.astype(np.int64)), per_chunk)
        if ref_payload is None:
            ref_payload = payload
        np.testing.assert_array_equal(payload, ref_payload)


# --------------------------------------------------------------------- C8 round trip and corruption
@pytest.mark.parametrize("n", [0, 1, 2, 255, 256, 257, 4095, 4097, 30_001])
@pytest.mark.parametrize("cb", [256, 4096])
def test_round_trip(n, cb):
    x = (np.clip(np.round(RNG.normal(0, 20, n)), -128, 127)).astype(np.int8).view(np.uint8)
    if n == 0:
        ln = oracle.code_lengths(np.ones(256, dtype=np.uint64))
        cd = oracle.canonical_codes(ln)
        payload, off = oracle.encode(x, ln, cd, cb)
        assert list(off) == [0]
        return
    ln, cd, payload, off = oracle.compress_plane(x, cb)
    assert payload.size == (int(off[-1]) + 7) // 8
    np.testing.assert_array_equal(oracle.decode(payload, off, n, cb, ln), x)


def test_decode_detects_moved_offset():
    x = RNG.integers(0, 50, 5000, dtype=np.uint8)
    ln, cd, payload, off = oracle.compress_plane(x, 256)
    bad = off.copy()
    bad[3] += 1
    with pytest.raises(oracle.OracleError) as e:
        oracle.decode(payload, bad, x.size, 256, ln)
    assert e.value.status == oracle.REF_ERR_CORRUPT_STREAM


def test_decode_detects_truncated_payload():
    x = RNG.integers(0, 50, 5000, dtype=np.uint8)
    ln, cd, payload, off = oracle.compress_plane(x, 256)
    with pytest.raises(oracle.OracleError):
        oracle.decode(payload[:-10], off, x.size, 256, ln)


# --------------------------------------------------------------------- C9 exhaustive
def test_split_merge_xor_exhaustive_over_all_patterns():
    w = np.arange(1 << 16, dtype=np.uint16)
    hi, lo = oracle.bytegroup_split(w)
    np.testing.assert_array_equal(hi, (np.arange(1 << 16) // 256).astype(np.uint8))
    np.testing.assert_array_equal(lo, (np.arange(1 << 16) % 256).astype(np.uint8))
    np.testing.assert_array_equal(oracle.bytegroup_merge(hi, lo), w)
    b = RNG.permutation(w)
    d = oracle.delta_xor(w, b)
    np.testing.assert_array_equal(oracle.delta_xor(d, b), w)
    np.testing.assert_array_equal(oracle.delta_xor(w, w), np.zeros_like(w))


def test_bf16_specials_round_trip_through_planes():
    import torch
    specials = torch.tensor([0.0, -0.0, float("inf"), float("-inf"), float("nan"), 1e-40, -3.5],
                            dtype=torch.bfloat16)
    w = specials.view(torch.int16).numpy().view(np.uint16)
    hi, lo = oracle.bytegroup_split(w)
    back = oracle.bytegroup_merge(hi, lo)
    np.testing.assert_array_equal(back, w)
    assert hi[1] == 0x80 and lo[1] == 0  # -0.0 keeps its sign bit in the high plane


# --------------------------------------------------------------------- C10
def test_entropy_of_discretised_gaussian():
    # H of round(N(0, 8)) is close to the differential entropy 0.5*log2(2*pi*e*64)
    x = np.clip(np.round(np.random.default_rng(0).normal(0, 8, 1 << 20)), -128, 127).astype(np.int8)
    H = oracle.entropy(oracle.histogram(x))
    assert H == pytest.approx(0.5 * math.log2(2 * math.pi * math.e * 64), abs=0.01)


def test_entropy_uniform_and_point_mass():
    assert oracle.entropy(np.full(256, 3, dtype=np.uint64)) == pytest.approx(8.0, abs=1e-12)
    h = np.zeros(256, dtype=np.uint64)
    h[9] = 5
    assert oracle.entropy(h) == 0.0


# --------------------------------------------------------------------- the two oracles agree
@pytest.mark.parametrize("seed", range(6))
def test_c_oracle_matches_python_tiny_oracle(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 20_000))
    kind = seed % 3
    if kind == 0:
        x = np.clip(np.round(rng.normal(0, 3 + 10 * seed, n)), -128, 127).astype(np.int8).view(np.uint8)
    elif kind == 1:
        x = rng.integers(0, 256, n, dtype=np.uint8)
    else:
        x = rng.choice(np.array([0, 1, 2, 250], dtype=np.uint8), n, p=[0.9, 0.05, 0.04, 0.01])
    cb = int(rng.choice([256, 512, 4096]))
    flags = oracle.REF_COVER_ALL if seed % 2 else 0
    h = oracle.histogram(x)
    assert [int(v) for v in h] == tiny.histogram(x.tobytes())
    ln = oracle.code_lengths(h, 24, flags)
    tl = tiny.code_lengths([int(v) for v in h], 24, flags)
    assert [int(v) for v in ln] == tl
    cd = oracle.canonical_codes(ln)
    tw = tiny.canonical_codes(tl)
    assert all((_bits(cd[s], ln[s]) if ln[s] else "") == tw[s] for s in range(256))
    payload, off = oracle.encode(x, ln, cd, cb)
    tp, toff = tiny.encode(x.tobytes(), tl, cb)
    assert payload.tobytes() == tp and [int(v) for v in off] == toff
    assert tiny.decode(tp, toff, n, cb, tl) == x.tobytes()
    assert oracle.entropy(h) == pytest.approx(tiny.entropy([int(v) for v in h]), rel=1e-12)


# ------------------------------------------------------------------ byte planes of other widths (P2 byte grouping)
def test_bytegroup_split_w_ieee_encodings():
    # IEEE 754 encodings of exact values, most significant byte first
    cases = [
        (np.array([1.0], dtype=np.float32), [0x3F, 0x80, 0x00, 0x00]),
        (np.array([-2.0], dtype=np.float32), [0xC0, 0x00, 0x00, 0x00]),
        (np.array([0.1], dtype=np.float32), [0x3D, 0xCC, 0xCC, 0xCD]),
        (np.array([np.inf], dtype=np.float32), [0x7F, 0x80, 0x00, 0x00]),
        (np.array([1.0], dtype=np.float64), [0x3F, 0xF0, 0, 0, 0, 0, 0, 0]),
        (np.array([-0.5], dtype=np.float16), [0xB8, 0x00]),
    ]
    for x, want in cases:
        planes = oracle.bytegroup_split_w(x, x.itemsize)
        assert [int(p[0]) for p in planes] == want


def test_bytegroup_split_w_width2_equals_c_split_on_all_patterns():
    w = np.arange(1 << 16, dtype=np.uint16)
    hi, lo = oracle.bytegroup_split(w)
    p0, p1 = oracle.bytegroup_split_w(w, 2)
    assert np.array_equal(p0, hi) and np.array_equal(p1, lo)


@pytest.mark.parametrize("width", [1, 2, 4, 8])
def test_bytegroup_merge_w_inverts_split(width):
    rng = np.random.default_rng(width)
    b = rng.integers(0, 256, 1000 * width, dtype=np.uint8)
    planes = oracle.bytegroup_split_w(b, width)
    assert len(planes) == width and all(p.size == 1000 for p in planes)
    assert np.array_equal(oracle.bytegroup_merge_w(planes), b)


def test_fp32_plane0_holds_the_sign_bit():
    rng = np.random.default_rng(5)
    x = rng.normal(0, 1, 10000).astype(np.float32)
    p0 = oracle.bytegroup_split_w(x, 4)[0]
    assert np.array_equal(p0 >> 7, np.signbit(x).astype(np.uint8))


# ------------------------------------------------------------------ drift of a shard against a fixed codebook
def test_drift_gap_closed_forms():
    L = np.zeros(256, dtype=np.uint8)
    # uniform over 256 symbols with 8-bit codes: T = 8 n = n H
    assert oracle.drift_gap(np.full(256, 10), np.full(256, 8)) == 0.0
    # dyadic (1/2, 1/4, 1/8, 1/8) with lengths (1, 2, 3, 3): T / n = H = 1.75
    h = np.zeros(256, dtype=np.uint64)
    h[:4] = [4, 2, 1, 1]
    L[:4] = [1, 2, 3, 3]
    assert oracle.drift_gap(h, L) == pytest.approx(0.0, abs=1e-15)
    # uniform over 4 symbols (H = 2) with the same lengths: T / n = 9 / 4, gap 1/8
    h[:4] = [5, 5, 5, 5]
    assert oracle.drift_gap(h, L) == pytest.approx(0.125, rel=1e-15)
    # (0.9, 0.1) with two 1-bit codes: H = 0.469 < 1, so the bound is one bit per symbol: gap 0
    h2 = np.zeros(256, dtype=np.uint64)
    h2[:2] = [9, 1]
    L2 = np.zeros(256, dtype=np.uint8)
    L2[:2] = [1, 1]
    assert oracle.drift_gap(h2, L2) == 0.0
    # a present symbol without a code: infinite; an empty shard: 0
    h2[7] = 1
    assert oracle.drift_gap(h2, L2) == float("inf")
    assert oracle.drift_gap(np.zeros(256), L2) == 0.0
