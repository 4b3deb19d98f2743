"""The pins have teeth: plausible mistakes planted in a copy of the tiny oracle fail them.

Each mutant swaps one step of ``oracle.tiny`` for a wrong variant (a flipped
tie-break, reversed canonical order, LSB-first packing, a dropped term of the
length-limit repair, the over-long lengths walked shortest first, J taken as the
shortest used length, the wrong merge rule, natural log for log2) and the same
pin checks that the real oracle passes must reject it.

A walk shortest-first that repeats until no length is over the limit (rather
than one pass) ended at the same BITS as the prescribed walk on every one of
20,000 random Huffman depth profiles tried, so it is not a distinct result and
has no mutant here.
"""
import heapq
import json
import math
import os

import pytest

from oracle import tiny


def _golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


class Impl:
    """The steps under test; mutants override one of them."""

    depths = staticmethod(tiny.huffman_depths)
    entropy = staticmethod(tiny.entropy)

    def lengths(self, counts, max_len=24):
        return _lengths_with(self, counts, max_len)

    def codes(self, lengths):
        return tiny.canonical_codes(lengths)

    def pack(self, words):
        bits = "".join(words)
        bits += "0" * (-len(bits) % 8)
        return bytes(int(bits[k:k + 8], 2) for k in range(0, len(bits), 8))

    def repair(self, bl, i, j):
        bl[i] -= 2
        bl[i - 1] += 1
        bl[j + 1] += 2
        bl[j] -= 1

    def pick_j(self, bl, i):
        j = i - 2
        while bl[j] == 0:
            j -= 1
        return j

    def limit(self, bl, max_len):
        for i in range(len(bl) - 1, max_len, -1):
            while bl[i] > 0:
                self.repair(bl, i, self.pick_j(bl, i))

    def order(self, present, cnt):
        return sorted(present, key=lambda s: (-cnt[s], s))


def _lengths_with(impl, counts, max_len):
    depths = impl.depths(counts)
    lengths = [0] * 256
    if len(depths) == 1:
        (s,) = depths
        lengths[s] = 1
        return lengths
    bl = [0] * (max(depths.values()) + 2)
    for d in depths.values():
        bl[d] += 1
    impl.limit(bl, max_len)
    it = iter(impl.order(list(depths), counts))
    for L in range(1, len(bl)):
        for _ in range(max(bl[L], 0)):
            lengths[next(it)] = L
    return lengths


def run_pins(impl, golden_dir):
    """The pin checks of test_oracle_pins.py, restated over an Impl."""
    # RFC 1951 worked example
    g = _golden(golden_dir, "rfc1951_canonical.json")
    ln = [0] * 256
    for k, v in g["lengths"].items():
        ln[int(k)] = v
    cw = impl.codes(ln)
    assert all(cw[int(k)] == v for k, v in g["codes"].items()), "rfc1951"
    # hand example: bit order
    g = _golden(golden_dir, "hand_small.json")
    counts = tiny.histogram(bytes(g["input"]))
    ln = impl.lengths(counts)
    cw = impl.codes(ln)
    assert impl.pack([cw[s] for s in g["input"]]).hex() == g["payload_hex"], "hand_small"
    # hand example: tie-break and reassignment
    g = _golden(golden_dir, "hand_ties.json")
    counts = [0] * 256
    for k, v in g["counts"].items():
        counts[int(k)] = v
    assert {str(k): v for k, v in impl.depths(counts).items()} == g["tree_depths"], "tree depths"
    ln = impl.lengths(counts)
    assert all(ln[int(k)] == v for k, v in g["lengths"].items()), "reassignment"
    # dyadic closed form
    g = _golden(golden_dir, "dyadic.json")
    counts = [0] * 256
    for k, v in g["counts"].items():
        counts[int(k)] = v
    assert abs(impl.entropy(counts) - g["entropy_bits"]) < 1e-12, "entropy"
    # brute-force optimality on tiny alphabets
    for cs in ([5, 1, 1, 1, 1, 9], [3, 3, 3, 3, 2], [40, 20, 10, 5, 3, 1, 1]):
        counts = cs + [0] * (256 - len(cs))
        ln = impl.lengths(counts)
        assert sum(c * l for c, l in zip(counts, ln)) == tiny.brute_force_min_cost(counts), "optimality"
    # Kraft equality after the length limit (Fibonacci counts, depth 29 > 24)
    fib = [1, 1]
    while len(fib) < 30:
        fib.append(fib[-1] + fib[-2])
    ln = impl.lengths(fib + [0] * 226, 24)
    top = max(ln)
    assert top <= 24 and sum(1 << (top - l) for l in ln if l) == 1 << top, "kraft"
    # the length-limit repair, hand-derived move by move from T.81 Annex K.3
    for case in _golden(golden_dir, "adjust_bits.json")["cases"]:
        counts = [0] * 256
        if "counts" in case:
            for k, v in case["counts"].items():
                counts[int(k)] = v
            want = [0] * 256
            for k, v in case["lengths"].items():
                want[int(k)] = v
        else:
            counts[:30] = fib
            want = case["lengths_by_symbol"] + [0] * 226
        assert impl.lengths(counts, case["max_len"]) == want, case["name"]


class WrongTieBreak(Impl):
    @staticmethod
    def depths(counts):
        heap = [(c, -s) for s, c in enumerate(counts) if c > 0]
        heapq.heapify(heap)
        parent = {}
        nid = 256
        while len(heap) > 1:
            c1, a = heapq.heappop(heap)
            c2, b = heapq.heappop(heap)
            parent[-a if a <= 0 else a] = nid
            parent[-b if b <= 0 else b] = nid
            heapq.heappush(heap, (c1 + c2, nid))
            nid += 1
        out = {}
        for s, c in enumerate(counts):
            if c > 0:
                d, v = 0, s
                while v in parent:
                    v = parent[v]
                    d += 1
                out[s] = d
        return out


class ReversedCanonicalOrder(Impl):
    def codes(self, lengths):
        rev = tiny.canonical_codes(lengths[::-1])
        return rev[::-1]


class LsbFirstPacking(Impl):
    def pack(self, words):
        bits = "".join(words)
        bits += "0" * (-len(bits) % 8)
        return bytes(int(bits[k:k + 8][::-1], 2) for k in range(0, len(bits), 8))


class RepairDropsATerm(Impl):
    def repair(self, bl, i, j):
        bl[i] -= 2
        bl[i - 1] += 1
        bl[j + 1] += 1
        bl[j] -= 1


class RepairShortestDepthFirst(Impl):
    """Walks the over-long lengths from the shortest one up, once each (instead of from the longest)."""

    def limit(self, bl, max_len):
        for i in range(max_len + 1, len(bl)):
            while bl[i] > 0:
                self.repair(bl, i, self.pick_j(bl, i))


class RepairJShortestUsed(Impl):
    """Takes J as the shortest used length instead of the longest used one at most I - 2."""

    def pick_j(self, bl, i):
        return min(k for k in range(1, len(bl)) if bl[k] > 0)


class ReassignSymbolDescending(Impl):
    def order(self, present, cnt):
        return sorted(present, key=lambda s: (-cnt[s], -s))


class MergeLargest(Impl):
    @staticmethod
    def depths(counts):
        nodes = {s: c for s, c in enumerate(counts) if c > 0}
        parent = {}
        nid = 256
        while len(nodes) > 1:
            a = max(nodes, key=lambda v: (nodes[v], -v))
            ca = nodes.pop(a)
            b = max(nodes, key=lambda v: (nodes[v], -v))
            cb = nodes.pop(b)
            parent[a] = parent[b] = nid
            nodes[nid] = ca + cb
            nid += 1
        out = {}
        for s, c in enumerate(counts):
            if c > 0:
                d, v = 0, s
                while v in parent:
                    v = parent[v]
                    d += 1
                out[s] = d
        return out


class NaturalLogEntropy(Impl):
    @staticmethod
    def entropy(counts):
        t = sum(counts)
        return -sum(c / t * math.log(c / t) for c in counts if c)


def test_real_oracle_passes_the_pins(golden_dir):
    run_pins(Impl(), golden_dir)


@pytest.mark.parametrize("mutant", [WrongTieBreak, ReversedCanonicalOrder, LsbFirstPacking,
                                    RepairDropsATerm, RepairShortestDepthFirst, RepairJShortestUsed,
                                    ReassignSymbolDescending, MergeLargest,
                                    NaturalLogEntropy])
def test_planted_mistake_is_caught(mutant, golden_dir):
    with pytest.raises(AssertionError):
        run_pins(mutant(), golden_dir)
