"""Pure-Python tiny oracle -- TEST INFRASTRUCTURE, small inputs only (<= 1 MiB).

A second, independent restatement of the method, used to cross-check the C
oracle in ``huff_oracle.c``.  It uses a binary heap keyed by (count, id) for
Huffman's procedure, strings of '0'/'1' for bit streams and a dictionary of
code words for decoding, so it shares no step of its arithmetic with the C
oracle beyond the definitions themselves.

Sources: "Single-stage Huffman encoder for ML compression" (arXiv 2601.10673),
Methodology steps 1-4; "Lossless Compression for LLM Tensor Incremental
Snapshots" (arXiv 2505.09810), Method details / technical framework; RFC 1951
section 3.2.2 for canonical codes; ITU-T T.81 Annex K.3 for the length limit.
"""
from __future__ import annotations

import heapq
import itertools
import math
from collections import Counter

COVER_ALL = 1


def histogram(data: bytes) -> list[int]:
    """Symbol counts (C1)."""
    c = Counter(bytes(data))
    return [c.get(s, 0) for s in range(256)]


def huffman_depths(counts: list[int]) -> dict[int, int]:
    """Leaf depths of Huffman's tree; ties broken by (count, id) (C3).

    Leaves have id = symbol, internal nodes 256, 257, ... in creation order.
    """
    heap = [(c, s) for s, c in enumerate(counts) if c > 0]
    if not heap:
        return {}
    if len(heap) == 1:
        return {heap[0][1]: 1}
    heapq.heapify(heap)
    children: dict[int, tuple[int, int]] = {}
    next_id = 256
    while len(heap) > 1:
        c1, a = heapq.heappop(heap)
        c2, b = heapq.heappop(heap)
        children[next_id] = (a, b)
        heapq.heappush(heap, (c1 + c2, next_id))
        next_id += 1
    root = heap[0][1]
    depths: dict[int, int] = {}
    stack = [(root, 0)]
    while stack:
        node, d = stack.pop()
        if node < 256:
            depths[node] = d
        else:
            a, b = children[node]
            stack.append((a, d + 1))
            stack.append((b, d + 1))
    return depths


def code_lengths(counts: list[int], max_len: int = 24, flags: int = 0) -> list[int]:
    """Lengths after the max_len repair and the (count desc, symbol asc) reassignment (C4, C5)."""
    cnt = [max(c, 1) if (flags & COVER_ALL) else c for c in counts]
    if sum(cnt) >= 1 << 63:
        raise ValueError("counts must sum below 2^63")
    depths = huffman_depths(cnt)
    lengths = [0] * 256
    if not depths:
        return lengths
    if len(depths) == 1:
        (s,) = depths
        lengths[s] = 1
        return lengths
    bl = [0] * (max(depths.values()) + 2)
    for d in depths.values():
        bl[d] += 1
    for i in range(len(bl) - 1, max_len, -1):
        while bl[i] > 0:
            j = i - 2
            while bl[j] == 0:
                j -= 1
            bl[i] -= 2
            bl[i - 1] += 1
            bl[j + 1] += 2
            bl[j] -= 1
    order = sorted(depths, key=lambda s: (-cnt[s], s))
    it = iter(order)
    for L in range(1, len(bl)):
        for _ in range(bl[L]):
            lengths[next(it)] = L
    return lengths


def canonical_codes(lengths: list[int]) -> list[str]:
    """Canonical code words as bit strings; '' for absent symbols (C6).

    Codes of one length are consecutive integers in symbol order, and the
    first code of length L+1 is (last code of length L + 1) shifted left.
    """
    words = [""] * 256
    code = 0
    prev_len = 0
    for L, s in sorted((L, s) for s, L in enumerate(lengths) if L > 0):
        if prev_len:
            code = (code + 1) << (L - prev_len)
        prev_len = L
        words[s] = format(code, f"0{L}b")
    return words


def encode(data: bytes, lengths: list[int], chunk_bytes: int) -> tuple[bytes, list[int]]:
    """Bit string concatenation, MSB first, zero-padded to a byte (C7)."""
    words = canonical_codes(lengths)
    parts = []
    offsets = []
    pos = 0
    for i, s in enumerate(bytes(data)):
        if i % chunk_bytes == 0:
            offsets.append(pos)
        w = words[s]
        if not w:
            raise ValueError(f"symbol {s} not in codebook")
        parts.append(w)
        pos += len(w)
    offsets.append(pos)
    bits = "".join(parts)
    bits += "0" * (-len(bits) % 8)
    payload = bytes(int(bits[k:k + 8], 2) for k in range(0, len(bits), 8))
    return payload, offsets


def decode(payload: bytes, offsets: list[int], n: int, chunk_bytes: int, lengths: list[int]) -> bytes:
    """Prefix-code dictionary walk per chunk (C8)."""
    table = {w: s for s, w in enumerate(canonical_codes(lengths)) if w}
    bits = "".join(format(b, "08b") for b in payload)
    out = bytearray()
    n_chunks = (n + chunk_bytes - 1) // chunk_bytes
    for c in range(n_chunks):
        pos = offsets[c]
        want = min(chunk_bytes, n - c * chunk_bytes)
        for _ in range(want):
            w = ""
            while w not in table:
                if pos >= len(bits) or len(w) > 64:
                    raise ValueError("corrupt stream")
                w += bits[pos]
                pos += 1
            out.append(table[w])
        if pos != offsets[c + 1]:
            raise ValueError("chunk does not end at its offset")
    return bytes(out)


def entropy(counts: list[int]) -> float:
    """Shannon entropy in bits per symbol (C10)."""
    total = sum(counts)
    if total == 0:
        return 0.0
    return -sum(c / total * math.log2(c / total) for c in counts if c > 0)


def brute_force_min_cost(counts: list[int], max_len: int | None = None) -> int:
    """Minimum of sum(count * len) over all prefix codes (Kraft <= 1), tiny alphabets.

    Enumerates non-decreasing length multisets and pairs them with counts in
    descending order (the rearrangement inequality makes that pairing the best
    for a given multiset).
    """
    present = sorted((c for c in counts if c > 0), reverse=True)
    m = len(present)
    if m == 0:
        return 0
    if m == 1:
        return present[0]
    top = m - 1 if max_len is None else min(max_len, m - 1)
    best = None
    for ls in itertools.combinations_with_replacement(range(1, top + 1), m):
        if sum(2.0 ** -L for L in ls) > 1.0 + 1e-12:
            continue
        cost = sum(c * L for c, L in zip(present, ls))
        if best is None or cost < best:
            best = cost
    return best
