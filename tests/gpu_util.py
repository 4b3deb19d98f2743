"""Helpers shared by the GPU parity tests (comparison plumbing only; no codec arithmetic)."""
import numpy as np
import torch

import oracle
from lossless_huffman_compression_gb300 import _lib, codec


def dev_u8(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def host_u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().reshape(-1).view(torch.uint8).cpu().numpy()


def bits_of(payload: np.ndarray, start: int, end: int) -> np.ndarray:
    """Stream bits [start, end) as a 0/1 array (MSB-first byte order)."""
    if end <= start:
        return np.zeros(0, dtype=np.uint8)
    b0, b1 = start // 8, (end + 7) // 8
    bits = np.unpackbits(payload[b0:b1])
    return bits[start - 8 * b0:end - 8 * b0]


def oracle_codebook(hist, max_len=24, flags=0):
    ln = oracle.code_lengths(hist, max_len, flags)
    return ln, oracle.canonical_codes(ln)


def assert_stream_equal(gpu_stream: codec.Stream, ref_payload: np.ndarray, ref_off: np.ndarray):
    off = host(gpu_stream.off).astype(np.uint64)
    np.testing.assert_array_equal(off, ref_off)
    T = int(ref_off[-1])
    nb = (T + 7) // 8
    pay = host(gpu_stream.payload)
    np.testing.assert_array_equal(pay[:nb], ref_payload[:nb])
    # zero padding up to the end of the last written 32-bit word
    end_word = ((T + 31) // 32) * 4
    assert not pay[nb:end_word].any()


def check_sampled_chunks(payload: np.ndarray, off: np.ndarray, symbols: np.ndarray, ln, cd, chunk: int,
                         chunks) -> None:
    """The GPU bits of each sampled chunk equal the oracle's encoding of that chunk alone."""
    n = symbols.size
    for c in chunks:
        s = symbols[c * chunk: min(n, (c + 1) * chunk)]
        ref_pay, ref_off = oracle.encode(s, ln, cd, chunk)
        got = bits_of(payload, int(off[c]), int(off[c + 1]))
        want = bits_of(ref_pay, 0, int(ref_off[-1]))
        assert got.size == want.size, f"chunk {c}: {got.size} bits, oracle {want.size}"
        np.testing.assert_array_equal(got, want, err_msg=f"chunk {c}")


def assert_offsets_match_lengths(off: torch.Tensor, symbols, n: int, ln, chunk: int, block: int = 1 << 27):
    """Every chunk's bit count off[c+1] - off[c] equals the sum of len[x] over its symbols, and off[0] = 0.

    ``symbols(lo, hi)`` returns the device uint8 symbols [lo, hi).  Lengths are gathered with torch on
    the device, block by block, so the check covers every chunk of a multi-GB stream without the
    decoder or the oracle's encoder."""
    offs = off.to(torch.int64)
    assert int(offs[0].item()) == 0
    diff = offs[1:] - offs[:-1]
    lens = torch.as_tensor(np.asarray(ln, dtype=np.int64), device=off.device)
    per = max(1, block // chunk)  # chunks per block
    n_chunks = (n + chunk - 1) // chunk
    assert diff.numel() == n_chunks
    for c0 in range(0, n_chunks, per):
        c1 = min(n_chunks, c0 + per)
        lo, hi = c0 * chunk, min(n, c1 * chunk)
        L = lens.gather(0, symbols(lo, hi).to(torch.int64))
        pad = (c1 - c0) * chunk - (hi - lo)  # the ragged last chunk
        if pad:
            L = torch.cat([L, torch.zeros(pad, dtype=torch.int64, device=L.device)])
        want = L.view(c1 - c0, chunk).sum(1)
        bad = torch.nonzero(want != diff[c0:c1])
        assert bad.numel() == 0, f"chunk {c0 + int(bad[0, 0])}: offsets differ from the summed code lengths"
        del L, want
