"""The whole-stream offsets check used by the full-size GPU tests, run on CPU tensors against the
oracle's own offsets: it accepts them, rejects a moved offset, and handles a ragged last chunk."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_offsets_match_lengths


@pytest.mark.parametrize("n,chunk,block", [(10_000, 256, 1024), (65_536, 4096, 8192), (5, 256, 1 << 27)])
def test_offsets_check_agrees_with_the_oracle(n, chunk, block):
    rng = np.random.default_rng(n)
    x = np.clip(np.round(rng.normal(0, 6, n)), -128, 127).astype(np.int8).view(np.uint8)
    ln = oracle.code_lengths(oracle.histogram(x))
    _, off = oracle.encode(x, ln, oracle.canonical_codes(ln), chunk)
    xt = torch.from_numpy(x)
    ot = torch.from_numpy(off.astype(np.int64))
    assert_offsets_match_lengths(ot, lambda a, b: xt[a:b], n, ln, chunk, block)
    if off.size > 2:
        bad = ot.clone()
        bad[1] += 1  # a chunk boundary moved by one bit
        with pytest.raises(AssertionError):
            assert_offsets_match_lengths(bad, lambda a, b: xt[a:b], n, ln, chunk, block)
