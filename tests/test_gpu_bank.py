"""A bank of fixed codebooks, one per tensor type (weights, activations,
gradients): each built from that type's warm-up histogram, each tensor encoded
with its type's codebook, bit for bit against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from lossless_huffman_compression_gb300 import _lib, codec, workloads
from gpu_util import assert_stream_equal, host, host_u8

pytestmark = pytest.mark.gpu

TYPES = workloads.TENSOR_TYPES
WARMUP = 3
SMALL = (256, 1024)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    _lib.load()
    assert torch.cuda.is_available()


@pytest.fixture(scope="module")
def bank_and_ref():
    bank = codec.CodebookBank(TYPES)
    ref = {t: np.zeros(256, dtype=np.uint64) for t in TYPES}
    for t in TYPES:
        for k in range(WARMUP):
            x = workloads.tensor_type_shard(t, k, warmup=True, device="cuda", shape=SMALL)
            bank.observe(t, x)
            ref[t] += oracle.histogram(host_u8(x))
    bank.build()
    return bank, ref


def test_bank_histograms_and_lengths(bank_and_ref):
    bank, ref = bank_and_ref
    for i, t in enumerate(TYPES):
        np.testing.assert_array_equal(host(bank.hists[i]).astype(np.uint64), ref[t])
        np.testing.assert_array_equal(bank.codebook(t).lengths(), oracle.code_lengths(ref[t], 24, oracle.REF_COVER_ALL))


@pytest.mark.parametrize("t", TYPES)
def test_bank_streams_match_oracle(bank_and_ref, t):
    bank, ref = bank_and_ref
    ln = oracle.code_lengths(ref[t], 24, oracle.REF_COVER_ALL)
    cd = oracle.canonical_codes(ln)
    x = workloads.tensor_type_shard(t, 0, warmup=False, device="cuda", shape=SMALL)
    s = bank.encode(t, x, 4096)
    pay, off = oracle.encode(host_u8(x), ln, cd, 4096)
    assert_stream_equal(s, pay, off)
    assert torch.equal(bank.decode(t, s), x.reshape(-1).view(torch.uint8))


def test_own_type_codebook_is_the_cheapest(bank_and_ref):
    # each type's shards cost least under its own codebook, and less than under one codebook of all types
    bank, ref = bank_and_ref
    pooled = sum(ref.values())
    ln_pool = oracle.code_lengths(pooled, 24, oracle.REF_COVER_ALL)
    for t in TYPES:
        x = workloads.tensor_type_shard(t, 1, warmup=False, device="cuda", shape=SMALL)
        h = oracle.histogram(host_u8(x))
        cost = {u: oracle.total_bits(h, bank.codebook(u).lengths()) for u in TYPES}
        assert cost[t] == min(cost.values())
        assert cost[t] < oracle.total_bits(h, ln_pool)
        assert bank.encode(t, x, 16384).total_bits() == cost[t]


def test_bank_errors():
    with pytest.raises(ValueError):
        codec.CodebookBank(["a", "a"])
    bank = codec.CodebookBank(["a", "b"])
    with pytest.raises(RuntimeError):
        bank.codebook("a")
    bank.build()  # no observations: every symbol gets a code all the same
    assert (bank.codebook("b").lengths() == 8).all()
    with pytest.raises(KeyError):
        bank.codebook("c")
