"""Drift-adaptive codebook refresh on the GPU against the oracle: the drift
gap of a shard under a codebook, the refresh decision, the conditional
rebuild, and an adaptive encode over a stream whose distribution changes."""
import numpy as np
import pytest
import torch

import oracle
from lossless_huffman_compression_gb300 import _lib, codec, workloads
from gpu_util import assert_stream_equal, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    _lib.load()
    assert torch.cuda.is_available()


def _hist(kind, n, rng):
    if kind == "gauss4":
        x = np.clip(np.round(rng.normal(0, 4, n)), -128, 127)
    elif kind == "gauss48":
        x = np.clip(np.round(rng.normal(0, 48, n)), -128, 127)
    elif kind == "laplace8":
        x = np.clip(np.round(rng.laplace(0, 8, n)), -128, 127)
    else:
        x = rng.integers(-128, 128, n)
    return oracle.histogram(x.astype(np.int8).view(np.uint8))


def _gpu_gap(h, cb, threshold):
    dh = torch.from_numpy(h.astype(np.int64)).cuda()
    flag = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    gap = torch.zeros(1, dtype=torch.float64, device="cuda")
    _lib.huff_drift_check(dh, cb.buf, threshold, flag, gap)
    return float(gap.item()), int(flag.item())


KINDS = ["gauss4", "gauss48", "laplace8", "uniform"]


@pytest.mark.parametrize("built_from", KINDS)
@pytest.mark.parametrize("shard", KINDS)
def test_gap_and_decision_match_oracle(built_from, shard):
    rng = np.random.default_rng(KINDS.index(built_from) * 10 + KINDS.index(shard))
    hb = _hist(built_from, 200_000, rng)
    cb = codec.build_codebook(torch.from_numpy(hb.astype(np.int64)).cuda(), 24, _lib.HUFF_COVER_ALL)
    ln = oracle.code_lengths(hb, 24, oracle.REF_COVER_ALL)
    np.testing.assert_array_equal(cb.lengths(), ln)
    hs = _hist(shard, 300_000, rng)
    want = oracle.drift_gap(hs, ln)
    # thresholds clear of the gap: the decision is then independent of rounding order
    for thr in [t for t in (want * 0.5, want * 2 + 1e-3) if t >= 0 and abs(t - want) > 1e-9]:
        got, flag = _gpu_gap(hs, cb, thr)
        assert got == pytest.approx(want, rel=1e-12, abs=1e-15)
        assert flag == int(want > thr)


def test_missing_symbol_is_infinite_drift():
    h = np.zeros(256, dtype=np.uint64)
    h[:3] = [100, 50, 25]
    cb = codec.build_codebook(torch.from_numpy(h.astype(np.int64)).cuda())
    h[200] = 1
    gap, flag = _gpu_gap(h, cb, 1e9)
    assert gap == float("inf") and flag == 1


def test_build_if_keeps_or_rebuilds():
    rng = np.random.default_rng(4)
    ha, hb = _hist("gauss4", 100_000, rng), _hist("uniform", 100_000, rng)
    cb = codec.build_codebook(torch.from_numpy(ha.astype(np.int64)).cuda(), 24, _lib.HUFF_COVER_ALL)
    before = cb.buf.clone()
    dh = torch.from_numpy(hb.astype(np.int64)).cuda()
    st = codec.new_status()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    _lib.huff_build_codebook_if(dh, flag, cb.buf, st, 24, _lib.HUFF_COVER_ALL)
    assert torch.equal(cb.buf, before)
    flag.fill_(1)
    _lib.huff_build_codebook_if(dh, flag, cb.buf, st, 24, _lib.HUFF_COVER_ALL)
    assert int(st.item()) == 0
    np.testing.assert_array_equal(cb.lengths(), oracle.code_lengths(hb, 24, oracle.REF_COVER_ALL))


def test_adaptive_encode_over_a_drifting_stream():
    seg = 1 << 20
    segments = [workloads.sweep_segment(k, device="cuda", nbytes=seg) for k in range(10)]
    head = segments[0][: seg // 4].view(torch.uint8)
    cb = codec.build_codebook(codec.histogram(head), 24, _lib.HUFF_COVER_ALL)
    ad = codec.DriftAdaptiveCodebook(cb, threshold=0.02)
    ln = oracle.code_lengths(oracle.histogram(host(head)), 24, oracle.REF_COVER_ALL)
    refreshes = 0
    for k, x in enumerate(segments):
        xb = host(x.view(torch.uint8))
        h = oracle.histogram(xb)
        refresh = oracle.drift_gap(h, ln) > 0.02
        if refresh:
            ln = oracle.code_lengths(h, 24, oracle.REF_COVER_ALL)
            refreshes += 1
        s = ad.encode(x.view(torch.uint8), 65536)
        assert int(ad.refreshed.item()) == int(refresh), f"segment {k}"
        np.testing.assert_array_equal(ad.cb.lengths(), ln)
        if k % 3 == 0:
            pay, off = oracle.encode(xb, ln, oracle.canonical_codes(ln), 65536)
            assert_stream_equal(s, pay, off)
        assert torch.equal(codec.decode(s, ad.cb), x.view(torch.uint8))
    assert refreshes >= 4  # the kind changes every segment
