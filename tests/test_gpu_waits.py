"""The bounded device waits give up with HUFF_ERR_TIMEOUT instead of hanging.

The encode kernels wait in two places: the decoupled lookback over segment
descriptors (a warp polls earlier segments' published bit counts) and the
bulk-copy mbarriers of each warp's ring.  huff_debug_wait runs each of them on
its own with a small poll limit, against a descriptor the host leaves
unpublished and an mbarrier that nothing arrives on and no copy targets, so the
wait runs out with nothing in flight.  Checks: the kernel returns, the status
is HUFF_ERR_TIMEOUT, the polls stop at the limit, a waiter that finds an error
already recorded stops at its first check (256 polls) rather than the limit,
and a lookback whose descriptors are all published sums them exactly.
"""
import pytest
import torch

from lossless_huffman_compression_gb300 import _lib

pytestmark = pytest.mark.gpu

AGG = 1 << 62
PRE = 2 << 62


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    _lib.load()
    assert torch.cuda.is_available()


def _desc(values):
    """Descriptors as device int64 (the uint64 bit patterns)."""
    return torch.tensor([v - (1 << 64) if v >= 1 << 63 else v for v in values], dtype=torch.int64, device="cuda")


def _run(kind, desc, seg, limit, status=None):
    out = torch.zeros(2, dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda") if status is None else status
    _lib.huff_debug_wait(kind, desc, seg, limit, out, st)
    torch.cuda.synchronize()
    return int(out[0].item()), int(out[1].item()), int(st.item())


def test_lookback_over_published_descriptors_sums_them():
    # segment 0 holds its inclusive prefix; 1 and 2 their aggregates: the prefix of segment 3 is 5 + 7 + 9
    excl, polls, st = _run(0, _desc([PRE | 5, AGG | 7, AGG | 9]), 3, 1024)
    assert (excl, polls, st) == (21, 0, 0)
    # the nearest inclusive prefix ends the walk: 100 (prefix of segment 1) + 9
    excl, polls, st = _run(0, _desc([PRE | 5, PRE | 100, AGG | 9]), 3, 1024)
    assert (excl, polls, st) == (109, 0, 0)


def test_lookback_on_an_unpublished_descriptor_times_out():
    excl, polls, st = _run(0, _desc([PRE | 5, 0, AGG | 3]), 3, 1024)
    assert st == _lib.HUFF_ERR_TIMEOUT
    assert polls == 1025  # gave up on the first poll past the limit


def test_a_second_waiter_stops_early_once_an_error_is_recorded():
    st = torch.full((1,), _lib.HUFF_ERR_TIMEOUT, dtype=torch.int32, device="cuda")
    _, polls, s = _run(0, _desc([PRE | 5, 0, AGG | 3]), 3, 1 << 20, st)
    assert s == _lib.HUFF_ERR_TIMEOUT  # the first error stays
    assert polls == 256  # the first check of the status, far below the limit


def test_mbarrier_wait_with_nothing_arriving_times_out():
    _, polls, st = _run(1, None, 0, 1000)
    assert st == _lib.HUFF_ERR_TIMEOUT
    assert polls == 1000


def test_debug_wait_rejects_bad_arguments():
    out = torch.zeros(2, dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = _desc([PRE | 1])
    for kind, desc, seg, limit in ((2, d, 1, 10), (0, d, 0, 10), (0, d, 2, 10), (0, d, 1, 0), (1, None, 0, (1 << 20) + 1)):
        with pytest.raises(_lib.HuffError):
            _lib.huff_debug_wait(kind, desc, seg, limit, out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
