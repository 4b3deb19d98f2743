"""The C ABI library builds here, loads without a GPU, and exports every
function include/huff.h declares; host-only helpers agree with the oracle."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "huff.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b((?:huff|lmc)_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from lossless_huffman_compression_gb300 import _lib
    return _lib


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 19
    so = ctypes.CDLL(lib.LIB_PATH)
    for name in names:
        assert hasattr(so, name), f"{name} declared in huff.h but not exported"
    assert sorted(lib.EXPORTS) == names


def test_header_compiles_as_plain_c(tmp_path):
    c = tmp_path / "t.c"
    c.write_text('#include "huff.h"\nint main(void){ return (int)sizeof(huff_codebook) > 0 ? 0 : 1; }\n')
    import subprocess
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                           "-o", str(tmp_path / "t"), str(c)])


def test_host_queries(lib):
    assert lib.huff_version() > 0
    assert lib.huff_status_string(-4) == "corrupt stream"
    assert lib.huff_codebook_size() >= 256 + 1024 + 4 * 4096
    assert lib.huff_encode_bound(1000, 24) >= 1000 * 3
    assert lib.huff_num_chunks(0, 256) == 0 and lib.huff_num_chunks(257, 256) == 2
    assert lib.huff_workspace_size(8192 * 3 + 1, 4096) >= 4 * 16


def test_code_stats_match_oracle(lib):
    rng = np.random.default_rng(1)
    x = np.clip(np.round(rng.normal(0, 8, 100_000)), -128, 127).astype(np.int8)
    h = oracle.histogram(x)
    ln = oracle.code_lengths(h)
    st = lib.huff_code_stats(h, ln)
    assert st["total_bits"] == oracle.total_bits(h, ln)
    assert st["entropy_bits"] == pytest.approx(oracle.entropy(h), rel=1e-12)
    assert st["n"] == x.size


def test_binding_fails_loudly_without_library(lib, tmp_path):
    import importlib
    mod = importlib.import_module("lossless_huffman_compression_gb300._lib")
    saved = mod._lib
    try:
        mod._lib = None
        with pytest.raises(RuntimeError):
            mod.load(str(tmp_path / "missing.so"))
    finally:
        mod._lib = saved


def test_chunk_size_limits_rejected_before_any_device_work(lib):
    """chunk_bytes must be a positive multiple of 32 and at most 2^30 (a chunk's symbol count
    stays an int with room for the decoder's ring arithmetic).  Argument checks come before
    any CUDA call, so rejected calls run here without a GPU; the pointers are aligned
    placeholders that a rejected call never touches."""
    L = lib.load()
    fake = ctypes.c_void_p(1 << 20)
    n = (1 << 31) + 512
    for chunk in (0, 1000, (1 << 30) + 256, 1 << 31):
        assert L.huff_decode(fake, 64, fake, n, chunk, fake, fake, fake, None) == lib.HUFF_ERR_INVALID_ARG
        assert L.huff_encode(fake, n, fake, chunk, fake, 64, fake, fake, 64, fake, None) == lib.HUFF_ERR_INVALID_ARG
        assert L.lmc_decode_bf16(fake, 64, fake, fake, 64, fake, n, chunk, fake, fake, fake, fake, fake,
                                 None) == lib.HUFF_ERR_INVALID_ARG
