"""bench.py's host-side bookkeeping (CPU only): the kernel-source hash that keys
the committed DRAM-traffic records ignores comments and blank space but not
code, a record whose hash no longer matches reports null, and the committed
records are well formed."""
import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    csrc = tmp_path / "lossless_huffman_compression_gb300" / "csrc"
    csrc.mkdir(parents=True)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setitem(bench.KERNEL_SOURCES, "k_probe", "probe.cu")
    f = csrc / "probe.cu"
    f.write_text("// a kernel\nint f(int x) {  /* doubles */\n    return 2 * x;\n}\n")
    h0 = bench.kernel_hash("k_probe")
    f.write_text("// the same kernel, other words\n\nint f(int x) {\n    return 2 * x;  // twice\n}\n")
    assert bench.kernel_hash("k_probe") == h0
    f.write_text("int f(int x) {\n    return 3 * x;\n}\n")
    assert bench.kernel_hash("k_probe") != h0


def test_stale_record_reports_null(tmp_path, monkeypatch):
    csrc = tmp_path / "lossless_huffman_compression_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setitem(bench.KERNEL_SOURCES, "k_probe", "probe.cu")
    (csrc / "probe.cu").write_text("int f() { return 1; }\n")
    rec = {"k_probe": {"source": "probe.cu", "source_sha256_16": bench.kernel_hash("k_probe"),
                       "dram_bytes_per_unit": 2.5}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic("k_probe", 4.0) == 10.0
    (csrc / "probe.cu").write_text("int f() { return 2; }\n")
    assert bench.recorded_traffic("k_probe", 4.0) is None


def test_committed_records_are_well_formed():
    """Each record names a kernel the bench knows, its source file, a 16-hex-digit hash and a
    positive byte count (whether it still matches its source is the bench's to report)."""
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    for name, r in rec.items():
        if name.startswith("_"):
            continue
        assert name in bench.KERNEL_SOURCES and r["source"] == bench.KERNEL_SOURCES[name]
        assert len(r["source_sha256_16"]) == 16 and int(r["source_sha256_16"], 16) >= 0
        assert r["dram_bytes_per_unit"] > 0 and os.path.exists(os.path.join(ROOT, r["capture"]))


def test_host_info():
    h = bench.host_info()
    assert h["machine"] and h["cpus"] >= 1
