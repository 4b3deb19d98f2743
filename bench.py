#!/usr/bin/env python3
"""Throughput of the canonical Huffman hot path on one GB300 (or N, weak-scaled).

Default workload: the incremental snapshot delta.  x0 = bf16(N(0, 0.02)) and
x1 = bf16(x0 + N(0, 1e-4)) of shape [65536, 30518] (2.0e9 elements, 4.0 GB
each), resident in HBM.  One step is one pass of the whole path:
  lmc_histogram_bf16_counted(x1, x0)  XOR delta + byte planes + two histograms
                                      (+ per-segment counts)
  huff_build_codebooks (both planes)  lengths, canonical codes, decode tables
  lmc_encode_bf16_counted(x1, x0)     XOR delta + byte planes + one-pass encode of both planes
  lmc_decode_bf16(..., x0)        decode both planes, merge, XOR x0 back in
value = snapshot bytes (2n) / step time: uncompressed GB/s of a full
compress + decompress round trip.  Inputs (8 GB) exceed the 129 MB L2, so no
flush is needed between steps.

--impl reference times the CPU oracle (the only reference this method has)
on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Huffman encode/decode GB/s (uncompressed) at 1 GB300; % HBM roofline; ratio"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = {"k_decode_bf16": "decode.cu", "k_encode_counted": "encode.cu", "k_histogram_bf16_counted": "histogram.cu"}


# ------------------------------------------------------------------ environment
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group(backend=backend)
        return dist
    return None


def max_over_ranks(dist, v: float, device) -> float:
    if dist is None:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, v: float, device) -> float:
    if dist is None:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t)
    return float(t.item())


def whole_job(dist, units_local: float, ms_local: float, device):
    """Weak scaling over replicas: (units all ranks processed / max step time over ranks, that time)."""
    ms = max_over_ranks(dist, ms_local, device)
    total = sum_over_ranks(dist, units_local, device)
    return total / (ms / 1e3), ms


def barrier(dist):
    if dist is not None:
        dist.barrier()


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def host_info() -> dict:
    """The machine the numbers come from (the GPU host may be Arm or x86)."""
    return {"machine": platform.machine(), "cpus": os.cpu_count()}


def kernel_hash(name: str) -> str:
    """Hash of the kernel's source file without its comments and blank space, so that a comment edit
    keeps a traffic record that the code it was measured on still matches."""
    src = os.path.join(ROOT, "lossless_huffman_compression_gb300", "csrc", KERNEL_SOURCES[name])
    with open(src, encoding="utf-8") as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    text = " ".join(text.split())
    return hashlib.sha256(text.encode()).hexdigest()[:16]


def recorded_traffic(name: str, units: float):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            j = json.load(f)
        e = j[name]
        if e.get("source_sha256_16") != kernel_hash(name):
            return None
        return float(e["dram_bytes_per_unit"]) * units
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 50 ms.

    start() returns once the first sample has arrived, so that sampling is
    already running when the timed region opens; begin()/end() bracket that
    region on the host clock, and the summary keeps the samples taken inside
    it (all samples only if none fell inside, which the summary says)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.lines = []
        self.thread = None
        self.first = threading.Event()
        self.t_begin = None
        self.t_end = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.period_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        self.first.wait(timeout=10.0)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))
            self.first.set()

    def begin(self):
        self.t_begin = time.monotonic()

    def end(self):
        self.t_end = time.monotonic()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(self.period_ms / 1000.0)  # one more sample after the region
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for t, ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((t, float(f[1]), float(f[2]), f[5:9]))
            except ValueError:
                continue
        if not rows:
            return None
        inside = [r for r in rows if self.t_begin is not None and self.t_end is not None
                  and self.t_begin <= r[0] <= self.t_end]
        window = "timed region" if inside else "around the timed region"
        use = inside or rows
        reasons = set()
        for r in use:
            for nm, v in zip(names, r[3]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "samples": len(use), "window": window, "period_ms": self.period_ms, "reasons": sorted(reasons)}


# ------------------------------------------------------------------ our arm
class SnapshotPath:
    """Buffers and the step for the snapshot-delta workload."""

    def __init__(self, x0, x1, chunk, max_len=24):
        from lossless_huffman_compression_gb300 import _lib, codec
        self.L = _lib
        self.codec = codec
        dev = x1.device
        self.x0 = x0.reshape(-1).view(torch.int16)
        self.x1 = x1.reshape(-1).view(torch.int16)
        self.n = n = self.x1.numel()
        self.chunk = chunk
        self.max_len = max_len
        self.hists = torch.zeros((2, 256), dtype=torch.int64, device=dev)  # high plane, low plane
        self.h_hi, self.h_lo = self.hists[0], self.hists[1]
        self.cbs = torch.zeros((2, _lib.huff_codebook_size()), dtype=torch.uint8, device=dev)
        self.cb_hi, self.cb_lo = codec.Codebook(buf=self.cbs[0]), codec.Codebook(buf=self.cbs[1])
        cap = _lib.huff_encode_bound(n, max_len)
        self.p_hi = torch.empty(cap, dtype=torch.uint8, device=dev)
        self.p_lo = torch.empty(cap, dtype=torch.uint8, device=dev)
        self.nc = _lib.huff_num_chunks(n, chunk)
        self.o_hi = torch.empty(self.nc + 1, dtype=torch.int64, device=dev)
        self.o_lo = torch.empty(self.nc + 1, dtype=torch.int64, device=dev)
        self.ws = torch.empty(_lib.lmc_workspace_size(n, chunk) // 8 + 2, dtype=torch.int64, device=dev)
        self.seg = torch.empty(_lib.lmc_segment_counts_size(n) // 4 + 4, dtype=torch.int32, device=dev)
        self.ws_counted = torch.empty(_lib.lmc_counted_workspace_size(n) // 8 + 2, dtype=torch.int64, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.out = torch.empty(n, dtype=torch.int16, device=dev)
        # kernels launched per step: hist (1 zero of both adjacent histograms + 1), build (1 for both planes),
        # encode (1 zero of the scan ticket + segment bits and scan + main + fix-up), decode (2: the kernels of
        # the high plane's two cases, of which one returns at once)
        self.launches_per_step = 9

    def compress(self, w=None, x0=None):
        L = self.L
        w = self.x1 if w is None else w
        x0 = self.x0 if x0 is None else x0
        L.lmc_histogram_bf16_counted(w, x0, self.h_hi, self.h_lo, self.seg)
        L.huff_build_codebooks(self.hists, self.cbs, self.status, self.max_len, 0)
        L.lmc_encode_bf16_counted(w, x0, self.cb_hi.buf, self.cb_lo.buf, self.chunk, self.seg, self.p_hi, self.o_hi,
                                  self.p_lo, self.o_lo, self.ws_counted, self.status)

    def decompress(self, x0=None, out=None):
        x0 = self.x0 if x0 is None else x0
        out = self.out if out is None else out
        self.L.lmc_decode_bf16(self.p_hi, self.o_hi, self.p_lo, self.o_lo, self.n, self.chunk, self.cb_hi.buf,
                               self.cb_lo.buf, x0, out, self.status)

    def step_with_events(self, ev):
        L = self.L
        ev[0].record()
        L.lmc_histogram_bf16_counted(self.x1, self.x0, self.h_hi, self.h_lo, self.seg)
        ev[1].record()
        L.huff_build_codebooks(self.hists, self.cbs, self.status, self.max_len, 0)
        ev[2].record()
        L.lmc_encode_bf16_counted(self.x1, self.x0, self.cb_hi.buf, self.cb_lo.buf, self.chunk, self.seg, self.p_hi,
                                  self.o_hi, self.p_lo, self.o_lo, self.ws_counted, self.status)
        ev[3].record()
        L.lmc_decode_bf16(self.p_hi, self.o_hi, self.p_lo, self.o_lo, self.n, self.chunk, self.cb_hi.buf,
                          self.cb_lo.buf, self.x0, self.out, self.status)
        ev[4].record()

    def check(self):
        torch.cuda.synchronize()
        st = int(self.status.item())
        if st != 0:
            raise RuntimeError(f"device status {st}: {self.L.status_string(st)}")
        if not torch.equal(self.out, self.x1):
            raise RuntimeError("decoded snapshot differs from x1")

    def sizes(self):
        T_hi = int(self.o_hi[-1].item())
        T_lo = int(self.o_lo[-1].item())
        return T_hi, T_lo


def run_ours(args, dist, rank, ws):
    from lossless_huffman_compression_gb300 import workloads
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    shape = (args.rows, workloads.SNAPSHOT_SHAPE[1])
    x0, x1 = workloads.snapshot_pair(device=dev, shape=shape)
    path = SnapshotPath(x0, x1, args.chunk)
    n = path.n
    snap_bytes = 2 * n

    for _ in range(args.warmup):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        path.step_with_events(ev)
    path.check()  # lossless and error-free before timing

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    barrier(dist)
    torch.cuda.synchronize()
    clocks.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks.begin()
    t0.record()
    for k in range(args.steps):
        path.step_with_events(evs[k])
    t1.record()
    torch.cuda.synchronize()
    clocks.end()
    barrier(dist)
    clk = clocks.stop()
    ms_local = t0.elapsed_time(t1) / args.steps
    units_per_s, ms = whole_job(dist, float(2 * n), ms_local, dev)
    path.check()

    stage_names = ["histogram_bf16_xor", "build_codebooks", "encode_bf16_xor", "decode_bf16_xor"]
    stage_ms = {nm: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs) for i, nm in enumerate(stage_names)}
    T_hi, T_lo = path.sizes()
    C = (T_hi + 7) // 8 + (T_lo + 7) // 8
    offs = 2 * 8 * (path.nc + 1)
    peak, peak_kind = hbm_peak()
    alg = {  # algorithmic bytes per launch
        "histogram_bf16_xor": 4 * n + 2 * 2048,
        "build_codebooks": 2 * (2048 + 21504),
        "encode_bf16_xor": 4 * n + C + offs,
        "decode_bf16_xor": C + offs + 4 * n,
    }
    stages = {}
    for nm in stage_names:
        t = stage_ms[nm] / 1e3
        stages[nm] = {"ms": round(stage_ms[nm], 4), "gbs_uncompressed": round(snap_bytes / t / 1e9, 1),
                      "alg_bytes": int(alg[nm]), "hbm_frac": round(alg[nm] / t / 1e9 / peak, 4)}
    dom = max(["histogram_bf16_xor", "encode_bf16_xor", "decode_bf16_xor"], key=lambda k: stage_ms[k])
    kname = {"histogram_bf16_xor": "k_histogram_bf16_counted", "encode_bf16_xor": "k_encode_counted",
             "decode_bf16_xor": "k_decode_bf16"}[dom]
    achieved = alg[dom] / (stage_ms[dom] / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} hbm_gbs",
                "traffic": recorded_traffic(kname, float(n))}

    # extra: encode / decode of the already-materialised delta (codebooks given), outside the step
    extra = materialised_delta_stages(path, args, peak)
    planes_fp32 = byte_planes_stage(args, peak) if not args.no_extras else None
    drift = drift_stage(args) if not args.no_extras else None
    loopback = loopback_stage(args) if not args.no_extras else None
    bank = bank_stage(args) if not args.no_extras else None

    # quality
    from lossless_huffman_compression_gb300 import _lib
    h_hi = path.h_hi.cpu().numpy().astype(np.uint64)
    h_lo = path.h_lo.cpu().numpy().astype(np.uint64)
    s_hi = _lib.huff_code_stats(h_hi, path.cb_hi.lengths())
    s_lo = _lib.huff_code_stats(h_lo, path.cb_lo.lengths())
    quality = {
        "payload_ratio": round(snap_bytes / C, 4),
        "container_ratio": round(snap_bytes / (C + offs + 512), 4),
        "hi_bits_per_symbol": round(s_hi["mean_len"], 4), "hi_entropy": round(s_hi["entropy_bits"], 4),
        "lo_bits_per_symbol": round(s_lo["mean_len"], 4), "lo_entropy": round(s_lo["entropy_bits"], 4),
        "hi_shannon_gap": round(s_hi["shannon_gap"], 5), "lo_shannon_gap": round(s_lo["shannon_gap"], 5),
    }

    e2e = None
    if not args.no_e2e:
        e2e = e2e_snapshot(path, x0, x1, args, dist, dev)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_snapshot(x0, x1, args)

    value = units_per_s / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": {"workload": f"snapshot_delta_bf16_{args.rows}x{workloads.SNAPSHOT_SHAPE[1]}",
                   "elements": n, "uncompressed_bytes": snap_bytes, "chunk_bytes": args.chunk,
                   "picked_chunk": _lib.huff_pick_chunk(n, delta=True), "max_len": 24,
                   "step": "xor+split+hist with segment counts, both codebooks in one launch, one-pass fused encode, "
                           "fused decode+merge+xor",
                   "l2": "inputs (8 GB) larger than L2; no flush", "parallelism": f"replicas{ws}"},
        "roofline": roofline, "stages": stages, "materialised_delta": extra, "byte_planes_fp32": planes_fp32,
        "drift_adaptive": drift, "loopback": loopback, "codebook_bank": bank,
        "quality": quality,
        "e2e": e2e, "cpu_baseline": cpu, "gpu_launches": path.launches_per_step * args.steps, "clocks": clk,
        # both planes' histograms of the input delta, hashed: the same seeds give the same inputs everywhere
        "input_hist_sha256_16": hashlib.sha256(path.hists.cpu().numpy().tobytes()).hexdigest()[:16],
        "host": host_info(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def byte_planes_stage(args, peak):
    """Byte grouping for another width: a 1 GiB fp32 tensor (the weights recipe in fp32) as 4 byte planes,
    compressed and decompressed through codec.compress_planes / decompress_planes (per-plane codebooks)."""
    from lossless_huffman_compression_gb300 import codec, workloads
    shape = (args.rows // 4, 16384) if args.rows < 65536 else (16384, 16384)
    x = workloads.bf16_weights(device="cuda", shape=shape, dtype=torch.float32)
    nbytes = x.numel() * 4
    chunk = 4096  # a plane of 2^28 bytes in 4 KiB chunks: 65536 chunks, enough lanes for every SM
    s = codec.compress_planes(x, chunk_bytes=chunk)
    back = codec.decompress_planes(s)
    if not torch.equal(back.view(torch.int32), x.view(torch.int32)):
        raise RuntimeError("fp32 byte-plane round trip differs")
    reps = 3
    res = {}
    for nm, fn in (("compress", lambda: codec.compress_planes(x, chunk_bytes=chunk)),
                   ("decompress", lambda: codec.decompress_planes(s))):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / reps
        res[nm] = {"ms": round(ms, 3), "gbs_uncompressed": round(nbytes / (ms / 1e3) / 1e9, 1)}
    payload = sum((st.total_bits() + 7) // 8 for _, st in s.planes)
    res.update({"shape": list(shape), "dtype": "fp32", "planes": 4, "chunk_bytes": chunk,
                "ratio": round(nbytes / payload, 4),
                "plane_bits_per_symbol": [round(st.total_bits() / x.numel(), 4) for _, st in s.planes],
                "api": "codec.compress_planes / decompress_planes (status checked per plane)"})
    del x, s, back
    torch.cuda.empty_cache()
    return res


def drift_stage(args):
    """Fixed vs drift-adaptive codebook on the sweep stream's first segments (kinds cycle every segment):
    codebook from the first 64 MiB with every symbol covered; adaptive = refresh when a segment's drift gap
    exceeds 2 % (huff_drift_check + huff_build_codebook_if before each segment's encode)."""
    from lossless_huffman_compression_gb300 import _lib, codec, workloads
    nseg = 20 if args.rows >= 65536 else 5
    seg = workloads.SWEEP_SEGMENT_BYTES
    segs = [workloads.sweep_segment(k, device="cuda").view(torch.uint8) for k in range(nseg)]
    head = segs[0][: 64 << 20]
    res = {"segments": nseg, "segment_bytes": seg, "threshold": 0.02, "chunk_bytes": args.chunk}
    for mode in ("fixed", "adaptive"):
        cb = codec.build_codebook(codec.histogram(head), 24, _lib.HUFF_COVER_ALL)
        ad = codec.DriftAdaptiveCodebook(cb, threshold=0.02) if mode == "adaptive" else None
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        bits, refreshes = 0, 0
        for x in segs:
            s = ad.encode(x, args.chunk) if ad else codec.encode(x, cb, args.chunk)
            bits += s.total_bits()
            if ad:
                refreshes += int(ad.refreshed.item())
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        res[mode] = {"ratio": round(nseg * seg * 8 / bits, 4), "refreshes": refreshes, "ms": round(ms, 2),
                     "gbs": round(nseg * seg / (ms / 1e3) / 1e9, 1)}
    del segs, head
    torch.cuda.empty_cache()
    return res


def _replay_ms(fn, reps):
    """Milliseconds per call of fn, replayed from a CUDA graph (launch costs out of the way); plain
    launches when capture is not possible.  Returns (ms, "graph" | "launches")."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    how = "graph"
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        run = g.replay
    except Exception:
        torch.cuda.synchronize()
        run, how = fn, "launches"
    for _ in range(3):
        run()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(reps):
        run()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps, how


def loopback_stage(args):
    """The one-GPU loopback of compressed communication: a message of int8 (the fixed-codebook
    workload's shards) goes encode -> device-to-device copy of the stream (its size read on the
    device) -> decode.  Fixed codebook (built once from 4 warm-up shards) against the per-shard
    pipeline, which also counts, builds a codebook and sends it with the stream.  Chunks of 1 KiB
    and 16 KiB: the decode runs one lane per chunk, so small messages want small chunks."""
    from lossless_huffman_compression_gb300 import _lib, codec, workloads
    hist = torch.zeros(256, dtype=torch.int64, device="cuda")
    for k in range(4):
        codec.histogram(workloads.fixed_codebook_shard(k, warmup=True, device="cuda"), hist, accumulate=True)
    cb = codec.build_codebook(hist, 24, _lib.HUFF_COVER_ALL)
    src = workloads.fixed_codebook_shard(0, warmup=False, device="cuda").reshape(-1).view(torch.uint8)
    big = torch.cat([src] * 16)  # 256 MiB
    res = {"sizes": []}
    for size, chunk in [(z, c) for z in (64 << 10, 1 << 20, 16 << 20, 256 << 20) for c in (1024, 16384)]:
        x = big[:size]
        cap = _lib.huff_encode_bound(size, 24)
        nc = _lib.huff_num_chunks(size, chunk)
        pay, pay2 = (torch.empty(cap, dtype=torch.uint8, device="cuda") for _ in range(2))
        off, off2 = (torch.empty(nc + 1, dtype=torch.int64, device="cuda") for _ in range(2))
        ws = torch.empty(max(_lib.huff_workspace_size(size, chunk), 16) // 8, dtype=torch.int64, device="cuda")
        out = torch.empty_like(x)
        st = codec.new_status()
        h2 = torch.zeros(256, dtype=torch.int64, device="cuda")
        cb_own, cb_sent = codec.Codebook(), codec.Codebook()

        def fixed():
            _lib.huff_encode(x, cb.buf, chunk, pay, off, ws, st)
            _lib.huff_stream_copy(pay, off, pay2, off2, st)
            _lib.huff_decode(pay2, off2, size, chunk, cb.buf, out, st)

        def per_shard():
            _lib.huff_histogram(x, h2)
            _lib.huff_build_codebook(h2, cb_own.buf, st)
            _lib.huff_encode(x, cb_own.buf, chunk, pay, off, ws, st)
            cb_sent.buf.copy_(cb_own.buf)  # the codebook travels with the stream
            _lib.huff_stream_copy(pay, off, pay2, off2, st)
            _lib.huff_decode(pay2, off2, size, chunk, cb_sent.buf, out, st)

        reps = 200 if size <= (1 << 20) else (40 if size <= (16 << 20) else 8)
        ms_f, how_f = _replay_ms(fixed, reps)
        ok_f = bool(torch.equal(out, x)) and int(st.item()) == 0
        bits_f = int(off2[-1].item())
        out.zero_()
        ms_p, how_p = _replay_ms(per_shard, reps)
        ok_p = bool(torch.equal(out, x)) and int(st.item()) == 0
        res["sizes"].append({
            "bytes": size, "chunk_bytes": chunk, "fixed_us": round(ms_f * 1e3, 1), "per_shard_us": round(ms_p * 1e3, 1),
            "fixed_gbs": round(size / (ms_f / 1e3) / 1e9, 1), "ratio_fixed": round(size * 8 / bits_f, 4),
            "timing": how_f if how_f == how_p else f"{how_f}/{how_p}", "lossless": ok_f and ok_p})
    del big, src
    torch.cuda.empty_cache()
    return res


def bank_stage(args):
    """Per-tensor-type codebook bank: 16 warm-up shards of each type observed, every type's codebook
    built in one launch, 8 test shards of each type encoded with their own type's codebook; compared
    with one codebook of all types pooled and with each shard's own codebook."""
    from lossless_huffman_compression_gb300 import _lib, codec, workloads
    types = workloads.TENSOR_TYPES
    bank = codec.CodebookBank(types)
    for t in types:
        for k in range(16):
            bank.observe(t, workloads.tensor_type_shard(t, k, warmup=True, device="cuda"))
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    bank.build()
    b.record()
    torch.cuda.synchronize()
    build_ms = a.elapsed_time(b)
    pooled = codec.build_codebook(bank.hists.sum(0), 24, _lib.HUFF_COVER_ALL)
    res = {"types": list(types), "warmup_shards": 16, "test_shards": 8, "build_ms": round(build_ms, 4),
           "ratio": {}}
    enc_ms, enc_bytes = 0.0, 0
    for t in types:
        tot = {"own_type": 0, "pooled": 0, "per_shard": 0}
        nbytes = 0
        for k in range(8):
            x = workloads.tensor_type_shard(t, k, warmup=False, device="cuda").reshape(-1).view(torch.uint8)
            nbytes += x.numel()
            a.record()
            s = bank.encode(t, x)
            b.record()
            torch.cuda.synchronize()
            enc_ms += a.elapsed_time(b)
            enc_bytes += x.numel()
            tot["own_type"] += s.total_bits()
            tot["pooled"] += codec.encode(x, pooled).total_bits()
            tot["per_shard"] += codec.encode(x, codec.build_codebook(codec.histogram(x))).total_bits()
            assert torch.equal(bank.decode(t, s), x)
        res["ratio"][t] = {kk: round(nbytes * 8 / v, 4) for kk, v in tot.items()}
    res["encode_gbs"] = round(enc_bytes / (enc_ms / 1e3) / 1e9, 1)
    res["encode_timing"] = "per call, including the status read"
    return res


def materialised_delta_stages(path, args, peak):
    """Encode and decode with the codebooks given (the fixed-codebook single stage): the snapshot delta
    straight from (x1, x0) and the byte-grouped delta d = x1 ^ x0 already held in HBM."""
    L = path.L
    n = path.n
    d = torch.empty_like(path.x1)
    L.lmc_delta_xor(path.x1, path.x0, d)
    reps = max(3, min(args.steps, 10))
    out = {}
    for nm, fn in (("encode_bf16_xor_given", lambda: L.lmc_encode_bf16(path.x1, path.x0, path.cb_hi.buf, path.cb_lo.buf,
                                                                       path.chunk, path.p_hi, path.o_hi, path.p_lo,
                                                                       path.o_lo, path.ws, path.status)),
                   ("encode_bf16", lambda: L.lmc_encode_bf16(d, None, path.cb_hi.buf, path.cb_lo.buf, path.chunk,
                                                             path.p_hi, path.o_hi, path.p_lo, path.o_lo, path.ws,
                                                             path.status)),
                   ("decode_bf16", lambda: L.lmc_decode_bf16(path.p_hi, path.o_hi, path.p_lo, path.o_lo, n,
                                                             path.chunk, path.cb_hi.buf, path.cb_lo.buf, None,
                                                             path.out, path.status))):
        fn()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / reps
        T_hi, T_lo = path.sizes()
        C = (T_hi + 7) // 8 + (T_lo + 7) // 8 + 2 * 8 * (path.nc + 1)
        alg = (4 * n if nm.endswith("xor_given") else 2 * n) + C
        out[nm] = {"ms": round(ms, 4), "gbs_uncompressed": round(2 * n / ms / 1e6, 1), "alg_bytes": alg,
                   "hbm_frac": round(alg / ms / 1e6 / peak, 4)}
    torch.cuda.synchronize()
    if not torch.equal(path.out, d):
        raise RuntimeError("materialised-delta decode differs")
    if int(path.status.item()) != 0:
        raise RuntimeError("materialised-delta status")
    out["note"] = ("codebooks given (the step's): encode_bf16_xor_given reads x1 and x0 (counting pass, then the "
                   "one-pass encode); encode_bf16 / decode_bf16 work on the byte-grouped delta already in HBM")
    del d
    return out


def host_link(h_a, h_b, h_out, d_a, d_b, d_out, s1, s2, s3):
    """The host link of this machine, measured after the e2e run with its own pinned buffers (its rate
    differs from box to box): host to device on two streams at once, device to host, and both
    directions at once; GB/s, CUDA events, the best of three."""
    def timed(copies):
        best = float("inf")
        for _ in range(3):
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(s1)
            for st in (s2, s3):
                st.wait_event(a)
            nbytes = 0
            for st, dst, src in copies:
                with torch.cuda.stream(st):
                    dst.copy_(src, non_blocking=True)
                nbytes += src.numel() * src.element_size()
            for st in (s2, s3):
                s1.wait_stream(st)
            b.record(s1)
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b))
        return round(nbytes / best / 1e6, 1)
    return {"h2d_gbs": timed([(s1, d_a, h_a), (s2, d_b, h_b)]),
            "d2h_gbs": timed([(s3, h_out, d_out)]),
            "both_gbs": timed([(s1, d_a, h_a), (s2, d_b, h_b), (s3, h_out, d_out)]),
            "how": "after the timed e2e steps: x1 and x0 to the device on two streams; the output to the host; "
                   "all three at once"}


def e2e_snapshot(path, x0, x1, args, dist, dev):
    """Same step through the public API with HOST buffers: copies inside the timed region.

    Every step copies that step's x1 and x0 from pinned host memory, compresses, copies the streams
    to the host and back (the stored form), decompresses with the x0 already on the device, and
    copies the result to the host.  The step is a pipeline over six streams: input copies (x1, x0),
    compress, the streams' round trip, decompress, output copy; inputs and outputs have three device
    buffers each and consecutive steps alternate between two sets of stream buffers, codebooks and
    workspaces, so no stage waits for a later stage of the step before it and the host-to-device
    link, the narrower direction, stays busy."""
    n = path.n
    paths = [path, SnapshotPath(x0, x1, path.chunk, path.max_len)]
    h_x1 = torch.empty(n, dtype=torch.int16, pin_memory=True)
    h_x0 = torch.empty(n, dtype=torch.int16, pin_memory=True)
    h_x1.copy_(path.x1)
    h_x0.copy_(path.x0)
    T_hi, T_lo = path.sizes()
    cap_hi = ((T_hi + 31) // 32) * 4
    cap_lo = ((T_lo + 31) // 32) * 4
    h_p_hi = torch.empty(cap_hi, dtype=torch.uint8, pin_memory=True)
    h_p_lo = torch.empty(cap_lo, dtype=torch.uint8, pin_memory=True)
    h_o_hi = torch.empty(path.nc + 1, dtype=torch.int64, pin_memory=True)
    h_o_lo = torch.empty(path.nc + 1, dtype=torch.int64, pin_memory=True)
    h_out = torch.empty(n, dtype=torch.int16, pin_memory=True)
    nbuf = 3
    d_x1 = [torch.empty_like(path.x1) for _ in range(nbuf)]
    d_x0 = [torch.empty_like(path.x0) for _ in range(nbuf)]
    d_out = [torch.empty_like(path.out) for _ in range(nbuf)]
    s_in, s_in2, s_comp, s_rt, s_dec, s_out = (torch.cuda.Stream() for _ in range(6))
    steps = max(3, min(args.steps, 24))  # the pipeline fills and drains over about one step
    free_in = [torch.cuda.Event() for _ in range(nbuf)]   # buffer k % nbuf's inputs may be overwritten
    free_out = [torch.cuda.Event() for _ in range(nbuf)]  # buffer k % nbuf's output has reached the host
    free_path = [torch.cuda.Event() for _ in paths]       # path k % 2's streams and codebooks are done with
    for e in free_in + free_out + free_path:
        e.record(torch.cuda.current_stream())

    def one(k):
        i = k % nbuf
        j = k % len(paths)
        P = paths[j]
        arrived, arrived2, compressed, restored, decoded = (torch.cuda.Event() for _ in range(5))
        with torch.cuda.stream(s_in):  # the two inputs on two streams: two copy engines at once
            s_in.wait_event(free_in[i])
            d_x1[i].copy_(h_x1, non_blocking=True)
            arrived.record(s_in)
        with torch.cuda.stream(s_in2):
            s_in2.wait_event(free_in[i])
            d_x0[i].copy_(h_x0, non_blocking=True)
            arrived2.record(s_in2)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(arrived)
            s_comp.wait_event(arrived2)
            s_comp.wait_event(free_path[j])
            P.compress(d_x1[i], d_x0[i])
            compressed.record(s_comp)
        with torch.cuda.stream(s_rt):  # the stored form: to the host and back (in order on this stream)
            s_rt.wait_event(compressed)
            h_p_hi.copy_(P.p_hi[:cap_hi], non_blocking=True)
            h_p_lo.copy_(P.p_lo[:cap_lo], non_blocking=True)
            h_o_hi.copy_(P.o_hi, non_blocking=True)
            h_o_lo.copy_(P.o_lo, non_blocking=True)
            P.p_hi[:cap_hi].copy_(h_p_hi, non_blocking=True)
            P.p_lo[:cap_lo].copy_(h_p_lo, non_blocking=True)
            P.o_hi.copy_(h_o_hi, non_blocking=True)
            P.o_lo.copy_(h_o_lo, non_blocking=True)
            restored.record(s_rt)
        with torch.cuda.stream(s_dec):
            s_dec.wait_event(restored)
            s_dec.wait_event(free_out[i])
            P.decompress(d_x0[i], d_out[i])
            decoded.record(s_dec)
            free_in[i].record(s_dec)
            free_path[j].record(s_dec)
        with torch.cuda.stream(s_out):
            s_out.wait_event(decoded)
            h_out.copy_(d_out[i], non_blocking=True)
            free_out[i].record(s_out)

    one(0)
    torch.cuda.synchronize()
    barrier(dist)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for k in range(steps):
        one(k + 1)
    for s in (s_in2, s_comp, s_rt, s_dec, s_out):
        s_in.wait_stream(s)
    b.record(s_in)
    torch.cuda.synchronize()
    ms = max_over_ranks(dist, a.elapsed_time(b) / steps, dev)
    for P in paths:
        st = int(P.status.item())
        if st != 0:
            raise RuntimeError(f"e2e device status {st}: {P.L.status_string(st)}")
    if not torch.equal(h_out, h_x1):
        raise RuntimeError("e2e round trip differs")
    total = sum_over_ranks(dist, float(2 * n), dev)
    h2d = 2 * n * 2 + cap_hi + cap_lo + 2 * 8 * (path.nc + 1)
    d2h = 2 * n + cap_hi + cap_lo + 2 * 8 * (path.nc + 1)
    link = host_link(h_x1, h_x0, h_out, d_x1[0], d_x0[0], d_out[0], s_in, s_in2, s_out)
    link["moved_gbs"] = round((h2d + d2h) / ms / 1e6, 1)  # both directions, the e2e step's own rate
    del d_x1, d_x0, d_out, paths
    return {"value": round(total / ms / 1e6, 2), "unit": "GB/s", "ms_per_step": round(ms, 3), "steps": steps,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "link": link,
            "api": "lmc_histogram_bf16_counted, huff_build_codebooks, lmc_encode_bf16_counted, lmc_decode_bf16 with pinned host "
                   "inputs, streams copied to host and back; a pipeline over six streams (input copies, compress, "
                   "round trip, decompress, output copy), consecutive steps on alternating buffer sets"}


# ------------------------------------------------------------------ oracle timing
def oracle_snapshot_step(x0h: np.ndarray, x1h: np.ndarray, chunk: int):
    """The oracle's full path on one sample: delta, planes, codebooks, encode, decode, merge, re-apply."""
    import oracle
    d = oracle.delta_xor(x1h, x0h)
    hi, lo = oracle.bytegroup_split(d)
    planes = []
    for p in (hi, lo):
        ln = oracle.code_lengths(oracle.histogram(p))
        cd = oracle.canonical_codes(ln)
        pay, off = oracle.encode(p, ln, cd, chunk)
        planes.append(oracle.decode(pay, off, p.size, chunk, ln))
    back = oracle.delta_xor(oracle.bytegroup_merge(planes[0], planes[1]), x0h)
    if not np.array_equal(back, x1h):
        raise RuntimeError("oracle round trip failed")


def snapshot_sample(x0, x1, elems):
    a = x0.reshape(-1)[:elems].view(torch.int16).cpu().numpy().view(np.uint16)
    b = x1.reshape(-1)[:elems].view(torch.int16).cpu().numpy().view(np.uint16)
    return a, b


PAGES_16CORE = {"compress_gibs": 2.78, "decompress_gibs": 3.76,
                "source": "Lossless Compression for LLM Tensor Incremental Snapshots, English abstract / "
                          "experiment highlights (16-core CPU)"}


def _thread_counts():
    n = os.cpu_count() or 1
    return sorted({t for t in (1, 16, n) if t <= n})


def cpu_baseline_snapshot(x0, x1, args):
    """The oracle on the host's cores: the sequential oracle on one thread, and its per-chunk steps over
    16 and all host threads (oracle/huff_oracle_mt.c, payload byte-identical to the sequential oracle's),
    each on the first elements of the snapshot pair; compress and decompress timed apart, as the pages
    report them."""
    import oracle
    from oracle import mt
    oracle.build()
    elems = args.cpu_sample
    a, b = snapshot_sample(x0, x1, elems)
    rows = {}
    for t in _thread_counts():
        if t == 1:  # the sequential oracle as it stands, on a quarter of the sample
            e1 = max(1, elems // 4)
            t0 = time.perf_counter()
            oracle_snapshot_step(a[:e1], b[:e1], args.chunk)
            dt = time.perf_counter() - t0
            rows["1"] = {"elements": e1, "round_trip_gbs": round(2 * e1 / dt / 1e9, 4), "seconds": round(dt, 2),
                         "how": "sequential oracle (delta, planes, histograms, codebooks, encode, decode, merge)"}
            continue
        size, tc, td = mt.snapshot_round_trip(a, b, args.chunk, t)
        rows[str(t)] = {"elements": elems, "compress_gibs": round(2 * elems / tc / 2 ** 30, 3),
                        "decompress_gibs": round(2 * elems / td / 2 ** 30, 3),
                        "round_trip_gbs": round(2 * elems / (tc + td) / 1e9, 4), "seconds": round(tc + td, 2)}
    top = str(max(_thread_counts()))
    return {"value": rows[top]["round_trip_gbs"], "unit": "GB/s", "cores": int(top), "kind": "oracle",
            "sample": f"first {elems} elements of x0/x1 (the snapshot's own distribution), compress + decompress "
                      f"round trip; one thread: the sequential oracle on {rows['1']['elements']} elements",
            "by_threads": rows, "pages_16core": PAGES_16CORE, "host": host_info()}


def run_reference(args, dist, rank, ws):
    """The oracle on the host's cores (its per-chunk steps over every host thread), on a bounded sample
    per step; rank 0 only."""
    if rank != 0:
        return
    import oracle
    from oracle import mt
    oracle.build()
    from lossless_huffman_compression_gb300 import workloads
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    shape = (args.rows, workloads.SNAPSHOT_SHAPE[1])
    x0, x1 = workloads.snapshot_pair(device=dev, shape=shape)
    elems = min(args.ref_sample, x0.numel())
    a, b = snapshot_sample(x0, x1, elems)
    del x0, x1
    threads = os.cpu_count() or 1
    for _ in range(args.warmup):
        mt.snapshot_round_trip(a[: max(1, elems // 8)], b[: max(1, elems // 8)], args.chunk, threads)
    times = []
    for _ in range(args.steps):
        _, tc, td = mt.snapshot_round_trip(a, b, args.chunk, threads)
        times.append(tc + td)
    ms = 1e3 * sum(times) / len(times)
    value = 2 * elems / (ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "impl": "reference", "value": round(value, 4), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": {"workload": f"snapshot_delta_bf16_{args.rows}x30518", "chunk_bytes": args.chunk,
                   "sample_elements": elems},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"first {elems} elements of x0/x1 per step, compress + decompress round trip "
                                   f"over {threads} host threads"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "host": host_info(),
    }
    print(json.dumps(line), flush=True)


def _timed(fn, reps):
    fn()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def run_workload(args):
    """One JSON line per stage for the four other workloads (parity cases, measured for the record):
    per_shard (int8 1 MiB), fixed_codebook (16 warm-up + 64 test int8 shards), bf16_weights (1 GiB,
    2 planes), sweep (16 GiB int8, chunk sizes 16 KiB .. 1 MiB).  GB/s of uncompressed bytes; codec API
    calls (status checked per call)."""
    from lossless_huffman_compression_gb300 import _lib, codec, workloads
    torch.cuda.set_device(0)
    peak, peak_kind = hbm_peak()
    reps = max(3, args.steps)
    out = {"metric": METRIC, "workload": args.workload, "n_gpus": 1, "data": "synthetic", "peak_gbs": peak,
           "peak_source": peak_kind, "host": host_info()}
    def hist_sha(t):  # the byte histogram of an input, hashed: the same seeds give the same inputs everywhere
        return hashlib.sha256(codec.histogram(t.reshape(-1).view(torch.uint8)).cpu().numpy().tobytes()).hexdigest()[:16]

    if args.workload == "per_shard":
        x = workloads.per_shard_int8(device="cuda").view(torch.uint8)
        out["input_hist_sha256_16"] = hist_sha(x)
        n = x.numel()
        cb, s = codec.compress(x, args.chunk)
        comp = _timed(lambda: codec.compress(x, args.chunk), reps)
        dec = _timed(lambda: codec.decode(s, cb), reps)
        stats = _lib.huff_code_stats(codec.histogram(x).cpu().numpy(), cb.lengths())
        out.update({"elements": n, "chunk_bytes": args.chunk, "l2": "1 MiB: L2-resident, latency-bound",
                    "compress_us": round(comp * 1e3, 1), "decode_us": round(dec * 1e3, 1),
                    "compress_gbs": round(n / comp / 1e6, 2), "decode_gbs": round(n / dec / 1e6, 2),
                    "ratio": round(8 * n / s.total_bits(), 4), "entropy_bits": round(stats["entropy_bits"], 4),
                    "mean_len": round(s.total_bits() / n, 4)})
    elif args.workload == "fixed_codebook":
        hist = torch.zeros(256, dtype=torch.int64, device="cuda")
        for k in range(workloads.WARMUP_SHARDS):
            codec.histogram(workloads.fixed_codebook_shard(k, warmup=True, device="cuda"), hist, accumulate=True)
        cb = codec.build_codebook(hist, 24, _lib.HUFF_COVER_ALL)
        shards = [workloads.fixed_codebook_shard(k, warmup=False, device="cuda").view(torch.uint8).reshape(-1)
                  for k in range(workloads.TEST_SHARDS)]
        out["input_hist_sha256_16"] = hashlib.sha256(hist.cpu().numpy().tobytes()).hexdigest()[:16]  # warm-up
        n = sum(x.numel() for x in shards)
        res = {}
        fixed_bits = 0
        # the bench's chunk size, and the one huff_pick_chunk gives a shard (one wave of full decode blocks:
        # small chunks, whose offsets cost ratio)
        for chunk in dict.fromkeys((args.chunk, _lib.huff_pick_chunk(shards[0].numel()))):
            streams = [codec.encode(x, cb, chunk) for x in shards]
            enc = _timed(lambda: [codec.encode(x, cb, chunk) for x in shards], 3)
            dec = _timed(lambda: [codec.decode(st, cb) for st in streams], 3)
            # the same calls back to back, each with its own status, all statuses read once at the end
            sts = [codec.new_status() for _ in shards]
            outs = [torch.empty_like(x) for x in shards]

            def enc_pipe():
                for x, st in zip(shards, sts):
                    codec.encode(x, cb, chunk, status=st)

            def dec_pipe():
                for s_, o, st in zip(streams, outs, sts):
                    codec.decode(s_, cb, out=o, status=st)

            enc_p = _timed(enc_pipe, 3)
            dec_p = _timed(dec_pipe, 3)
            for st in sts:
                codec.raise_on_status(st, "fixed-codebook shard")
            for x, o in zip(shards, outs):
                if not torch.equal(x, o):
                    raise RuntimeError("fixed-codebook decode differs")
            fixed_bits = sum(st.total_bits() for st in streams)
            container = sum(_lib.huff_container_size(x.numel(), chunk, st.total_bits(), False)
                            for x, st in zip(shards, streams))
            res[str(chunk)] = {"encode_gbs": round(n / enc / 1e6, 1), "decode_gbs": round(n / dec / 1e6, 1),
                               "pipelined": {"encode_gbs": round(n / enc_p / 1e6, 1),
                                             "decode_gbs": round(n / dec_p / 1e6, 1)},
                               "container_ratio": round(n / container, 4)}
            del streams, outs
        shard_bits, nh = 0, 0.0
        for x in shards:  # per-shard Huffman of each shard, through the library's own statistics
            h = codec.histogram(x).cpu().numpy().astype(np.uint64)
            ln = codec.build_codebook(torch.from_numpy(h.astype(np.int64)).cuda()).lengths()
            st_ = _lib.huff_code_stats(h, ln)
            shard_bits += st_["total_bits"]
            nh += st_["entropy_bits"] * x.numel()
        first = res[str(args.chunk)]
        out.update({"elements": n, "shards": len(shards), "chunk_bytes": args.chunk,
                    "encode_gbs": first["encode_gbs"], "decode_gbs": first["decode_gbs"],
                    "pipelined": dict(first["pipelined"],
                                      how="the 64 shard calls back to back, statuses read once at the end"),
                    "picked_chunk": _lib.huff_pick_chunk(shards[0].numel()), "per_chunk_size": res,
                    "ratio": round(8 * n / fixed_bits, 4),
                    "gap_vs_per_shard_huffman": round((fixed_bits - shard_bits) / shard_bits, 5),
                    "gap_vs_entropy": round((fixed_bits - nh) / nh, 5)})
    elif args.workload == "bf16_weights":
        x = workloads.bf16_weights(device="cuda")
        n = x.numel()
        out["input_hist_sha256_16"] = hist_sha(x)
        res = {}
        # the bench's chunk size, and the one huff_pick_chunk gives for this size without a delta (one
        # wave of full decode blocks on every SM)
        for chunk in dict.fromkeys((args.chunk, _lib.huff_pick_chunk(n))):
            s = codec.compress_bf16(x, None, chunk)
            comp = _timed(lambda: codec.compress_bf16(x, None, chunk), reps)
            dec = _timed(lambda: codec.decompress_bf16(s), reps)
            C = s.hi.nbytes() + s.lo.nbytes()
            offs = 2 * 8 * (s.hi.n_chunks() + 1)
            res[str(chunk)] = {"compress_gbs": round(2 * n / comp / 1e6, 1), "decode_gbs": round(2 * n / dec / 1e6, 1),
                               "compress_hbm_frac": round((C + offs + 2 * n) / (comp / 1e3) / 1e9 / peak, 4),
                               "decode_hbm_frac": round((C + offs + 2 * n) / (dec / 1e3) / 1e9 / peak, 4),
                               "ratio": round(2 * n / C, 4), "container_ratio": round(2 * n / (C + offs + 512), 4),
                               "bits_per_symbol": [round(s.hi.total_bits() / n, 4), round(s.lo.total_bits() / n, 4)]}
            del s
        out.update({"elements": n, "picked_chunk": _lib.huff_pick_chunk(n), "per_chunk_size": res})
    elif args.workload == "sweep":
        seg = workloads.SWEEP_SEGMENT_BYTES
        nseg = args.segments or workloads.SWEEP_SEGMENTS
        n = nseg * seg
        x = torch.empty(n, dtype=torch.uint8, device="cuda")
        for k in range(nseg):
            x[k * seg:(k + 1) * seg] = workloads.sweep_segment(k, device="cuda").view(torch.uint8)
        cb = codec.build_codebook(codec.histogram(x[: 64 << 20]), 24, _lib.HUFF_COVER_ALL)
        out["input_hist_sha256_16"] = hist_sha(x)
        res = {}
        dst = torch.empty_like(x)
        chunks = [int(c) for c in args.chunks.split(",")] if args.chunks else [16 << 10, 64 << 10, 256 << 10, 1 << 20]
        for chunk in chunks:
            st = codec.encode(x, cb, chunk)
            enc = _timed(lambda: codec.encode(x, cb, chunk), 2)
            dec = _timed(lambda: codec.decode(st, cb, out=dst), 2)
            C = st.nbytes()
            res[str(chunk)] = {"encode_gbs": round(n / enc / 1e6, 1), "decode_gbs": round(n / dec / 1e6, 1),
                               "decode_hbm_frac": round((C + n) / (dec / 1e3) / 1e9 / peak, 4),
                               "ratio": round(n / C, 4)}
            del st
        out.update({"elements": n, "segments": nseg, "per_chunk_size": res})
    print(json.dumps(out), flush=True)


def relaunch_ranks(n: int) -> int:
    """--gpus N > 1 outside a torchrun job: run this same command as N ranks (one per GPU, rendezvous on
    127.0.0.1) under torch.distributed.run and return its exit status."""
    import socket
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        port = sock.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


# The snapshot's chunk: 2.0e9 elements in 136 168 chunk pairs, 896-lane decode blocks (the widest whose x0
# staging fits in shared memory; 7 warps per scheduler) on all 152 SMs; huff_pick_chunk's choice for this
# size with a delta.
SNAPSHOT_CHUNK = 14688


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--chunk", type=int, default=None,
                    help=f"symbols per chunk (default {SNAPSHOT_CHUNK} for the snapshot, 16384 for the other workloads)")
    ap.add_argument("--rows", type=int, default=65536,
                    help="snapshot rows of 30518 bf16 (65536 = the 4.0 GB workload; fewer for quick checks)")
    ap.add_argument("--small", action="store_true", help="same as --rows 4096 (a 250 MB snapshot)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the fp32 byte-plane and drift measurements")
    ap.add_argument("--workload", choices=["snapshot", "per_shard", "fixed_codebook", "bf16_weights", "sweep"],
                    default="snapshot", help="snapshot = the default benchmark line; the others print their own")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--segments", type=int, default=0,
                    help="sweep: 256 MiB segments (0 = all 64, the 16 GiB workload; fewer for profiling runs)")
    ap.add_argument("--chunks", default="", help="sweep: comma-separated chunk sizes (default 16K,64K,256K,1M)")
    ap.add_argument("--cpu-sample", type=int, default=256 << 20, help="elements for the oracle baseline (about 10 s)")
    ap.add_argument("--ref-sample", type=int, default=64 << 20, help="elements per reference step")
    args = ap.parse_args()
    if args.small:
        args.rows = 4096
    if args.chunk is None:
        args.chunk = SNAPSHOT_CHUNK if args.workload == "snapshot" else 16384
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ and args.workload == "snapshot":
        sys.exit(relaunch_ranks(args.gpus))
    ws, rank, local = dist_env()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.workload != "snapshot":
        run_workload(args)
        return
    if args.impl == "reference":
        dist = init_dist(ws, "gloo")
        run_reference(args, dist, rank, ws)
        if dist is not None:
            dist.destroy_process_group()
        return
    dist = init_dist(ws, "nccl")
    run_ours(args, dist, rank, ws)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
