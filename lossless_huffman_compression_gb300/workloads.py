"""Seeded synthetic inputs for the five tensor workloads.

This module only draws random tensors; it holds none of the codec's
arithmetic, so both the GPU path and the CPU oracle consume its output.
Each generator is deterministic for a given (seed, device, size).  GPU and
CPU draws differ (different generator engines), so a comparison always runs
both sides on the same materialised bytes.

Workloads (stand-ins for the pages' Gemma 2B tensors and LLM checkpoints,
which are not available):

* ``per_shard_int8``    -- int8 clamp(round(N(0, 8))), 1 Mi elements, seed 0.
* ``fixed_codebook_shard`` -- int8 shards; per shard sigma ~ U(10, 14); each
  element is clamp(round(N(0, sigma))) with probability 0.999, else a uniform
  integer in [-128, 127].  Warm-up shards [2048, 2048] use seeds 1000 + k,
  test shards [8192, 2048] seeds 2000 + k.
* ``bf16_weights``      -- bf16 [16384, 32768] from fp32 N(0, 0.02), round to
  nearest even; a Bernoulli(1e-4) mask of outliers with random sign and
  magnitude U(0.5, 4).  Seed 3.
* ``snapshot_pair``     -- x0 = bf16(N(0, 0.02)) [65536, 30518] (seed 4);
  x1 = bf16(fp32(x0) + N(0, 1e-4)) (noise seed 5).
* ``sweep_segment``     -- int8 segment k (256 MiB) of a 16 GiB stream; the
  distribution cycles N(0,4), N(0,16), N(0,48), Laplace(b=8), uniform
  [-128, 127]; seed 5000 + k.
* ``tensor_type_shard`` -- int8 shards of three tensor types for a codebook
  bank: "weight" clamp(round(N(0, 12))); "activation" 0 with probability 0.5,
  else clamp(round(Exp(mean 16))) (non-negative, like ReLU outputs);
  "gradient" clamp(round(Laplace(b = 3))).  Warm-up shard k of type t uses
  seed 7000 + 100 t + k, test shard k seed 7050 + 100 t + k.
"""
from __future__ import annotations

import math
import torch

PER_SHARD_N = 1 << 20
WARMUP_SHARDS = 16
WARMUP_SHAPE = (2048, 2048)
TEST_SHARDS = 64
TEST_SHAPE = (8192, 2048)
BF16_WEIGHTS_SHAPE = (16384, 32768)
SNAPSHOT_SHAPE = (65536, 30518)
SWEEP_SEGMENTS = 64
SWEEP_SEGMENT_BYTES = 256 << 20
SWEEP_KINDS = ("gauss4", "gauss16", "gauss48", "laplace8", "uniform")
TENSOR_TYPES = ("weight", "activation", "gradient")
TYPE_WARMUP_SHAPE = (1024, 2048)
TYPE_TEST_SHAPE = (4096, 2048)

_BLOCK = 1 << 26  # elements drawn per block, bounds temporary memory


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(seed)
    return g


def _clamp_round_int8(x: torch.Tensor) -> torch.Tensor:
    return torch.round(x).clamp_(-128, 127).to(torch.int8)


def int8_gaussian(n: int, sigma: float, seed: int, device="cpu") -> torch.Tensor:
    """clamp(round(N(0, sigma)), -128, 127) as int8[n]."""
    g = _gen(seed, device)
    out = torch.empty(n, dtype=torch.int8, device=device)
    for s in range(0, n, _BLOCK):
        e = min(n, s + _BLOCK)
        x = torch.randn(e - s, generator=g, device=device, dtype=torch.float32)
        out[s:e] = _clamp_round_int8(x.mul_(sigma))
    return out


def per_shard_int8(device="cpu", n: int = PER_SHARD_N, seed: int = 0) -> torch.Tensor:
    """Per-shard workload: int8 clamp(round(N(0, 8)))."""
    return int8_gaussian(n, 8.0, seed, device)


def fixed_codebook_shard(k: int, warmup: bool, device="cpu", shape=None) -> torch.Tensor:
    """Warm-up shard k (seed 1000 + k) or test shard k (seed 2000 + k)."""
    if shape is None:
        shape = WARMUP_SHAPE if warmup else TEST_SHAPE
    n = int(math.prod(shape))
    g = _gen((1000 if warmup else 2000) + k, device)
    sigma = 10.0 + 4.0 * float(torch.rand(1, generator=g, device=device).item())
    out = torch.empty(n, dtype=torch.int8, device=device)
    for s in range(0, n, _BLOCK):
        e = min(n, s + _BLOCK)
        x = _clamp_round_int8(torch.randn(e - s, generator=g, device=device).mul_(sigma))
        mask = torch.rand(e - s, generator=g, device=device) < 1e-3
        uni = torch.randint(-128, 128, (e - s,), generator=g, device=device, dtype=torch.int32).to(torch.int8)
        out[s:e] = torch.where(mask, uni, x)
    return out.view(shape)


def bf16_weights(device="cpu", shape=BF16_WEIGHTS_SHAPE, seed: int = 3, dtype=torch.bfloat16) -> torch.Tensor:
    """bf16 N(0, 0.02) with 1e-4 outliers of magnitude U(0.5, 4) and random sign (the same recipe in
    another float dtype with `dtype`, e.g. the fp32 byte-plane measurement)."""
    n = int(math.prod(shape))
    g = _gen(seed, device)
    out = torch.empty(n, dtype=dtype, device=device)
    for s in range(0, n, _BLOCK):
        e = min(n, s + _BLOCK)
        x = torch.randn(e - s, generator=g, device=device).mul_(0.02)
        mask = torch.rand(e - s, generator=g, device=device) < 1e-4
        sign = torch.where(torch.rand(e - s, generator=g, device=device) < 0.5, -1.0, 1.0)
        mag = torch.rand(e - s, generator=g, device=device).mul_(3.5).add_(0.5)
        out[s:e] = torch.where(mask, sign * mag, x).to(dtype)
    return out.view(shape)


def snapshot_pair(device="cpu", shape=SNAPSHOT_SHAPE, seeds=(4, 5)):
    """(x0, x1): x0 = bf16(N(0, 0.02)), x1 = bf16(fp32(x0) + N(0, 1e-4))."""
    n = int(math.prod(shape))
    g0 = _gen(seeds[0], device)
    g1 = _gen(seeds[1], device)
    x0 = torch.empty(n, dtype=torch.bfloat16, device=device)
    x1 = torch.empty(n, dtype=torch.bfloat16, device=device)
    for s in range(0, n, _BLOCK):
        e = min(n, s + _BLOCK)
        a = torch.randn(e - s, generator=g0, device=device).mul_(0.02).to(torch.bfloat16)
        x0[s:e] = a
        x1[s:e] = (a.float() + torch.randn(e - s, generator=g1, device=device).mul_(1e-4)).to(torch.bfloat16)
    return x0.view(shape), x1.view(shape)


def sweep_kind(k: int) -> str:
    return SWEEP_KINDS[k % len(SWEEP_KINDS)]


def sweep_segment(k: int, device="cpu", nbytes: int = SWEEP_SEGMENT_BYTES) -> torch.Tensor:
    """Segment k of the chunk-size sweep stream, int8[nbytes], seed 5000 + k."""
    g = _gen(5000 + k, device)
    kind = sweep_kind(k)
    out = torch.empty(nbytes, dtype=torch.int8, device=device)
    for s in range(0, nbytes, _BLOCK):
        e = min(nbytes, s + _BLOCK)
        m = e - s
        if kind.startswith("gauss"):
            sigma = float(kind[5:])
            out[s:e] = _clamp_round_int8(torch.randn(m, generator=g, device=device).mul_(sigma))
        elif kind == "laplace8":
            u = torch.rand(m, generator=g, device=device, dtype=torch.float64) - 0.5
            x = -8.0 * torch.sign(u) * torch.log1p(-2.0 * u.abs())
            out[s:e] = _clamp_round_int8(x.float())
        else:
            out[s:e] = torch.randint(-128, 128, (m,), generator=g, device=device, dtype=torch.int32).to(torch.int8)
    return out


def tensor_type_shard(kind: str, k: int, warmup: bool, device="cpu", shape=None) -> torch.Tensor:
    """Warm-up or test shard k of a tensor type (int8)."""
    t = TENSOR_TYPES.index(kind)
    if shape is None:
        shape = TYPE_WARMUP_SHAPE if warmup else TYPE_TEST_SHAPE
    n = int(math.prod(shape))
    g = _gen(7000 + 100 * t + (0 if warmup else 50) + k, device)
    out = torch.empty(n, dtype=torch.int8, device=device)
    for s in range(0, n, _BLOCK):
        e = min(n, s + _BLOCK)
        m = e - s
        if kind == "weight":
            out[s:e] = _clamp_round_int8(torch.randn(m, generator=g, device=device).mul_(12.0))
        elif kind == "activation":
            u = torch.rand(m, generator=g, device=device, dtype=torch.float64)
            x = -16.0 * torch.log1p(-torch.rand(m, generator=g, device=device, dtype=torch.float64))
            out[s:e] = _clamp_round_int8(torch.where(u < 0.5, torch.zeros_like(x), x).float())
        else:
            u = torch.rand(m, generator=g, device=device, dtype=torch.float64) - 0.5
            x = -3.0 * torch.sign(u) * torch.log1p(-2.0 * u.abs())
            out[s:e] = _clamp_round_int8(x.float())
    return out.view(shape)
