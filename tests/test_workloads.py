"""The seeded input generators (CPU): shapes, determinism and the
distribution properties the workloads are described by."""
import numpy as np
import torch

from lossless_huffman_compression_gb300 import workloads


def test_tensor_type_shards_are_seeded_and_shaped():
    for t in workloads.TENSOR_TYPES:
        a = workloads.tensor_type_shard(t, 2, warmup=True, shape=(64, 128))
        b = workloads.tensor_type_shard(t, 2, warmup=True, shape=(64, 128))
        c = workloads.tensor_type_shard(t, 2, warmup=False, shape=(64, 128))
        assert a.shape == (64, 128) and a.dtype == torch.int8
        assert torch.equal(a, b)
        assert not torch.equal(a, c)  # warm-up and test shards use other seeds


def test_tensor_type_distributions():
    n = (512, 512)
    w = workloads.tensor_type_shard("weight", 0, warmup=True, shape=n).numpy().astype(np.float64)
    a = workloads.tensor_type_shard("activation", 0, warmup=True, shape=n).numpy().astype(np.float64)
    g = workloads.tensor_type_shard("gradient", 0, warmup=True, shape=n).numpy().astype(np.float64)
    assert abs(w.std() - 12.0) < 0.3 and abs(w.mean()) < 0.2
    assert a.min() >= 0 and abs((a == 0).mean() - 0.5 - 0.5 * (1 - np.exp(-0.5 / 16))) < 0.01
    assert abs(a[a > 0].mean() - 16.5) < 1.0  # rounded Exp(mean 16) above zero
    assert abs(np.abs(g).mean() - 3.0) < 0.15 and abs(g.mean()) < 0.05  # Laplace(b = 3): E|x| = b
