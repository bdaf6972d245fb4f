"""The seeded input generator: deterministic, device-independent bits, and
the stated value distribution (CPU only; the GPU bit-identity check lives in
the GPU tests)."""

import numpy as np
import torch

from paged_decode_attention_store_gb300 import workloads as wl


def test_values_are_a_pure_function_of_the_index():
    k1, v1 = wl.kv_rows(7, 3, [1, 2, 3], [10, 11, 12], 8, 128)
    k2, _ = wl.kv_rows(7, 3, [3], [12], 8, 128)
    assert torch.equal(k1[2], k2[0])
    assert not torch.equal(k1, v1)
    k3, _ = wl.kv_rows(8, 3, [1, 2, 3], [10, 11, 12], 8, 128)
    assert not torch.equal(k1, k3)


def test_distribution_and_exact_grid():
    x = wl.hash_normal(0, 1, torch.arange(1 << 20, dtype=torch.int64))
    assert abs(x.mean().item()) < 0.01 and abs(x.std().item() - 1.0) < 0.01
    assert x.min().item() >= -382 / 128 and x.max().item() <= 383 / 128
    assert torch.equal(x * 128, torch.round(x * 128))  # multiples of 1/128: exact in float32
    # a bounded Irwin-Hall(3) shape: the fraction within one sigma is ~0.66
    frac = (x.abs() < 1.0).float().mean().item()
    assert 0.6 < frac < 0.72


def test_lengths_and_pools():
    w = wl.gqa_decode(0)
    assert len(w.lengths) == 64 and min(w.lengths) >= 512 and max(w.lengths) <= 4096
    need = sum(-(-L // 16) for L in w.lengths)
    assert w.num_pages == int(np.ceil(need * 1.1))
    assert sorted(w.free_order) == list(range(w.num_pages))
    lb = wl.large_batch(0, P=1)
    assert len(lb.lengths) == 256 and max(lb.lengths) <= 16384 - 256
    assert 700 < float(np.median(lb.lengths)) < 1400
