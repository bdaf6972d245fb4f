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


def test_distribution_is_standard_normal():
    import statistics

    x = wl.hash_normal(0, 1, torch.arange(1 << 21, dtype=torch.int64)).double()
    assert abs(x.mean().item()) < 0.005 and abs(x.std().item() - 1.0) < 0.005
    # the empirical CDF follows Phi everywhere (Kolmogorov-Smirnov distance
    # at a grid of points, well inside the 1% critical value 1.63 / sqrt(n))
    nd = statistics.NormalDist()
    xs = torch.sort(x).values
    n = xs.numel()
    for z in (-3.0, -2.0, -1.0, -0.5, 0.0, 0.5, 1.0, 2.0, 3.0):
        emp = torch.searchsorted(xs, torch.tensor(z, dtype=torch.float64), right=True).item() / n
        assert abs(emp - nd.cdf(z)) < 1.63 / n ** 0.5, z
    # the tails reach past 4 sigma (a bounded stand-in would not)
    assert xs[0].item() < -4.0 and xs[-1].item() > 4.0
    # every value is one of the 2^16 midpoint quantiles, exact in float32
    lv = torch.tensor([nd.inv_cdf((i + 0.5) / 65536) for i in (0, 32767, 32768, 65535)], dtype=torch.float64)
    assert torch.isin(lv.float(), wl.hash_normal(0, 1, torch.arange(1 << 21, dtype=torch.int64))).sum() == 4


def test_lengths_and_pools():
    w = wl.gqa_decode(0)
    assert len(w.lengths) == 64 and min(w.lengths) >= 512 and max(w.lengths) <= 4096
    need = sum(-(-L // 16) for L in w.lengths)
    assert w.num_pages == int(np.ceil(need * 1.1))
    assert sorted(w.free_order) == list(range(w.num_pages))
    lb = wl.large_batch(0, P=1)
    assert len(lb.lengths) == 256 and max(lb.lengths) <= 16384 - 256
    assert 700 < float(np.median(lb.lengths)) < 1400
