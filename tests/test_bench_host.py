"""Host-side arithmetic of bench.py (no GPU): the batched run's lower bound
against a step-by-step, sequence-by-sequence count on a tiny workload."""
import numpy as np

import bench


def test_batched_run_bound_matches_explicit_count():
    cfg = dict(dim=8, hidden_dim=12, n_layers=2, n_heads=2, n_kv_heads=1, vocab_size=10)
    lens = np.array([1, 3, 2])
    steps, B, hbm, p3 = 4, 3, 2.0, 1e-9  # GB/s and TFLOP/s chosen so both terms matter
    d, F, L, V, kvd = 8, 12, 2, 10, 4
    weights = 4.0 * (L * (2 * d * d + 2 * d * kvd + 3 * d * F + 2 * d) + d + V * d + B * d)
    flops = 2.0 * B * (L * (d * (d + 2 * kvd) + d * d + 3 * d * F) + V * d)
    total = 0.0
    n_lock = max(lens) + steps - 1
    for t in range(n_lock):
        total += max(weights / (hbm * 1e9), flops / (p3 * 1e12))
        for b in range(B):
            if t < lens[b] + steps - 1:  # sequence b still decoding at step t
                total += 4.0 * L * 2 * kvd * ((t + 1) + 1) / (hbm * 1e9)
    got, gemm = bench.batched_run_bound(cfg, lens, steps, B, hbm, p3)
    assert np.isclose(got, total, rtol=1e-12)
    assert np.isclose(gemm, n_lock * max(weights / (hbm * 1e9), flops / (p3 * 1e12)))
