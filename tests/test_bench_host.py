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


def test_batched_attention_traffic_scales_and_follows_the_kernel(monkeypatch):
    # the committed capture's DRAM bytes were taken at 301 positions; at any
    # other position they scale with the algorithmic bytes, and they are
    # withdrawn (None) when the kernel's source text no longer matches
    vals = bench.summary_values(bench.BATTN_PROFILE)
    ratio = float(vals["dram bytes per launch (read + write)"]) / float(
        vals["algorithmic bytes per launch"])
    assert 1.0 <= ratio < 1.05  # every K and V row read once
    if vals["battn4_kernel source sha256"] == bench.kernel_text_sha256(bench.BATTN_SOURCE,
                                                                       bench.BATTN_HEAD):
        alg = 4.0 * 256 * (2 * 321 * 512 + 2 * 512)
        assert np.isclose(bench.profiled_battn_traffic(alg), ratio * alg)
    monkeypatch.setattr(bench, "BATTN_HEAD", "no such kernel head")
    assert bench.profiled_battn_traffic(1e8) is None


def test_kernel_text_hash_ignores_the_rest_of_the_file(tmp_path):
    head = "template <int A>\n__global__ void"
    body = head + " k() {\n    x();\n}\n"
    a, b, c = tmp_path / "a.cu", tmp_path / "b.cu", tmp_path / "c.cu"
    a.write_text("// one\n" + body + "void other() {}\n")
    b.write_text("// two\nint y;\n" + body)
    c.write_text("// one\n" + body.replace("x()", "z()"))
    ha = bench.kernel_text_sha256(str(a), head)
    assert ha is not None and ha == bench.kernel_text_sha256(str(b), head)
    assert ha != bench.kernel_text_sha256(str(c), head)


def test_clock_records_that_reject_a_timed_region():
    ok = {"sm_mhz": 2032.0, "sm_max_mhz": 2032.0, "reasons": []}
    assert not bench.clocks_rejected(ok)
    assert not bench.clocks_rejected(None)  # no sampler: nothing to judge
    assert not bench.clocks_rejected(dict(ok, sm_mhz=1500.0, reasons=["sw_power_cap"]))
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert bench.clocks_rejected(dict(ok, reasons=[r]))
    assert bench.clocks_rejected(dict(ok, sm_mhz=1200.0))  # held low with no reason
    assert not bench.clocks_rejected(dict(ok, sm_mhz=1900.0))
