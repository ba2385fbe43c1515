"""Pins for the seeded input generator (synth/), which both sides read."""
import math

import numpy as np

import synth

G = 0x9E3779B97F4A7C15
M64 = (1 << 64) - 1


def test_splitmix64_published_outputs():
    # SplitMix64 seeded with 0 emits mix64(k * G) for k = 1, 2, 3; these are
    # the widely published first three outputs of that generator.
    assert synth.mix64(G) == 0xE220A8397B1DCDAF
    assert synth.mix64((2 * G) & M64) == 0x6E789E6AA1B965F4
    assert synth.mix64((3 * G) & M64) == 0x06C45D188009454F


def test_uniform_open_interval_and_moments():
    u = np.array([synth.uniform(7, 1, k) for k in range(20000)])
    assert u.min() > 0.0 and u.max() < 1.0
    assert abs(u.mean() - 0.5) < 0.01
    assert abs(u.var() - 1.0 / 12.0) < 0.003


def test_box_muller_pair_identity():
    # For a Box-Muller pair, z0^2 + z1^2 = -2 ln u1 and atan2(z1, z0) = 2 pi u2.
    for j in range(50):
        z0 = synth.normal(3, 9, 2 * j)
        z1 = synth.normal(3, 9, 2 * j + 1)
        u1 = synth.uniform(3, 9, 2 * j)
        u2 = synth.uniform(3, 9, 2 * j + 1)
        assert math.isclose(z0 * z0 + z1 * z1, -2.0 * math.log(u1), rel_tol=1e-12)
        ang = math.atan2(z1, z0) % (2 * math.pi)
        assert math.isclose(ang, 2 * math.pi * u2, rel_tol=1e-9, abs_tol=1e-9)


def test_fill_matches_elementwise_and_is_counter_based():
    n = 1001
    out = np.empty(n, np.float32)
    lib = synth._lib()
    lib.synth_fill_normal(5, 2, 17, n, 0.02, out.ctypes.data, 4)
    ref = np.array([np.float32(0.02 * synth.normal(5, 2, 17 + i)) for i in range(n)], np.float32)
    assert np.array_equal(out, ref)
    # a slice drawn alone equals the same slice of a longer draw (odd offset)
    part = np.empty(100, np.float32)
    lib.synth_fill_normal(5, 2, 17 + 333, 100, 0.02, part.ctypes.data, 1)
    assert np.array_equal(part, out[333:433])


def test_normal_moments():
    out = np.empty(1 << 20, np.float32)
    synth._lib().synth_fill_normal(11, 4, 0, out.size, 1.0, out.ctypes.data, 8)
    assert abs(out.mean()) < 0.005
    assert abs(out.std() - 1.0) < 0.005
    # fourth moment of a standard normal is 3
    assert abs(np.mean(out.astype(np.float64) ** 4) - 3.0) < 0.05


def test_blob_layout_gains_and_size():
    cfg = dict(dim=16, hidden_dim=24, n_layers=2, n_heads=4, n_kv_heads=2, vocab_size=10,
               seq_len=8, shared_classifier=0)
    b = synth.make_blob(cfg, 1)
    d, F, L, V, kvd = 16, 24, 2, 10, 8
    assert b.size == V * d + L * d + L * d * d + 2 * L * kvd * d + L * d * d + L * d \
        + 3 * L * F * d + d + V * d
    off = 0
    for name, n, gain in synth.blob_segments(cfg):
        seg = b[off:off + n]
        if gain:
            assert np.all(seg == 1.0), name
        else:
            assert not np.any(seg == 1.0), name
        off += n
    tied = dict(cfg, shared_classifier=1)
    assert synth.blob_floats(tied) == b.size - V * d


def test_prompt_ids_range_and_determinism():
    p = synth.prompt_ids(1, 5000, 32000)
    assert p.min() >= 3 and p.max() < 32000
    assert np.array_equal(p, synth.prompt_ids(1, 5000, 32000))
    assert not np.array_equal(p, synth.prompt_ids(2, 5000, 32000))
    lens = synth.batch_lengths(4, 256, 1, 128)
    assert lens.min() >= 1 and lens.max() <= 128
    w = synth.workload("batched")
    lens2, prompts = synth.batch_inputs(w)
    assert np.array_equal(lens, lens2) and prompts.size == lens.sum()
