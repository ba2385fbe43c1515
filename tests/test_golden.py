"""Stored fixtures under tests/golden/ (CPU).

page_model_shapes.txt: the model shapes the pages print; the synthetic
workloads must use them, and the parameter count of each shape (tied
classifier, as the pages' checkpoints) must match the pages' approximate
figure.
oracle_tiny.txt: the oracle's logits on a tiny seeded model, written by
make_oracle_tiny.py (seeded generator + oracle only): any change to the
oracle's arithmetic shows here first.
"""
import importlib.util
import os

import numpy as np

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_workloads_use_the_pages_model_shapes():
    workload = {"15M": "15m", "44M": "44m"}
    for name, dim, layers, heads, ctx, approx in _rows("page_model_shapes.txt"):
        w = synth.workload(workload[name])
        assert (w["dim"], w["n_layers"], w["n_heads"], w["seq_len"]) == (
            int(dim), int(layers), int(heads), int(ctx)), name
        d, F, L, V = w["dim"], w["hidden_dim"], w["n_layers"], w["vocab_size"]
        tied = V * d + L * (4 * d * d + 3 * d * F + 2 * d) + d
        assert abs(tied / float(approx) - 1.0) < 0.06, (name, tied)


def test_oracle_matches_stored_logits():
    spec = importlib.util.spec_from_file_location(
        "make_oracle_tiny", os.path.join(GOLDEN, "make_oracle_tiny.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    stored = np.array([[float(v) for v in r] for r in _rows("oracle_tiny.txt")])
    now = mod.compute()
    assert now.shape == stored.shape == (mod.POSITIONS, mod.CFG["vocab_size"])
    np.testing.assert_allclose(now, stored, rtol=1e-6, atol=1e-8)
