"""Pins for the oracle's building blocks: closed forms, invariants and special
cases fixed by the mathematics of the Llama-2 decode step (RMSNorm, RoPE,
causal softmax attention, SwiGLU, greedy choice). None of these retypes the
oracle's code: each checks a value or a law that a wrong sign, index, term or
operand order would break."""
import math

import numpy as np
import pytest

import oracle

rng = np.random.default_rng(1234)


# ---------------------------------------------------------------- RMSNorm

def test_rmsnorm_unit_rms_when_eps_zero():
    x = rng.normal(0, 3.0, 4096).astype(np.float32)
    out = oracle.rmsnorm(x, np.ones_like(x), eps=0.0)
    assert abs(np.sqrt(np.mean(out.astype(np.float64) ** 2)) - 1.0) < 1e-6


def test_rmsnorm_rms_below_one_by_eps():
    # RMS of the output is sqrt(m / (m + eps)) with m = mean(x^2)
    x = np.full(64, 0.01, np.float32)  # m = 1e-4, eps = 1e-5
    out = oracle.rmsnorm(x, np.ones_like(x), eps=1e-5)
    assert math.isclose(float(out[0]), math.sqrt(1e-4 / 1.1e-4), rel_tol=1e-6)


def test_rmsnorm_eps_inside_root():
    # x = (1e-3, 0, 0, 0): mean(x^2) = 2.5e-7, so out0 = 1e-3 / sqrt(2.5e-7 + 1e-5)
    # = 0.3123475...; with eps added outside the root it would be 1.96.
    x = np.array([1e-3, 0, 0, 0], np.float32)
    out = oracle.rmsnorm(x, np.ones(4, np.float32), eps=1e-5)
    assert math.isclose(float(out[0]), 0.31234752377721214, rel_tol=1e-6)
    assert out[1] == 0.0


def test_rmsnorm_scale_invariance_and_gain():
    x = rng.normal(0, 1, 288).astype(np.float32)
    g = rng.uniform(0.5, 2.0, 288).astype(np.float32)
    a = oracle.rmsnorm(x, np.ones_like(x), eps=0.0)
    b = oracle.rmsnorm(np.float32(37.0) * x, np.ones_like(x), eps=0.0)
    np.testing.assert_allclose(a, b, rtol=2e-6, atol=1e-7)
    np.testing.assert_allclose(oracle.rmsnorm(x, g, eps=0.0), g * a, rtol=2e-6, atol=1e-7)


def test_rmsnorm_mean_over_n():
    # 3-4-0-0 with eps 0: mean(x^2) = 25/4, so the root is 2.5 and out = (1.2, 1.6, 0, 0)
    out = oracle.rmsnorm(np.array([3, 4, 0, 0], np.float32), np.ones(4, np.float32), 0.0)
    np.testing.assert_allclose(out, [1.2, 1.6, 0, 0], rtol=1e-7)


# ---------------------------------------------------------------- matvec

def test_matvec_orientation_and_exact_integers():
    # y = W x with W [out][in]; a non-square integer matrix exposes a transpose
    W = np.array([[1, 2, 3], [4, 5, 6]], np.float32)
    x = np.array([1, 10, 100], np.float32)
    np.testing.assert_array_equal(oracle.matvec(W, x), [321, 654])
    P = np.eye(5, dtype=np.float32)[[2, 0, 4, 1, 3]]
    v = np.arange(5, dtype=np.float32)
    np.testing.assert_array_equal(oracle.matvec(P, v), [2, 0, 4, 1, 3])


# ---------------------------------------------------------------- softmax

def test_softmax_sums_to_one_and_shift_invariant():
    s = rng.normal(0, 5, 1000).astype(np.float32)
    p = oracle.softmax(s)
    assert abs(p.astype(np.float64).sum() - 1.0) < 1e-5
    np.testing.assert_allclose(oracle.softmax(s + np.float32(50.0)), p, rtol=1e-4, atol=1e-9)
    assert np.all(p > 0)
    assert np.argmax(p) == np.argmax(s)


def test_softmax_closed_forms():
    p = oracle.softmax(np.array([0.0, math.log(3.0)], np.float32))
    np.testing.assert_allclose(p, [0.25, 0.75], rtol=1e-6)
    p = oracle.softmax(np.array([0.0, 200.0, 0.0], np.float32))
    np.testing.assert_array_equal(p, [0.0, 1.0, 0.0])  # exp(-200) underflows
    p = oracle.softmax(np.array([1000.0, 1000.0], np.float32))  # needs max subtraction
    np.testing.assert_array_equal(p, [0.5, 0.5])


# ---------------------------------------------------------------- RoPE

def test_rope_identity_at_pos_zero():
    v = rng.normal(0, 1, 64).astype(np.float32)
    np.testing.assert_array_equal(oracle.rope(v, 2, 32, 0), v)


def test_rope_adjacent_pairs_and_frequencies():
    hd = 4
    # pair (0, 1) has frequency theta^0 = 1: at pos 1, (1, 0) turns by 1 rad
    out = oracle.rope(np.array([1, 0, 0, 0], np.float32), 1, hd, 1)
    np.testing.assert_allclose(out, [math.cos(1), math.sin(1), 0, 0], atol=1e-7)
    # pair (2, 3) has frequency 10000^(-2/4) = 0.01: at pos 100 it turns by 1 rad
    out = oracle.rope(np.array([0, 0, 1, 0], np.float32), 1, hd, 100)
    np.testing.assert_allclose(out, [0, 0, math.cos(1), math.sin(1)], atol=1e-7)
    # (0, 1) turns to (-sin, cos): counter-clockwise, as multiplying by e^{i angle}
    out = oracle.rope(np.array([0, 1, 0, 0], np.float32), 1, hd, 1)
    np.testing.assert_allclose(out, [-math.sin(1), math.cos(1), 0, 0], atol=1e-7)
    # every head uses the same table
    out = oracle.rope(np.array([0, 0, 0, 0, 1, 0, 0, 0], np.float32), 2, hd, 1)
    np.testing.assert_allclose(out[4:6], [math.cos(1), math.sin(1)], atol=1e-7)


def test_rope_preserves_pair_norms():
    v = rng.normal(0, 1, 128).astype(np.float32)
    out = oracle.rope(v, 1, 128, 1777)
    n_in = np.hypot(v[0::2].astype(np.float64), v[1::2])
    n_out = np.hypot(out[0::2].astype(np.float64), out[1::2])
    np.testing.assert_allclose(n_out, n_in, rtol=1e-6)


def test_rope_composition_and_relative_position():
    v = rng.normal(0, 1, 64).astype(np.float32)
    np.testing.assert_allclose(oracle.rope(oracle.rope(v, 1, 64, 5), 1, 64, 7),
                               oracle.rope(v, 1, 64, 12), rtol=1e-5, atol=1e-5)
    q = rng.normal(0, 1, 64).astype(np.float32)
    k = rng.normal(0, 1, 64).astype(np.float32)
    a = np.dot(oracle.rope(q, 1, 64, 9).astype(np.float64), oracle.rope(k, 1, 64, 4))
    b = np.dot(oracle.rope(q, 1, 64, 105).astype(np.float64), oracle.rope(k, 1, 64, 100))
    assert abs(a - b) < 1e-4 * (abs(a) + 1)


# ---------------------------------------------------------------- attention

def test_attention_single_position_returns_v_exactly():
    q = rng.normal(0, 1, 48).astype(np.float32)
    k = rng.normal(0, 1, (1, 48)).astype(np.float32)
    v = rng.normal(0, 1, (1, 48)).astype(np.float32)
    np.testing.assert_array_equal(oracle.attention_head(q, k, v), v[0])


def test_attention_equal_keys_give_mean_of_values():
    q = rng.normal(0, 1, 64).astype(np.float32)
    k = np.tile(rng.normal(0, 1, 64).astype(np.float32), (7, 1))
    v = rng.normal(0, 1, (7, 64)).astype(np.float32)
    np.testing.assert_allclose(oracle.attention_head(q, k, v), v.mean(0), rtol=1e-5, atol=1e-6)


def test_attention_scale_is_inverse_sqrt_head_dim():
    # q . k1 = sqrt(hd) ln 3 and q . k0 = 0, so the weights are 1/4 and 3/4
    hd = 16
    q = np.zeros(hd, np.float32)
    q[3] = 1.0
    k = np.zeros((2, hd), np.float32)
    k[1, 3] = math.sqrt(hd) * math.log(3.0)
    v = np.zeros((2, hd), np.float32)
    v[0, 0] = 1.0
    v[1, 1] = 1.0
    out = oracle.attention_head(q, k, v)
    np.testing.assert_allclose(out[:2], [0.25, 0.75], rtol=1e-6)


# ---------------------------------------------------------------- SwiGLU

def test_swiglu_gate_and_up_roles():
    # silu(1) * 2 = 2 / (1 + e^-1); swapping gate and up would give silu(2) * 1
    out = oracle.swiglu(np.array([1.0, 0.0, -30.0, 30.0], np.float32),
                        np.array([2.0, 5.0, 1.0, 1.0], np.float32))
    np.testing.assert_allclose(out[0], 2.0 / (1.0 + math.exp(-1.0)), rtol=1e-6)
    assert out[1] == 0.0
    assert abs(out[2]) < 1e-11  # silu(-30) ~ -30 e^-30
    np.testing.assert_allclose(out[3], 30.0, rtol=1e-12)


# ---------------------------------------------------------------- greedy

def test_argmax_planted_and_ties():
    v = rng.normal(0, 1, 32000).astype(np.float32)
    v[12345] = 10.0
    assert oracle.argmax(v) == 12345
    v[20000] = 10.0
    assert oracle.argmax(v) == 12345  # lowest index wins a tie
    v[7] = 10.0
    assert oracle.argmax(v) == 7
    assert oracle.argmax(np.full(5, -3.0, np.float32)) == 0


@pytest.mark.parametrize("n", [1, 2, 31999])
def test_argmax_last_and_first(n):
    v = np.zeros(n, np.float32)
    v[-1] = 1.0
    assert oracle.argmax(v) == n - 1
