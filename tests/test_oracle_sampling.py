"""Pins of the oracle's sampler (oracle_sample): closed forms, the nucleus
rule, the inversion order, edges and the empirical distribution.

Reading pinned here (the pages show sampled stories but give no rule):
p_i = exp((l_i - max) / T); top-p keeps the smallest set of highest p whose
mass reaches topp * total, widened to ties of the last one taken; the draw
u in [0, 1) picks the first kept token, in index order, whose running sum of
p exceeds u times the kept mass. T <= 0 is the greedy choice.
"""
import math

import numpy as np

import oracle


def test_temperature_zero_is_greedy_with_lowest_index_on_ties():
    assert oracle.sample([0.1, 0.7, 0.7, 0.2], 0.0, 1.0, 0.99)[0] == 1
    assert oracle.sample([3.0, -1.0], -1.0, 0.5, 0.0)[0] == 0


def test_two_tokens_closed_form():
    # p = [1, 3] / 4: tokens split the unit interval at 1/4
    lg = [0.0, math.log(3.0)]
    assert oracle.sample(lg, 1.0, 1.0, 0.20)[0] == 0
    assert oracle.sample(lg, 1.0, 1.0, 0.30)[0] == 1
    t, margin = oracle.sample(lg, 1.0, 1.0, 0.20)
    assert abs(margin - 0.05) < 1e-6


def test_temperature_divides_the_logits():
    lg = [0.0, math.log(3.0)]
    # T = 0.5: p proportional to [1, 9], boundary at 0.1
    assert oracle.sample(lg, 0.5, 1.0, 0.09)[0] == 0
    assert oracle.sample(lg, 0.5, 1.0, 0.11)[0] == 1
    # T = 2: p proportional to [1, sqrt(3)], boundary at 1 / (1 + sqrt 3) = 0.366
    assert oracle.sample(lg, 2.0, 1.0, 0.36)[0] == 0
    assert oracle.sample(lg, 2.0, 1.0, 0.37)[0] == 1


def test_nucleus_cut():
    lg = np.log([0.5, 0.3, 0.2])
    # top-p 0.7: 0.5 < 0.7 <= 0.8, nucleus {0, 1} of mass 0.8
    assert oracle.sample(lg, 1.0, 0.7, 0.60)[0] == 0          # r = 0.48 < 0.5
    assert oracle.sample(lg, 1.0, 0.7, 0.65)[0] == 1          # r = 0.52
    assert oracle.sample(lg, 1.0, 0.7, 0.999)[0] == 1         # token 2 never drawn
    # top-p 0.5: the single top token already reaches it
    assert all(oracle.sample(lg, 1.0, 0.5, u)[0] == 0 for u in (0.0, 0.5, 0.999))
    # top-p 0.81 > 0.8: every token
    assert oracle.sample(lg, 1.0, 0.81, 0.95)[0] == 2


def test_nucleus_inverted_in_index_order_not_rank_order():
    # nucleus {1 (0.5), 0 (0.3)}: index order puts token 0 first
    lg = np.log([0.3, 0.5, 0.2])
    assert oracle.sample(lg, 1.0, 0.7, 0.2)[0] == 0           # r = 0.16 < 0.3
    assert oracle.sample(lg, 1.0, 0.7, 0.5)[0] == 1           # r = 0.40 > 0.3


def test_ties_at_the_nucleus_edge_are_kept():
    lg = np.log([0.4, 0.3, 0.3])
    # 0.4 + 0.3 reaches 0.6 at token 1; token 2 ties with it and is kept
    assert oracle.sample(lg, 1.0, 0.6, 0.95)[0] == 2


def test_u_close_to_one_takes_the_last_member():
    lg = np.log([0.25, 0.25, 0.5])
    assert oracle.sample(lg, 1.0, 1.0, 0.9999999)[0] == 2


def test_empirical_distribution_matches_softmax():
    rng = np.random.default_rng(0)
    lg = np.array([0.3, -1.2, 2.0, 0.0, 1.1], np.float32)
    T, n = 0.8, 20000
    p = np.exp((lg - lg.max()) / T)
    p /= p.sum()
    counts = np.bincount([oracle.sample(lg, T, 1.0, float(u))[0] for u in rng.random(n)],
                         minlength=5)
    sigma = np.sqrt(n * p * (1 - p))
    assert np.all(np.abs(counts - n * p) < 5 * sigma + 1), (counts, n * p)
    # top-p 0.8: the nucleus and its renormalised distribution
    order = np.argsort(-p, kind="stable")
    k = int(np.searchsorted(np.cumsum(p[order]), 0.8)) + 1
    keep = np.zeros(5, bool)
    keep[order[:k]] = True
    q = np.where(keep, p, 0.0) / p[keep].sum()
    counts = np.bincount([oracle.sample(lg, T, 0.8, float(u))[0] for u in rng.random(n)],
                         minlength=5)
    assert np.all(counts[~keep] == 0)
    sigma = np.sqrt(n * q * (1 - q))
    assert np.all(np.abs(counts - n * q) < 5 * sigma + 1), (counts, n * q)


def test_generate_sampled_draws_one_uniform_per_token():
    from parity_util import config
    import synth
    cfg = config(dim=32, hidden_dim=64, n_layers=1, n_heads=2, vocab_size=50, seq_len=12)
    blob = synth.make_blob(cfg, 3, std=0.3)
    m = oracle.Model(cfg, blob)
    prompt = np.array([1, 2, 3], np.int32)
    u = np.random.default_rng(1).random(8).astype(np.float32)
    toks, margins = m.generate_sampled(prompt, 8, 0.9, 0.95, u)
    # replaying the draws on the oracle's own logits gives the same tokens
    consumed = np.concatenate([prompt, toks[:-1]])
    m2 = oracle.Model(cfg, blob)
    for p, t in enumerate(consumed):
        lg = m2.forward(int(t), p)
        if p >= len(prompt) - 1:
            k = p - (len(prompt) - 1)
            assert oracle.sample(lg, 0.9, 0.95, float(u[k]))[0] == toks[k]
    assert np.all(margins >= 0)
    # temperature 0 reproduces greedy generation
    g, _ = m.generate_sampled(prompt, 8, 0.0, 1.0, u)
    np.testing.assert_array_equal(g, oracle.Model(cfg, blob).generate(prompt, 8))
