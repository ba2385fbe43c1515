"""GPU parity of decoding beyond seq_len with a rolling KV cache.

With rolling_positions = N > seq_len = S, position p writes cache slot p % S
and attends over the last S positions; RoPE keeps the absolute position. The
oracle (rolling_cache = 1) gathers the window in position order; the GPU sums
over the cache slots in slot order (attention does not depend on the order).
Bar as for decode: logits within relative L2 1e-4 under teacher forcing, and
free-running tokens equal up to the first near-tie.
"""
import numpy as np
import pytest

import oracle
import synth
from parity_util import REL_L2_TOL, config, first_near_tie, oracle_run, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def l2():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import llama_fp32_token_decode_b300 as m
    return m


SHAPES = {
    "s16_gqa": config(dim=128, hidden_dim=344, n_layers=2, n_heads=8, n_kv_heads=2,
                      vocab_size=3001, seq_len=16, rolling_positions=64, rolling_cache=1),
    "s24_hd48": config(dim=288, hidden_dim=768, n_layers=2, n_heads=6, vocab_size=2000,
                       seq_len=24, rolling_positions=80, rolling_cache=1),
    "s32_hd64": config(dim=256, hidden_dim=512, n_layers=1, n_heads=4, vocab_size=1000,
                       seq_len=32, rolling_positions=100, rolling_cache=1),
}


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_rolling_cache_teacher_forced_and_free_running(l2, name):
    cfg = SHAPES[name]
    blob = synth.make_blob(cfg, 19, std=0.05)
    prompt = synth.prompt_ids(9, 6, cfg["vocab_size"])
    steps = cfg["rolling_positions"] - len(prompt) + 1
    toks, consumed, trace = oracle_run(cfg, blob, prompt, steps)
    assert trace.shape[0] == cfg["rolling_positions"] > 3 * cfg["seq_len"] - 1
    with l2.Decoder(cfg, blob) as dec:
        for p, t in enumerate(consumed):
            lg = dec.forward([t], [p])[0]
            e = rel_l2(lg, trace[p])
            assert e <= REL_L2_TOL, f"pos {p} (slot {p % cfg['seq_len']}): rel-L2 {e:.3e}"
        gen = dec.generate(prompt, steps)
    k = first_near_tie(trace, len(prompt))
    n = min(k + 1, steps)
    np.testing.assert_array_equal(gen[:n], toks[:n])
    assert n > cfg["seq_len"] or k < steps  # compared past the wrap unless a near-tie came first


def test_rolling_cache_limits_and_sampling(l2):
    cfg = SHAPES["s16_gqa"]
    blob = synth.make_blob(cfg, 5, std=0.3)
    prompt = synth.prompt_ids(2, 4, cfg["vocab_size"])
    N = cfg["rolling_positions"]
    with l2.Decoder(cfg, blob) as dec:
        with pytest.raises(l2.L2Error):
            dec.forward([1], [N])                          # past rolling_positions
        with pytest.raises(l2.L2Error):
            dec.generate(prompt, N - len(prompt) + 2)      # one position too many
        # sampling past seq_len against the oracle's sampled generation
        steps = N - len(prompt) + 1
        u = np.random.default_rng(4).random(steps).astype(np.float32)
        gpu = dec.generate_sample(prompt, steps, 0.8, 0.9, u)
    ref, margins = oracle.Model(cfg, blob).generate_sampled(prompt, steps, 0.8, 0.9, u)
    n = 0
    for k in range(steps):
        if gpu[k] != ref[k]:
            assert margins[k] <= 1e-4, f"draw {k} differs with margin {margins[k]:.2e}"
            break
        n += 1
    assert n >= 10
    plain = dict(cfg, rolling_positions=0)
    with l2.Decoder(plain, blob) as dec:
        with pytest.raises(l2.L2Error):
            dec.forward([1], [cfg["seq_len"]])             # no rolling: S is the limit


def test_rolling_cache_batched(l2):
    # three sequences in lockstep on the tensor-core path, each running past
    # the window (3 S positions): teacher-forced logits at every position, then
    # free-running generation compared per sequence up to its first near-tie
    cfg = dict(SHAPES["s16_gqa"], max_batch=3, rolling_positions=48)
    blob = synth.make_blob(cfg, 19, std=0.05)
    S, N = cfg["seq_len"], cfg["rolling_positions"]
    lens = np.array([1, 4, 6], np.int32)
    prompts = [synth.prompt_ids(30 + b, int(lens[b]), cfg["vocab_size"]) for b in range(3)]
    steps = N - int(lens.max()) + 1
    runs = [oracle_run(cfg, blob, prompts[b], steps) for b in range(3)]
    with l2.Decoder(cfg, blob) as dec:
        n_common = int(lens.min()) + steps - 1  # positions every sequence runs
        assert n_common > 2 * S
        for p in range(n_common):  # every sequence at position p (consumed tokens of its run)
            toks = [int(runs[b][1][p]) for b in range(3)]
            lg = dec.forward(toks, [p] * 3)
            for b in range(3):
                e = rel_l2(lg[b], runs[b][2][p])
                assert e <= REL_L2_TOL, f"seq {b} pos {p} (slot {p % S}): rel-L2 {e:.3e}"
        gen = dec.generate_batch(np.concatenate(prompts), lens, steps)
    for b in range(3):
        toks, _, trace = runs[b]
        k = first_near_tie(trace, int(lens[b]))
        n = min(k + 1, steps)
        np.testing.assert_array_equal(gen[b][:n], toks[:n])
