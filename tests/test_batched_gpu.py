"""GPU parity of batched decode (the 3xTF32 tensor-core path) against the C oracle.

B independent sequences, each with its own prompt, position and KV cache, are
decoded in lockstep. The oracle has no batch: every sequence is checked
against its own single-sequence oracle run. Protocol as for batch 1: teacher
forcing with per-step logits within relative L2 error 1e-4 and greedy tokens
equal wherever the oracle's top-2 gap exceeds 1e-3; free-running generation
equal to the oracle up to each sequence's first near-tie.
"""
import numpy as np
import pytest

import synth
from parity_util import (GAP_TOL, REL_L2_TOL, config, first_near_tie, oracle_run, rel_l2,
                         top2_gap)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def l2():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import llama_fp32_token_decode_b300 as m
    return m


def _sequences(cfg, B, seed, steps):
    lens = 1 + (np.arange(B) * 7 + seed) % 6
    runs = []
    for b in range(B):
        prompt = synth.prompt_ids(seed * 1000 + b, int(lens[b]), cfg["vocab_size"])
        runs.append(oracle_run(cfg, _BLOBS[(id(cfg), seed)], prompt, steps))
    return lens, runs


_BLOBS = {}


def _blob(cfg, seed):
    key = (id(cfg), seed)
    if key not in _BLOBS:
        _BLOBS[key] = synth.make_blob(cfg, seed, std=0.05)
    return _BLOBS[key]


BATCHED = {
    "b5": (config(dim=64, hidden_dim=160, n_layers=2, n_heads=4, vocab_size=1000, seq_len=24,
                  max_batch=5), 5),
    "b130_gqa": (config(dim=128, hidden_dim=344, n_layers=2, n_heads=8, n_kv_heads=2,
                        vocab_size=3001, seq_len=20, max_batch=130), 130),
    "b256_hd48_tied": (config(dim=288, hidden_dim=768, n_layers=1, n_heads=6, vocab_size=517,
                              seq_len=12, max_batch=256, shared_classifier=1), 256),
    # at most 64 rows with K of 4096: drained launches that split fp32
    # weights in shared memory (M = 64 MMAs), head_dim 128, GQA
    "b6_wide_drained": (config(dim=4096, hidden_dim=4096, n_layers=1, n_heads=32, n_kv_heads=8,
                               vocab_size=600, seq_len=12, max_batch=6), 6),
}


@pytest.mark.parametrize("name", sorted(BATCHED))
def test_batched_forward_teacher_forced_ragged_positions(l2, name):
    cfg, B = BATCHED[name]
    blob = _blob(cfg, 17)
    steps = cfg["seq_len"] - 6
    lens, runs = _sequences(cfg, B, 17, steps)
    n_fwd = [len(r[1]) for r in runs]
    offs = np.arange(B) % 4          # sequence b starts off_b calls late (pos 0 re-run)
    T = max(n + o for n, o in zip(n_fwd, offs))
    worst = 0.0
    with l2.Decoder(cfg, blob) as dec:
        for t in range(T):
            pos = np.array([min(max(t - offs[b], 0), n_fwd[b] - 1) for b in range(B)], np.int32)
            toks = np.array([runs[b][1][pos[b]] for b in range(B)], np.int32)
            lg = dec.forward(toks, pos)
            assert lg.shape == (B, cfg["vocab_size"])
            for b in range(B):
                ref = runs[b][2][pos[b]]
                e = rel_l2(lg[b], ref)
                worst = max(worst, e)
                assert e <= REL_L2_TOL, f"call {t} seq {b} pos {pos[b]}: rel-L2 {e:.3e}"
                if top2_gap(ref) > GAP_TOL:
                    assert int(np.argmax(lg[b])) == int(np.argmax(ref)), (t, b)
    print(f"{name}: worst rel-L2 {worst:.2e}")


@pytest.mark.parametrize("name", sorted(BATCHED))
def test_batched_generation_free_running(l2, name):
    cfg, B = BATCHED[name]
    blob = _blob(cfg, 23)
    steps = cfg["seq_len"] - 6
    lens, runs = _sequences(cfg, B, 23, steps)
    prompts = np.concatenate([r[1][:lens[b]] for b, r in enumerate(runs)])
    with l2.Decoder(cfg, blob) as dec:
        out = dec.generate_batch(prompts, lens, steps)
        again = dec.generate_batch(prompts, lens, steps)
    np.testing.assert_array_equal(out, again)
    assert out.shape == (B, steps)
    for b in range(B):
        toks, _, trace = runs[b]
        k = first_near_tie(trace, int(lens[b]))
        n = min(k + 1, steps)
        np.testing.assert_array_equal(out[b, :n], toks[:n], err_msg=f"sequence {b}")


def test_batched_matches_batch1_path_on_one_sequence(l2):
    # the GEMM path (B = 2, second row a copy) and the matvec path agree with each other
    cfg = config(dim=128, hidden_dim=344, n_layers=2, n_heads=4, vocab_size=2000, seq_len=16,
                 max_batch=4)
    blob = synth.make_blob(cfg, 3, std=0.05)
    prompt = synth.prompt_ids(5, 4, cfg["vocab_size"])
    toks, consumed, trace = oracle_run(cfg, blob, prompt, 8)
    with l2.Decoder(cfg, blob) as dec:
        single = dec.generate(prompt, 8)
        batch = dec.generate_batch(np.concatenate([prompt, prompt]), [4, 4], 8)
    np.testing.assert_array_equal(batch[0], batch[1])
    k = first_near_tie(trace, 4)
    np.testing.assert_array_equal(batch[0][:k + 1], single[:k + 1])


def test_batched_argument_errors(l2):
    cfg, B = BATCHED["b5"]
    blob = _blob(cfg, 17)
    with l2.Decoder(cfg, blob) as dec:
        S = cfg["seq_len"]
        with pytest.raises(l2.L2Error):
            dec.generate_batch([1] * 6, [1] * 6, 2)               # B > max_batch
        with pytest.raises(l2.L2Error):
            dec.generate_batch([1, 2], [1, 1], S + 1)             # too long
        with pytest.raises(l2.L2Error):
            dec.generate_batch([1, 2], [0, 2], 2)                 # empty prompt
        with pytest.raises(l2.L2Error):
            dec.generate_batch([1, cfg["vocab_size"]], [1, 1], 2)  # id out of range
        with pytest.raises(l2.L2Error):
            dec.forward([1, 2], [0, S])                           # position out of range
        # a valid call still works afterwards
        assert dec.generate_batch([1, 2], [1, 1], 3).shape == (2, 3)
