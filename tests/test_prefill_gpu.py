"""GPU parity of the parallel prompt prefill (one causal tensor-core pass over a
prompt) against the C oracle, which feeds the prompt one token per forward.

Every position's logits must match the oracle's teacher-forced trace within
relative L2 1e-4 (the same bar as decode), greedy tokens must agree where the
oracle's top-2 gap exceeds 1e-3, and generation with a prefilled prompt must
reproduce the oracle's tokens up to the first near-tie.
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


SHAPES = {
    "small": config(dim=64, hidden_dim=160, n_layers=2, n_heads=4, vocab_size=1000, seq_len=40,
                    max_prefill=32),
    "gqa_ragged_vocab": config(dim=128, hidden_dim=344, n_layers=2, n_heads=8, n_kv_heads=2,
                               vocab_size=3001, seq_len=48, max_prefill=40),
    "hd48_tied": config(dim=288, hidden_dim=768, n_layers=2, n_heads=6, vocab_size=517,
                        seq_len=160, max_prefill=150, shared_classifier=1),
    "hd128": config(dim=512, hidden_dim=1024, n_layers=1, n_heads=4, vocab_size=2000,
                    seq_len=32, max_prefill=20),
}


def _check_rows(lg, trace, positions):
    for i, p in enumerate(positions):
        e = rel_l2(lg[i], trace[p])
        assert e <= REL_L2_TOL, f"pos {p}: rel-L2 {e:.3e}"
        if top2_gap(trace[p]) > GAP_TOL:
            assert int(np.argmax(lg[i])) == int(np.argmax(trace[p])), f"pos {p}: argmax"


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_prefill_logits_every_position(l2, name):
    cfg = SHAPES[name]
    blob = synth.make_blob(cfg, 13, std=0.05)
    n = cfg["max_prefill"]
    prompt = synth.prompt_ids(21, n, cfg["vocab_size"])
    _, consumed, trace = oracle_run(cfg, blob, prompt, cfg["seq_len"] - n + 1)
    with l2.Decoder(cfg, blob) as dec:
        lg = dec.prefill(prompt)
        assert lg.shape == (n, cfg["vocab_size"])
        _check_rows(lg, trace, range(n))
        # continuing the same sequence: a second prefill at pos0 > 0 over the
        # oracle's next consumed tokens, then a decode forward after it
        k = min(6, cfg["seq_len"] - n - 1)
        lg2 = dec.prefill(consumed[n:n + k], pos0=n)
        _check_rows(lg2, trace, range(n, n + k))
        p = n + k
        one = dec.forward([consumed[p]], [p])[0]
        assert rel_l2(one, trace[p]) <= REL_L2_TOL


@pytest.mark.parametrize("name", ["small", "hd48_tied"])
def test_generate_with_prefill_matches_oracle(l2, name):
    cfg = SHAPES[name]
    blob = synth.make_blob(cfg, 29, std=0.05)
    n = cfg["max_prefill"] // 2
    prompt = synth.prompt_ids(5, n, cfg["vocab_size"])
    steps = cfg["seq_len"] - n + 1
    toks, _, trace = oracle_run(cfg, blob, prompt, steps)
    with l2.Decoder(cfg, blob) as dec:
        out = dec.generate_prefill(prompt, steps)
        ref = dec.generate(prompt, steps)
    k = first_near_tie(trace, n)
    np.testing.assert_array_equal(out[:k + 1], toks[:k + 1])
    np.testing.assert_array_equal(ref[:k + 1], toks[:k + 1])


def test_prefill_device_entry_point(l2):
    import torch
    cfg = SHAPES["gqa_ragged_vocab"]
    blob = synth.make_blob(cfg, 3, std=0.05)
    prompt = synth.prompt_ids(8, 30, cfg["vocab_size"])
    with l2.Decoder(cfg, blob) as dec:
        ref = dec.generate_prefill(prompt, 12)
        s = torch.cuda.Stream()
        d_prompt = torch.tensor(prompt, dtype=torch.int32, device="cuda")
        d_out = torch.zeros(12, dtype=torch.int32, device="cuda")
        l2.l2_generate_prefill_device(dec.h, d_prompt, len(prompt), 12, d_out, s)
        s.synchronize()
        np.testing.assert_array_equal(d_out.cpu().numpy(), ref)
        # prompt-only generation: steps = 1 is the prefill alone
        one = dec.generate_prefill(prompt, 1)
        assert one[0] == ref[0]


def test_prefill_errors(l2):
    cfg = SHAPES["small"]
    blob = synth.make_blob(cfg, 4, std=0.05)
    with l2.Decoder(cfg, blob) as dec:
        with pytest.raises(l2.L2Error):
            dec.prefill(np.ones(cfg["max_prefill"] + 1, np.int32))      # over capacity
        with pytest.raises(l2.L2Error):
            dec.prefill([1, 2, 3], pos0=cfg["seq_len"] - 2)                # past the cache
        with pytest.raises(l2.L2Error):
            dec.prefill([cfg["vocab_size"]])                              # bad id
        with pytest.raises(l2.L2Error):
            dec.generate_prefill([1] * 4, cfg["seq_len"])                  # too long
        assert dec.prefill([1, 2]).shape == (2, cfg["vocab_size"])
    plain = dict(cfg, max_prefill=0)
    with l2.Decoder(plain, blob) as dec:
        with pytest.raises(l2.L2Error):
            dec.prefill([1, 2])                                            # no prefill path


@pytest.mark.parametrize("max_prefill", [0, 7])
def test_batched_generation_with_prefill(l2, max_prefill):
    # five ragged prompts taken by prefill passes (max_prefill 7 with
    # max_batch 5: passes of 7 rows, so sequences straddle passes), then
    # lockstep generation; each sequence against the oracle up to its first
    # near-tie, and against the lockstep generation without prefill
    import torch
    cfg = config(dim=128, hidden_dim=344, n_layers=2, n_heads=8, n_kv_heads=2, vocab_size=3001,
                 seq_len=40, max_batch=5, max_prefill=max_prefill)
    blob = synth.make_blob(cfg, 21, std=0.05)
    lens = np.array([3, 1, 9, 5, 6], np.int32)
    prompts = [synth.prompt_ids(60 + b, int(lens[b]), cfg["vocab_size"]) for b in range(5)]
    flat = np.concatenate(prompts).astype(np.int32)
    steps = 20
    with l2.Decoder(cfg, blob) as dec:
        gen = dec.generate_batch_prefill(flat, lens, steps)
        lock = dec.generate_batch(flat, lens, steps)
        one = dec.generate_batch_prefill(flat, lens, 1)
        s = torch.cuda.Stream()
        d_p = torch.tensor(flat, device="cuda")
        d_o = torch.zeros((5, steps), dtype=torch.int32, device="cuda")
        l2.l2_generate_batch_prefill_device(dec.h, d_p, lens, steps, d_o, s)
        s.synchronize()
        np.testing.assert_array_equal(d_o.cpu().numpy(), gen)
        with pytest.raises(l2.L2Error):
            dec.generate_batch_prefill(flat, np.array([3, 1, 41, 5, 6], np.int32), steps)
    for b in range(5):
        toks, _, trace = oracle_run(cfg, blob, prompts[b], steps)
        k = first_near_tie(trace, int(lens[b]))
        n = min(k + 1, steps)
        np.testing.assert_array_equal(gen[b][:n], toks[:n])
        np.testing.assert_array_equal(lock[b][:n], toks[:n])
        assert one[b][0] == gen[b][0]
