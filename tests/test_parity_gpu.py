"""GPU parity of the batch-1 decode path against the C oracle.

Protocol (tolerance stated by the task this library serves): the GPU consumes
the oracle's own token sequence (teacher forcing); per-step logits must agree
within relative L2 error 1e-4, and the greedy token must agree wherever the
oracle's top-2 logit gap exceeds 1e-3. The free-running GPU generation must
reproduce the oracle's tokens up to the first step whose gap is <= 1e-3.
"""
import numpy as np
import pytest

import synth
from parity_util import (GAP_TOL, check_teacher_forced, config, first_near_tie, oracle_run,
                         rel_l2)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def l2():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import llama_fp32_token_decode_b300 as m
    return m


def _free_running(dec, prompt, steps, oracle_tokens, trace):
    gpu = dec.generate(prompt, steps)
    k = first_near_tie(trace, len(prompt))
    np.testing.assert_array_equal(gpu[:k + 1] if k < steps else gpu, oracle_tokens[:k + 1]
                                  if k < steps else oracle_tokens)
    return gpu


# Shapes chosen to cover every kernel plan: rows per ring stage >= 8 (small K),
# 1/2/4 rows per stage, rows split into chunks (K > 8192), row counts that do
# not divide the SM count, grouped kv heads, head_dim 12/48/64/128, a tied
# classifier, and a vocabulary with a ragged tail.
SHAPES = {
    "tiny_ragged": config(dim=72, hidden_dim=200, n_layers=2, n_heads=6, vocab_size=1001,
                          seq_len=24),
    "gqa": config(dim=128, hidden_dim=344, n_layers=3, n_heads=8, n_kv_heads=2, vocab_size=3000,
                  seq_len=40),
    "mqa_tied": config(dim=256, hidden_dim=688, n_layers=2, n_heads=4, n_kv_heads=1,
                       vocab_size=517, seq_len=20, shared_classifier=1),
    "wide_k": config(dim=2048, hidden_dim=8200, n_layers=1, n_heads=16, vocab_size=4099,
                     seq_len=12),
    "k4096": config(dim=4096, hidden_dim=256, n_layers=1, n_heads=32, vocab_size=300,
                    seq_len=8),
    "hd48": config(dim=288, hidden_dim=768, n_layers=2, n_heads=6, vocab_size=2000, seq_len=30),
}


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_small_shapes_teacher_forced_and_free_running(l2, name):
    cfg = SHAPES[name]
    blob = synth.make_blob(cfg, 11, std=0.05)
    prompt = synth.prompt_ids(3, 5, cfg["vocab_size"])
    steps = cfg["seq_len"] - len(prompt) + 1
    toks, consumed, trace = oracle_run(cfg, blob, prompt, steps)
    with l2.Decoder(cfg, blob) as dec:
        check_teacher_forced(dec, consumed, trace)
        _free_running(dec, prompt, steps, toks, trace)


def test_long_context_attention_all_positions(l2):
    # every position of a 2048-long cache, incl. pos = seq_len - 1
    cfg = config(dim=64, hidden_dim=128, n_layers=2, n_heads=2, vocab_size=256, seq_len=2048)
    blob = synth.make_blob(cfg, 5, std=0.08)
    prompt = np.array([1], np.int32)
    toks, consumed, trace = oracle_run(cfg, blob, prompt, cfg["seq_len"])
    with l2.Decoder(cfg, blob) as dec:
        check_teacher_forced(dec, consumed, trace)
        _free_running(dec, prompt, cfg["seq_len"], toks, trace)


def test_state_is_reset_between_calls(l2):
    cfg = SHAPES["gqa"]
    blob = synth.make_blob(cfg, 2, std=0.05)
    prompt = synth.prompt_ids(9, 4, cfg["vocab_size"])
    with l2.Decoder(cfg, blob) as dec:
        a = dec.generate(prompt, 20)
        b = dec.generate(prompt, 20)
        np.testing.assert_array_equal(a, b)
        # a lower position re-run overwrites its slot: same logits again
        l5 = dec.forward([a[3]], [5])
        dec.forward([a[4]], [6])
        np.testing.assert_array_equal(dec.forward([a[3]], [5]), l5)
        dec.reset()
        np.testing.assert_array_equal(dec.generate(prompt, 20), a)


def test_edge_tokens_and_positions(l2):
    cfg = SHAPES["tiny_ragged"]
    blob = synth.make_blob(cfg, 4, std=0.05)
    import oracle
    om = oracle.Model(cfg, blob)
    with l2.Decoder(cfg, blob) as dec:
        for p, t in enumerate([0, cfg["vocab_size"] - 1, 0]):
            assert rel_l2(dec.forward([t], [p])[0], om.forward(t, p)) <= 1e-4
        with pytest.raises(l2.L2Error):
            dec.forward([cfg["vocab_size"]], [0])
        with pytest.raises(l2.L2Error):
            dec.forward([0], [cfg["seq_len"]])
        with pytest.raises(l2.L2Error):
            dec.generate([1, 2], cfg["seq_len"])


def test_device_entry_points_match_host_ones(l2):
    import torch
    cfg = SHAPES["gqa"]
    blob = synth.make_blob(cfg, 8, std=0.05)
    prompt = synth.prompt_ids(1, 6, cfg["vocab_size"])
    with l2.Decoder(cfg, blob) as dec:
        ref = dec.generate(prompt, 16)
        s = torch.cuda.Stream()
        d_prompt = torch.tensor(prompt, dtype=torch.int32, device="cuda")
        d_out = torch.zeros(16, dtype=torch.int32, device="cuda")
        with torch.cuda.stream(s):
            l2.l2_generate_device(dec.h, d_prompt, len(prompt), 16, d_out, s)
        s.synchronize()
        np.testing.assert_array_equal(d_out.cpu().numpy(), ref)
        # forward through device buffers at the position after the prompt
        host = dec.forward([ref[0]], [len(prompt)])[0]
        d_tok = torch.tensor([ref[0]], dtype=torch.int32, device="cuda")
        d_pos = torch.tensor([len(prompt)], dtype=torch.int32, device="cuda")
        d_lg = torch.empty(cfg["vocab_size"], dtype=torch.float32, device="cuda")
        l2.l2_forward_device(dec.h, d_tok, d_pos, 1, d_lg, s)
        s.synchronize()
        np.testing.assert_array_equal(d_lg.cpu().numpy(), host)


def test_kernel_timing_hook(l2):
    cfg = SHAPES["hd48"]
    blob = synth.make_blob(cfg, 8, std=0.05)
    with l2.Decoder(cfg, blob) as dec:
        for kind in range(6):
            ms = l2.l2_time_kernel(dec.h, kind, 3, 4)
            assert 0.0 < ms < 100.0
            assert l2.l2_kernel_bytes(dec.h, kind, 3) > 0


def test_two_live_handles_of_different_shapes(l2):
    # kernel attributes are process-wide: creating a smaller model must not
    # break launches of a larger model that is still alive
    big, small = SHAPES["k4096"], SHAPES["tiny_ragged"]
    bb = synth.make_blob(big, 31, std=0.05)
    sb = synth.make_blob(small, 32, std=0.05)
    with l2.Decoder(big, bb) as d1:
        ref1 = d1.forward([5], [0])
        with l2.Decoder(small, sb) as d2:
            ref2 = d2.forward([7], [0])
            np.testing.assert_array_equal(d1.forward([5], [0]), ref1)
            np.testing.assert_array_equal(d2.forward([7], [0]), ref2)
