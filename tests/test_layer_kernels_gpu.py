"""The two ways a batch-1 forward can be split into kernels, against the oracle.

layer_kernels 5 runs five kernels per layer (QKV + RoPE + KV append,
attention, Wo + residual, W1/W3 + SwiGLU, W2 + residual); layer_kernels 2
runs an attention block (one cluster of 8 CTAs per query head: its Q/K/V
rows, attention, its share of Wo) and an FFN block (W1/W3, SwiGLU and W2 per
hidden-unit slice), the residual kept in 64-bit fixed point. Both compute the
same step; each must match the oracle under teacher forcing (logits within
relative L2 1e-4), generate the oracle's tokens up to its first near-tie, and
leave a KV cache that the other path's forwards can continue from. The long
shapes spread each CTA's share of the cache over several of its warps, whose
partials the CTA combines before the cluster's exchange.
"""
import numpy as np
import pytest

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
    "gqa": config(dim=128, hidden_dim=344, n_layers=3, n_heads=8, n_kv_heads=2, vocab_size=3000,
                  seq_len=40),
    "mqa_tied": config(dim=256, hidden_dim=688, n_layers=2, n_heads=4, n_kv_heads=1,
                       vocab_size=517, seq_len=48, shared_classifier=1),
    "hd48_15m_layers": config(dim=288, hidden_dim=768, n_layers=3, n_heads=6, vocab_size=32000,
                              seq_len=64),
    "hd64_110m_layers": config(dim=768, hidden_dim=2048, n_layers=2, n_heads=12, vocab_size=2000,
                               seq_len=40),
    "rolling": config(dim=128, hidden_dim=344, n_layers=2, n_heads=8, n_kv_heads=2,
                      vocab_size=3001, seq_len=16, rolling_positions=56, rolling_cache=1),
    # up to 25 / 13 cache slots per CTA of a head's cluster: several warps'
    # partials per CTA (8 slots a warp at head_dim <= 64, 4 at 128)
    "gqa_long": config(dim=128, hidden_dim=344, n_layers=2, n_heads=8, n_kv_heads=2,
                       vocab_size=3000, seq_len=200),
    "hd128_long": config(dim=512, hidden_dim=1376, n_layers=1, n_heads=4, vocab_size=1000,
                         seq_len=100),
}


@pytest.mark.parametrize("kernels", [2, 5])
@pytest.mark.parametrize("name", sorted(SHAPES))
def test_layer_kernels_against_oracle(l2, name, kernels):
    cfg = dict(SHAPES[name], layer_kernels=kernels)
    blob = synth.make_blob(cfg, 29, std=0.05)
    prompt = synth.prompt_ids(8, 5, cfg["vocab_size"])
    n_pos = cfg.get("rolling_positions") or cfg["seq_len"]
    steps = n_pos - len(prompt) + 1
    toks, consumed, trace = oracle_run(cfg, blob, prompt, steps)
    with l2.Decoder(cfg, blob) as dec:
        worst = 0.0
        for p, t in enumerate(consumed):
            lg = dec.forward([int(t)], [p])[0]
            e = rel_l2(lg, trace[p])
            worst = max(worst, e)
            assert e <= REL_L2_TOL, f"{name} ({kernels} kernels) pos {p}: rel-L2 {e:.3e}"
        gen = dec.generate(prompt, steps)
        gen2 = dec.generate(prompt, steps)  # deterministic: same tokens again
    np.testing.assert_array_equal(gen, gen2)
    k = first_near_tie(trace, len(prompt))
    n = min(k + 1, steps)
    np.testing.assert_array_equal(gen[:n], toks[:n])
    print(f"{name} ({kernels} kernels/layer): worst rel-L2 {worst:.3e}")


def test_two_kernel_path_is_taken_and_rejected_where_it_does_not_fit(l2):
    # head_dim 12: 3 * head_dim is not a multiple of 16
    cfg = config(dim=72, hidden_dim=200, n_layers=1, n_heads=6, vocab_size=100, seq_len=8,
                 layer_kernels=2)
    with pytest.raises(l2.L2Error) as e:
        l2.Decoder(cfg, synth.make_blob(cfg, 1, std=0.05))
    assert e.value.code == l2.L2_EINVAL
    # the same shape with the default choice falls back to five kernels
    cfg["layer_kernels"] = 0
    with l2.Decoder(cfg, synth.make_blob(cfg, 1, std=0.05)) as dec:
        assert l2.l2_layer_kernels(dec.h) == 5
        assert np.all(np.isfinite(dec.forward([3], [0])[0]))
        with pytest.raises(l2.L2Error) as e:  # the block kinds need the two-kernel path
            l2.l2_time_kernel(dec.h, 14, 0, 1)
        assert e.value.code == l2.L2_EINVAL
    # a shape that fits takes two kernels by default; its blocks time alone
    cfg = dict(SHAPES["gqa"])
    with l2.Decoder(cfg, synth.make_blob(cfg, 1, std=0.05)) as dec:
        assert l2.l2_layer_kernels(dec.h) == 2
        before = dec.forward([3], [0])[0]
        for kind in (14, 15):
            assert l2.l2_time_kernel(dec.h, kind, 5, 3) > 0.0
            assert l2.l2_kernel_bytes(dec.h, kind, 5) > 0.0
        # the timing launches leave nothing behind that a forward reads
        np.testing.assert_array_equal(dec.forward([3], [0])[0], before)
