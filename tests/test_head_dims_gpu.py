"""GPU parity at head sizes the vectorised attention kernels do not take.

The attention kernels read cache rows with 16-byte loads when head_dim is a
multiple of 4 and at most 128; other even head sizes (the config allows any
even head_dim up to 256) go through the scalar kernels, one element per
lane. Here head_dim 6 (not a multiple of 4) and 256 (above 128, with one
shared key/value head) are compared with the oracle on the batch-1 forward,
the batched forward and the prefill pass.
"""
import numpy as np
import pytest

import oracle
import synth
from parity_util import REL_L2_TOL, config, rel_l2


@pytest.fixture(scope="module")
def l2():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import llama_fp32_token_decode_b300 as m
    return m


SHAPES = {
    "hd6": config(dim=36, hidden_dim=96, n_layers=2, n_heads=6, vocab_size=503, seq_len=20,
                  max_batch=3, max_prefill=6),
    "hd256_mqa": config(dim=512, hidden_dim=1024, n_layers=2, n_heads=2, n_kv_heads=1,
                        vocab_size=700, seq_len=20, max_batch=3, max_prefill=6),
}


def test_shapes_take_the_scalar_attention():
    # CPU: the shapes really are outside the vectorised kernels' range
    for cfg in SHAPES.values():
        hd = cfg["dim"] // cfg["n_heads"]
        assert hd % 2 == 0 and (hd % 4 != 0 or hd > 128)


@pytest.mark.gpu
@pytest.mark.parametrize("name", sorted(SHAPES))
def test_scalar_attention_head_sizes_all_paths(l2, name):
    cfg = SHAPES[name]
    blob = synth.make_blob(cfg, 41, std=0.1)
    n_pos = 6
    rng = np.random.default_rng(7)
    toks = rng.integers(0, cfg["vocab_size"], size=(n_pos, 3)).astype(np.int32)  # [pos][seq]
    refs = []
    for b in range(3):
        m = oracle.Model(cfg, blob)
        refs.append([m.forward(int(toks[p][b]), p) for p in range(n_pos)])
        m.close()
    with l2.Decoder(cfg, blob) as dec:
        for p in range(n_pos):  # batched forward: three sequences in lockstep
            lg = dec.forward(toks[p], [p] * 3)
            for b in range(3):
                e = rel_l2(lg[b], refs[b][p])
                assert e <= REL_L2_TOL, f"{name} batched seq {b} pos {p}: rel-L2 {e:.3e}"
        dec.reset()
        for p in range(n_pos):  # batch-1 forward of sequence 1
            lg = dec.forward([int(toks[p][1])], [p])[0]
            e = rel_l2(lg, refs[1][p])
            assert e <= REL_L2_TOL, f"{name} batch-1 pos {p}: rel-L2 {e:.3e}"
        dec.reset()
        pre = dec.prefill(toks[:, 2])  # prefill pass of sequence 2
        for p in range(n_pos):
            e = rel_l2(pre[p], refs[2][p])
            assert e <= REL_L2_TOL, f"{name} prefill pos {p}: rel-L2 {e:.3e}"
