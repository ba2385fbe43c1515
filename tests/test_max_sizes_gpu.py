"""GPU parity at the row limits of the tensor-core path: a batched forward of
max_batch = 1024 sequences (eight 128-row GEMM tiles, 1024 x heads attention
CTAs) and one prefill pass of max_prefill = 1024 positions (attention over up
to 1024 cache slots per row), on a tiny model so the oracle stays fast."""
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


CFG = config(dim=64, hidden_dim=160, n_layers=2, n_heads=4, n_kv_heads=2, vocab_size=1000,
             seq_len=1024, max_batch=1024, max_prefill=1024)


@pytest.mark.gpu
def test_row_limits_batched_forward_and_prefill(l2):
    B, n_pos = CFG["max_batch"], 3
    blob = synth.make_blob(CFG, 53, std=0.1)
    rng = np.random.default_rng(11)
    toks = rng.integers(0, CFG["vocab_size"], size=(n_pos, B)).astype(np.int32)  # [pos][seq]
    checked = sorted({0, 1, 127, 128, 511, 777, 1022, 1023})  # tile edges and the last row
    refs = {}
    for b in checked:
        m = oracle.Model(CFG, blob)
        refs[b] = [m.forward(int(toks[p][b]), p) for p in range(n_pos)]
        m.close()
    prompt = rng.integers(0, CFG["vocab_size"], size=CFG["max_prefill"]).astype(np.int32)
    m = oracle.Model(CFG, blob)
    pre_ref = {p: None for p in (0, 1, 127, 128, 640, 1023)}
    for p, t in enumerate(prompt):
        lg = m.forward(int(t), p)
        if p in pre_ref:
            pre_ref[p] = lg
    m.close()
    with l2.Decoder(CFG, blob) as dec:
        for p in range(n_pos):
            lg = dec.forward(toks[p], [p] * B)
            assert lg.shape == (B, CFG["vocab_size"])
            for b in checked:
                e = rel_l2(lg[b], refs[b][p])
                assert e <= REL_L2_TOL, f"batched seq {b} pos {p}: rel-L2 {e:.3e}"
        dec.reset()
        pre = dec.prefill(prompt)
        assert pre.shape == (CFG["max_prefill"], CFG["vocab_size"])
        for p, ref in pre_ref.items():
            e = rel_l2(pre[p], ref)
            assert e <= REL_L2_TOL, f"prefill pos {p}: rel-L2 {e:.3e}"
