"""GPU parity with RMSNorm gains other than 1.

Every workload blob has unit norm gains (the configs say so), which would let
a gain that is dropped, misplaced or applied to the wrong layer go unseen.
Here the gain segments of the blob hold seeded values in [0.5, 1.5], and the
batch-1 forward, the batched forward (gains folded into the GEMM weights) and
the prefill pass are each compared with the oracle on the same blob (one
case with a RoPE theta and a norm epsilon other than the workloads').
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


def _blob_with_gains(cfg, seed):
    blob = synth.make_blob(cfg, seed, std=0.05)
    rng = np.random.default_rng(seed + 1000)
    off = 0
    n_gain = 0
    for _, cnt, is_gain in synth.blob_segments(cfg):
        if is_gain:
            blob[off:off + cnt] = rng.uniform(0.5, 1.5, cnt).astype(np.float32)
            n_gain += cnt
        off += cnt
    assert n_gain == cfg["n_layers"] * 2 * cfg["dim"] + cfg["dim"]
    return blob


@pytest.mark.gpu
@pytest.mark.parametrize("n_kv_heads,theta,eps", [(8, 10000.0, 1e-5), (2, 500000.0, 1e-6)])
def test_nonunit_gains_all_paths(l2, n_kv_heads, theta, eps):
    # the second case also moves RoPE theta and the norm epsilon off the
    # workloads' values, so neither can be a constant on any path
    cfg = config(dim=128, hidden_dim=344, n_layers=3, n_heads=8, n_kv_heads=n_kv_heads,
                 vocab_size=1000, seq_len=16, max_batch=3, max_prefill=4, rope_theta=theta,
                 norm_eps=eps)
    blob = _blob_with_gains(cfg, 31)
    toks = np.array([[5, 17, 99], [7, 3, 11], [42, 8, 600], [1, 2, 3]], np.int32)  # [pos][seq]
    refs = []
    for b in range(3):
        m = oracle.Model(cfg, blob)
        refs.append([m.forward(int(toks[p][b]), p) for p in range(4)])
        m.close()
    with l2.Decoder(cfg, blob) as dec:
        for p in range(4):  # batched forward: three sequences in lockstep
            lg = dec.forward(toks[p], [p] * 3)
            for b in range(3):
                e = rel_l2(lg[b], refs[b][p])
                assert e <= REL_L2_TOL, f"batched seq {b} pos {p}: rel-L2 {e:.3e}"
        dec.reset()
        for p in range(4):  # batch-1 forward of sequence 0
            lg = dec.forward([int(toks[p][0])], [p])[0]
            e = rel_l2(lg, refs[0][p])
            assert e <= REL_L2_TOL, f"batch-1 pos {p}: rel-L2 {e:.3e}"
        dec.reset()
        pre = dec.prefill(toks[:, 0])  # prefill pass of sequence 0
        for p in range(4):
            e = rel_l2(pre[p], refs[0][p])
            assert e <= REL_L2_TOL, f"prefill pos {p}: rel-L2 {e:.3e}"


def test_gain_segments_reach_the_oracle():
    # CPU: the modified gains change the oracle's logits (the test above would
    # otherwise compare unit-gain models)
    cfg = config(dim=64, hidden_dim=160, n_layers=2, n_heads=4, vocab_size=300, seq_len=8)
    unit = synth.make_blob(cfg, 31, std=0.05)
    gained = _blob_with_gains(cfg, 31)
    ma, mb = oracle.Model(cfg, unit), oracle.Model(cfg, gained)
    a, b = ma.forward(5, 0), mb.forward(5, 0)
    ma.close()
    mb.close()
    assert rel_l2(b, a) > 1e-2


@pytest.mark.gpu
def test_nonunit_gains_prefill_long_k(l2):
    # A prefill-only handle (at most 64 rows: 64-row A tiles, wave-balanced K
    # splits) with K ranges long enough that its GEMM CTAs drain accumulation
    # chunks, and RMSNorm gains other than 1 folded into the GEMM weights.
    # Every position against the oracle, in one pass and in two.
    cfg = config(dim=2048, hidden_dim=5632, n_layers=2, n_heads=16, n_kv_heads=4,
                 vocab_size=1000, seq_len=48, max_prefill=40)
    blob = _blob_with_gains(cfg, 37)
    toks = synth.prompt_ids(37, 40, cfg["vocab_size"])
    m = oracle.Model(cfg, blob)
    refs = [m.forward(int(t), p) for p, t in enumerate(toks)]
    m.close()
    with l2.Decoder(cfg, blob) as dec:
        pre = dec.prefill(toks)
        worst = 0.0
        for p in range(len(toks)):
            e = rel_l2(pre[p], refs[p])
            worst = max(worst, e)
            assert e <= REL_L2_TOL, f"prefill pos {p}: rel-L2 {e:.3e}"
        # and the second half again, after the first half is in the cache
        dec.reset()
        dec.prefill(toks[:20])
        pre2 = dec.prefill(toks[20:], pos0=20)
        for p in range(20, len(toks)):
            e = rel_l2(pre2[p - 20], refs[p])
            assert e <= REL_L2_TOL, f"second pass pos {p}: rel-L2 {e:.3e}"
    print(f"long-K prefill with gains: worst rel-L2 {worst:.3e}")
