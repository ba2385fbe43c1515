"""GPU parity of the attention kernels the full-size workloads run, over long
caches, against the C oracle.

The 7B-shape workload (dim 4096, 32 heads of 128) attends with one cluster of
8 CTAs per head; with 8 heads of 128 (dim 1024) the cluster has 16 CTAs. Both
tests below use those head layouts with one or two layers and small F and V
(so that the oracle finishes in seconds to a minute) and check every position
of the cache: each CTA of a cluster then walks its share of the positions in
more than one loop iteration, issues the early loads of earlier positions
before its dependency wait, and at position seq_len - 1 takes the path
without them. The batched test runs the 44M shape (dim 512, 8 layers, hidden
1376, vocab 32000) with 256 live rows at staggered positions, three of them
replayed by the oracle past position 300.

Protocol as elsewhere: teacher forcing, logits within relative L2 1e-4 of the
oracle, greedy tokens equal wherever the oracle's top-2 gap exceeds 1e-3; the
free-running generation equal to the oracle's up to its first near-tie.
"""
import numpy as np
import pytest

import synth
from parity_util import (GAP_TOL, REL_L2_TOL, OracleJobs, config, first_near_tie, rel_l2,
                         top2_gap)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def l2():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import llama_fp32_token_decode_b300 as m
    return m


def _check_positions(name, got, want):
    worst = 0.0
    for p in range(len(want)):
        assert np.all(np.isfinite(got[p])), f"{name} pos {p}: non-finite logits"
        e = rel_l2(got[p], want[p])
        worst = max(worst, e)
        assert e <= REL_L2_TOL, f"{name} pos {p}: rel-L2 {e:.3e}"
        if top2_gap(want[p]) > GAP_TOL:
            assert int(np.argmax(got[p])) == int(np.argmax(want[p])), f"{name} pos {p}: argmax"
    print(f"{name}: worst rel-L2 {worst:.3e} over {len(want)} positions")
    return worst


# (name, config, seed, generation prompt length)
HEAD128 = {
    # 32 heads of 128: the 7B shape's attention (8-CTA cluster per head)
    "h32_hd128": (config(dim=4096, hidden_dim=512, n_layers=1, n_heads=32, vocab_size=512,
                         seq_len=512), 31, 64),
    # 8 heads of 128: 16-CTA cluster per head, two layers
    "h8_hd128": (config(dim=1024, hidden_dim=512, n_layers=2, n_heads=8, vocab_size=512,
                        seq_len=1024), 32, 16),
}


@pytest.mark.parametrize("name", sorted(HEAD128))
def test_head_dim_128_every_position(l2, name):
    import torch
    cfg, seed, n_prompt = HEAD128[name]
    std = synth.WEIGHT_STD
    S = cfg["seq_len"]
    tokens = synth.prompt_ids(seed, S, cfg["vocab_size"])
    prompt = tokens[:n_prompt]
    steps = S - n_prompt + 1
    jobs = OracleJobs(2)
    try:
        tf = jobs.traces(cfg, seed, std, [tokens])
        gen = jobs.generate(cfg, seed, std, prompt, steps)
        blob = synth.make_blob(cfg, seed, std=std)
        with l2.Decoder(cfg, blob) as dec:
            got = np.stack([dec.forward([int(t)], [p])[0] for p, t in enumerate(tokens)])
            s = torch.cuda.Stream()
            d_prompt = torch.tensor(prompt, dtype=torch.int32, device="cuda")
            d_out = torch.zeros(steps, dtype=torch.int32, device="cuda")
            l2.l2_generate_device(dec.h, d_prompt, n_prompt, steps, d_out, s)
            s.synchronize()
            gpu_gen = d_out.cpu().numpy()
        want = tf.get()[0]
        o_tokens, o_trace = gen.get()
    finally:
        jobs.close()
    _check_positions(name, got, want)
    k = first_near_tie(o_trace, n_prompt)
    n = min(k + 1, steps)
    np.testing.assert_array_equal(gpu_gen[:n], o_tokens[:n])
    print(f"{name}: generation equal to the oracle for {n} of {steps} tokens")


def test_batched_44m_shape_past_position_300(l2):
    import torch
    w = synth.workload("batched")
    cfg = synth.model_config(w)
    B, V, seed, std = int(w["batch"]), cfg["vocab_size"], int(w["seed"]), synth.WEIGHT_STD
    T = 370                                       # lockstep steps
    start = synth.fill_ids(seed, 0x53544152, 0, B, 0, 64)   # row b starts at step start[b]
    toks = np.stack([synth.prompt_ids(seed * 4096 + b, T, V) for b in range(B)])
    order = np.argsort(start, kind="stable")
    rows = [int(order[0]), int(order[B // 2]), int(order[-1])]
    n_pos = [T - int(start[b]) for b in rows]     # positions 0 .. n_pos - 1 of each row
    assert min(n_pos) > 300
    jobs = OracleJobs(len(rows))
    try:
        tf = jobs.traces(cfg, seed, std, [toks[b, :n] for b, n in zip(rows, n_pos)])
        blob = synth.make_blob(cfg, seed, std=std)
        got = [np.empty((n, V), np.float32) for n in n_pos]
        with l2.Decoder(cfg, blob) as dec:
            del blob
            dev = torch.device("cuda")
            s = torch.cuda.Stream()
            d_logits = torch.empty((B, V), dtype=torch.float32, device=dev)
            for t in range(T):
                # a row that has not started yet rewrites its slot 0 with its first token
                pos = np.maximum(t - start, 0).astype(np.int32)
                tok = toks[np.arange(B), pos].astype(np.int32)
                d_tok = torch.from_numpy(tok).to(dev)
                d_pos = torch.from_numpy(pos).to(dev)
                torch.cuda.current_stream().synchronize()
                l2.l2_forward_device(dec.h, d_tok, d_pos, B, d_logits, s)
                s.synchronize()
                sel = d_logits[rows].cpu().numpy()
                for i, b in enumerate(rows):
                    if t >= start[b]:
                        got[i][pos[b]] = sel[i]
        want = tf.get()
    finally:
        jobs.close()
    for i, b in enumerate(rows):
        _check_positions(f"batched row {b} (start {int(start[b])})", got[i], want[i])
