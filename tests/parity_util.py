"""Shared helpers of the GPU parity tests (not collected by pytest)."""
import numpy as np

import oracle
import synth

REL_L2_TOL = 1e-4     # per-step logits, relative L2 error
GAP_TOL = 1e-3        # greedy tokens must agree where the top-2 gap exceeds this


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def top2_gap(logits) -> float:
    t = np.partition(np.asarray(logits, np.float64), -2)[-2:]
    return float(t[1] - t[0])


def config(**kw):
    c = dict(dim=64, hidden_dim=160, n_layers=2, n_heads=4, vocab_size=1000,
             seq_len=32, rope_theta=10000.0, norm_eps=1e-5, shared_classifier=0, max_batch=1)
    c.update(kw)
    c.setdefault("n_kv_heads", c["n_heads"])
    return c


def oracle_run(cfg, blob, prompt, steps):
    """Oracle tokens, the token consumed at every position, and per-position logits."""
    out, trace = oracle.Model(cfg, blob).generate(prompt, steps, trace=True)
    consumed = np.concatenate([np.asarray(prompt, np.int32), out[:-1]])
    return out, consumed, trace


def first_near_tie(trace, n_prompt):
    """Index (into generated tokens) of the first step whose top-2 gap <= GAP_TOL."""
    for k, p in enumerate(range(n_prompt - 1, trace.shape[0])):
        if top2_gap(trace[p]) <= GAP_TOL:
            return k
    return trace.shape[0] - n_prompt + 1


def check_teacher_forced(dec, consumed, trace, positions=None):
    """GPU logits at each position, fed the oracle's tokens, against the oracle."""
    positions = range(len(consumed)) if positions is None else positions
    worst = 0.0
    for p in positions:
        lg = dec.forward([consumed[p]], [p])[0]
        assert np.all(np.isfinite(lg)), f"non-finite logits at pos {p}"
        e = rel_l2(lg, trace[p])
        worst = max(worst, e)
        assert e <= REL_L2_TOL, f"pos {p}: rel-L2 {e:.3e}"
        if top2_gap(trace[p]) > GAP_TOL:
            assert int(np.argmax(lg)) == int(np.argmax(trace[p])), f"pos {p}: argmax differs"
    return worst


def _trace_worker(args):
    """Spawned worker: rebuild the seeded blob, then the oracle's logits at
    positions 0 .. len(tokens) - 1 of one sequence fed `tokens`."""
    cfg, seed, std, tokens = args
    blob = synth.make_blob(cfg, seed, std=std, threads=1)
    m = oracle.Model(cfg, blob)
    out = np.stack([m.forward(int(t), p) for p, t in enumerate(tokens)])
    m.close()
    return out


def _generate_worker(args):
    cfg, seed, std, prompt, steps = args
    blob = synth.make_blob(cfg, seed, std=std, threads=1)
    return oracle.Model(cfg, blob).generate(np.asarray(prompt, np.int32), steps, trace=True)


class OracleJobs:
    """Oracle runs in spawned processes (safe beside an initialised CUDA
    context), started before the GPU work so that both proceed at once."""

    def __init__(self, n: int):
        import multiprocessing
        import os
        ctx = multiprocessing.get_context("spawn")
        self.pool = ctx.Pool(max(1, min(n, os.cpu_count() or 1)))

    def traces(self, cfg, seed, std, token_lists):
        return self.pool.map_async(_trace_worker,
                                   [(cfg, seed, std, np.asarray(t, np.int32)) for t in token_lists])

    def generate(self, cfg, seed, std, prompt, steps):
        return self.pool.apply_async(_generate_worker, ((cfg, seed, std, prompt, steps),))

    def close(self):
        self.pool.close()
        self.pool.join()
