"""Pins for the oracle's whole decode step and generation loop.

* a hand-worked dim-8, two-layer, two-head model over two positions, whose
  logits are derived below step by step in scalar form;
* a zero-weight model, where the residual stream never changes and the logits
  have a closed form;
* a brute-force recompute: the full causal (masked T x T) forward over all
  positions at once, in float64, against the oracle's incremental KV-cache
  decode, including grouped kv heads;
* the loop's token feeding (prompt positions forced, then greedy).
"""
import math

import numpy as np
import pytest

import oracle
import synth

EPS = 1e-5


def _cfg(**kw):
    c = dict(dim=8, hidden_dim=16, n_layers=2, n_heads=2, n_kv_heads=2, vocab_size=8,
             seq_len=4, rope_theta=10000.0, norm_eps=EPS, shared_classifier=0)
    c.update(kw)
    return c


def _assemble(cfg, t):
    """Blob in the documented order from a dict of tensors."""
    order = ["E", "g_att", "Wq", "Wk", "Wv", "Wo", "g_ffn", "W1", "W2", "W3", "g_final", "Wcls"]
    parts = [np.asarray(t[k], np.float32).ravel() for k in order
             if not (k == "Wcls" and cfg["shared_classifier"])]
    b = np.concatenate(parts)
    assert b.size == oracle.blob_floats(cfg)
    return b


# ---------------------------------------------------------------- hand-worked model

def _handworked_blob(cfg):
    d, F, L, V = 8, 16, 2, 8
    I = np.eye(d)
    S = np.roll(I, 1, axis=0)  # S e_j = e_{j+1 mod 8}
    W1 = np.zeros((L, F, d)); W3 = np.zeros((L, F, d)); W2 = np.zeros((L, d, F))
    W1[0, :d] = I; W3[0, :d] = 0.5 * I; W2[0, :, :d] = I      # layer 1 has no FFN
    Wq = np.stack([I, 0 * I]); Wk = np.stack([I, 0 * I])
    Wv = np.stack([S, I]); Wo = np.stack([0.5 * I, 0.25 * S])
    Wcls = np.zeros((V, d))
    for v in range(V):
        Wcls[v, v] = v + 1
        Wcls[v, (v + 1) % d] += 0.5
    t = dict(E=2 * np.eye(V, d), g_att=np.ones((L, d)), Wq=Wq, Wk=Wk, Wv=Wv, Wo=Wo,
             g_ffn=np.ones((L, d)), W1=W1, W2=W2, W3=W3, g_final=np.ones(d), Wcls=Wcls)
    return _assemble(cfg, t)


def _silu(z):
    return z / (1.0 + math.exp(-z))


def _handworked_expected():
    """Logits at pos 0 (token 1) and pos 1 (token 6), derived by hand.

    Notation: e_j unit vectors of R^8, N(c) = c / sqrt(c^2/8 + eps) is the
    RMSNorm of c e_j, S e_j = e_{j+1}.  Head 0 holds dims 0-3, head 1 dims 4-7.
    """
    def cls(xn):  # logits_v = (v+1) xn_v + 0.5 xn_{v+1}
        return [(v + 1) * xn[v] + 0.5 * xn[(v + 1) % 8] for v in range(8)]

    def norm(x):  # RMSNorm with unit gain, x given as a dict {index: value}
        m = sum(val * val for val in x.values()) / 8 + EPS
        return {j: val / math.sqrt(m) for j, val in x.items()}

    a = 2 / math.sqrt(4 / 8 + EPS)  # N(2)
    # ---- pos 0, token 1: x = 2 e_1
    # layer 0: q = k = a e_1, v = S xb = a e_2, one position so att = v;
    #          x += 0.5 att
    x = {1: 2.0, 2: 0.5 * a}
    # FFN 0: h1 = xb, h3 = 0.5 xb on the first 8 rows; x += silu(h1) * h3
    xb = norm(x)
    x = {j: x[j] + _silu(xb[j]) * 0.5 * xb[j] for j in x}
    # layer 1: q = k = 0, v = xb, one position so att = xb; x += 0.25 S att
    v1_pos0 = norm(x)  # layer-1 value row cached at pos 0
    x = {1: x[1], 2: x[2] + 0.25 * v1_pos0[1], 3: 0.25 * v1_pos0[2]}
    xn = norm(x)
    logits0 = cls([xn.get(j, 0.0) for j in range(8)])

    # ---- pos 1, token 6: x = 2 e_6
    # layer 0: xb = a e_6, v = a e_7; q = k = a R(pos 1) e_6, where e_6 is pair
    #   (2, 3) of head 1 (angle 0.01 rad) -- norm preserved.
    #   head 0: q = 0, both scores 0, weights 1/2: att = 0.5 (a e_2 + 0)
    #   head 1: score(pos0) = 0 (k at pos 0 lives in head 0), score(pos1) =
    #           |q|^2 / sqrt(4) = a^2 / 2: att = w1 a e_7, w1 = sigmoid(a^2/2)
    w1 = 1 / (1 + math.exp(-a * a / 2))
    x = {2: 0.25 * a, 6: 2.0, 7: 0.5 * w1 * a}
    xb = norm(x)
    x = {j: x[j] + _silu(xb[j]) * 0.5 * xb[j] for j in x}
    # layer 1: keys are all zero, weights 1/2 over the cached v at pos 0 and
    #   this position's v = xb: att = 0.5 (v1_pos0 + xb); x += 0.25 S att
    xb = norm(x)
    att = {j: 0.5 * (v1_pos0.get(j, 0.0) + xb.get(j, 0.0)) for j in range(8)}
    x = {j: x.get(j, 0.0) + 0.25 * att[(j - 1) % 8] for j in range(8)}
    xn = norm(x)
    logits1 = cls([xn[j] for j in range(8)])
    return np.array(logits0), np.array(logits1)


def test_handworked_two_layer_model():
    cfg = _cfg()
    m = oracle.Model(cfg, _handworked_blob(cfg))
    l0 = m.forward(1, 0)
    l1 = m.forward(6, 1)
    e0, e1 = _handworked_expected()
    np.testing.assert_allclose(l0, e0, rtol=2e-6, atol=2e-6)
    np.testing.assert_allclose(l1, e1, rtol=2e-6, atol=2e-6)
    # the greedy choices of the two steps
    assert oracle.argmax(l0) == int(np.argmax(e0))
    assert oracle.argmax(l1) == int(np.argmax(e1))


# ---------------------------------------------------------------- zero-weight model

def test_zero_layer_weights_closed_form():
    cfg = _cfg(dim=32, hidden_dim=48, n_layers=3, n_heads=4, n_kv_heads=4, vocab_size=50,
               seq_len=8)
    d, V, L, F = 32, 50, 3, 48
    r = np.random.default_rng(7)
    E = r.normal(0, 1, (V, d)); gf = r.uniform(0.5, 1.5, d); Wcls = r.normal(0, 1, (V, d))
    z = lambda *s: np.zeros(s)
    t = dict(E=E, g_att=r.uniform(0.5, 1.5, (L, d)), Wq=z(L, d, d), Wk=z(L, d, d),
             Wv=z(L, d, d), Wo=z(L, d, d), g_ffn=r.uniform(0.5, 1.5, (L, d)), W1=z(L, F, d),
             W2=z(L, d, F), W3=z(L, F, d), g_final=gf, Wcls=Wcls)
    m = oracle.Model(cfg, _assemble(cfg, t))
    E32 = E.astype(np.float32).astype(np.float64)
    for pos, tok in enumerate([3, 17, 3, 49]):
        x = E32[tok]
        expect = Wcls.astype(np.float32).astype(np.float64) @ (
            gf.astype(np.float32) * x / np.sqrt(np.mean(x * x) + EPS))
        np.testing.assert_allclose(m.forward(tok, pos), expect, rtol=1e-5, atol=1e-5)


# ---------------------------------------------------------------- brute-force recompute

def _full_causal_forward(cfg, blob, tokens, window=None):
    """All positions at once in float64 with a T x T causal mask (position t
    attends to t - window + 1 .. t when a window is given); no KV cache."""
    d, F, L, V = cfg["dim"], cfg["hidden_dim"], cfg["n_layers"], cfg["vocab_size"]
    H, KVH = cfg["n_heads"], cfg["n_kv_heads"]
    hd = d // H
    kvd = KVH * hd
    b = blob.astype(np.float64)
    off = 0

    def take(*shape):
        nonlocal off
        n = int(np.prod(shape))
        out = b[off:off + n].reshape(shape)
        off += n
        return out

    E = take(V, d); ga = take(L, d); Wq = take(L, d, d); Wk = take(L, kvd, d)
    Wv = take(L, kvd, d); Wo = take(L, d, d); gf_ = take(L, d); W1 = take(L, F, d)
    W2 = take(L, d, F); W3 = take(L, F, d); gfin = take(d)
    Wc = E if cfg["shared_classifier"] else take(V, d)
    T = len(tokens)
    pos = np.arange(T)
    i = np.arange(hd // 2)
    ang = pos[:, None] * cfg["rope_theta"] ** (-2.0 * i / hd)[None, :]   # [T][hd/2]
    cos = np.cos(ang).astype(np.float32).astype(np.float64)
    sin = np.sin(ang).astype(np.float32).astype(np.float64)

    def rms(x, g):
        return g * x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + EPS)

    def rope(m, nh):  # m [T][nh*hd]
        m = m.reshape(T, nh, hd // 2, 2)
        a, bb = m[..., 0], m[..., 1]
        c, s = cos[:, None, :], sin[:, None, :]
        return np.stack([a * c - bb * s, a * s + bb * c], -1).reshape(T, nh * hd)

    mask = np.tril(np.ones((T, T), bool))
    if window is not None:
        mask &= ~np.tril(np.ones((T, T), bool), -window)
    x = E[np.asarray(tokens)]
    for l in range(L):
        xb = rms(x, ga[l])
        q = rope(xb @ Wq[l].T, H).reshape(T, H, hd)
        k = rope(xb @ Wk[l].T, KVH).reshape(T, KVH, hd)
        v = (xb @ Wv[l].T).reshape(T, KVH, hd)
        att = np.zeros((T, H, hd))
        for h in range(H):
            g = h // (H // KVH)
            s = q[:, h] @ k[:, g].T / math.sqrt(hd)
            s = np.where(mask, s, -np.inf)
            p = np.exp(s - s.max(1, keepdims=True))
            p /= p.sum(1, keepdims=True)
            att[:, h] = p @ v[:, g]
        x = x + att.reshape(T, d) @ Wo[l].T
        xb = rms(x, gf_[l])
        h1 = xb @ W1[l].T
        h3 = xb @ W3[l].T
        x = x + (h1 / (1 + np.exp(-h1)) * h3) @ W2[l].T
    return rms(x, gfin) @ Wc.T


@pytest.mark.parametrize("shape", [
    dict(dim=16, hidden_dim=40, n_layers=2, n_heads=4, n_kv_heads=4, vocab_size=23, seq_len=12),
    dict(dim=24, hidden_dim=36, n_layers=3, n_heads=4, n_kv_heads=2, vocab_size=31, seq_len=10),
    dict(dim=16, hidden_dim=24, n_layers=1, n_heads=2, n_kv_heads=1, vocab_size=9, seq_len=7,
         shared_classifier=1),
])
def test_incremental_decode_equals_full_causal_recompute(shape):
    cfg = _cfg(**shape)
    blob = synth.make_blob(cfg, 99, std=0.3)
    # distinct, non-unit norm gains so that every gain vector matters
    r = np.random.default_rng(17)
    off = 0
    for _, n, is_gain in synth.blob_segments(cfg):
        if is_gain:
            blob[off:off + n] = r.uniform(0.5, 1.5, n)
        off += n
    T = cfg["seq_len"]
    tokens = synth.prompt_ids(5, T, cfg["vocab_size"])
    m = oracle.Model(cfg, blob)
    inc = np.stack([m.forward(t, p) for p, t in enumerate(tokens)]).astype(np.float64)
    ref = _full_causal_forward(cfg, blob, tokens)
    err = np.linalg.norm(inc - ref) / np.linalg.norm(ref)
    assert err < 2e-6, err


@pytest.mark.parametrize("shape", [
    dict(dim=16, hidden_dim=40, n_layers=2, n_heads=4, n_kv_heads=4, vocab_size=23, seq_len=4),
    dict(dim=24, hidden_dim=36, n_layers=2, n_heads=4, n_kv_heads=2, vocab_size=31, seq_len=5),
])
def test_rolling_cache_equals_windowed_full_recompute(shape):
    # decoding past seq_len with a rolling cache == every position attending to
    # the last seq_len positions (itself included), RoPE at the absolute position
    cfg = _cfg(rolling_cache=1, **shape)
    blob = synth.make_blob(cfg, 7, std=0.3)
    S = cfg["seq_len"]
    T = 3 * S + 1
    tokens = synth.prompt_ids(8, T, cfg["vocab_size"])
    m = oracle.Model(cfg, blob)
    inc = np.stack([m.forward(t, p) for p, t in enumerate(tokens)]).astype(np.float64)
    ref = _full_causal_forward(cfg, blob, tokens, window=S)
    err = np.linalg.norm(inc - ref) / np.linalg.norm(ref)
    assert err < 2e-6, err
    # the full causal recompute differs once the window has rolled
    full = _full_causal_forward(cfg, blob, tokens)
    assert np.linalg.norm(inc[S:] - full[S:]) / np.linalg.norm(full[S:]) > 1e-3


def test_rolling_cache_before_the_wrap_is_the_plain_cache():
    shape = dict(dim=16, hidden_dim=40, n_layers=2, n_heads=4, n_kv_heads=4, vocab_size=23,
                 seq_len=6)
    blob = synth.make_blob(_cfg(**shape), 12, std=0.3)
    tokens = synth.prompt_ids(2, 6, shape["vocab_size"])
    a = oracle.Model(_cfg(**shape), blob)
    b = oracle.Model(_cfg(rolling_cache=1, **shape), blob)
    for p, t in enumerate(tokens):
        np.testing.assert_array_equal(a.forward(t, p), b.forward(t, p))
    with pytest.raises(ValueError):
        a.forward(1, 6)           # plain cache: position seq_len is out of range
    b.forward(1, 6)               # rolling cache: fine


# ---------------------------------------------------------------- loop semantics

def test_generate_feeds_prompt_then_greedy():
    cfg = _cfg(dim=16, hidden_dim=40, n_layers=2, n_heads=4, n_kv_heads=4, vocab_size=23,
               seq_len=9)
    blob = synth.make_blob(cfg, 3, std=0.3)
    prompt = [5, 9, 11]
    steps = 5
    out, trace = oracle.Model(cfg, blob).generate(prompt, steps, trace=True)
    m = oracle.Model(cfg, blob)
    tok, gen = prompt[0], []
    for pos in range(len(prompt) + steps - 1):
        lg = m.forward(tok, pos)
        np.testing.assert_array_equal(lg, trace[pos])
        best = int(np.argmax(lg))
        if pos >= len(prompt) - 1:
            gen.append(best)
        tok = prompt[pos + 1] if pos + 1 < len(prompt) else best
    assert list(out) == gen


def test_rejects_out_of_range():
    cfg = _cfg()
    m = oracle.Model(cfg, _handworked_blob(cfg))
    with pytest.raises(ValueError):
        m.forward(8, 0)
    with pytest.raises(ValueError):
        m.forward(0, 4)
    with pytest.raises(ValueError):
        m.generate([1, 2], 4)  # 2 + 4 - 1 > seq_len 4
    with pytest.raises(ValueError):
        oracle.Model(cfg, np.zeros(10, np.float32))
