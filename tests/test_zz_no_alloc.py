"""The no-allocation classifier entry point against the handle-based forward
and the oracle.

l2_classify_greedy_noalloc exists for callers that cannot allocate device
memory themselves (their device memory belongs to another framework's arena,
or their serving loop must not stall on cudaMalloc/cudaFree). It keeps its
scratch in a fixed device array inside the library, so it must give the same
result as the classifier of l2_forward, whose scratch a handle allocates.

A model whose layer matrices are all zero leaves the residual stream at the
embedding row (every projection adds exactly zero), so l2_forward's logits at
any position are the final norm + classifier of E[tok]. The no-allocation call
on that row must return their greedy token and its logit; two calls in a row
with different rows check that the shared scratch is cleared between calls.
This file is collected last on purpose.
"""
import numpy as np
import pytest

import synth
from parity_util import GAP_TOL, REL_L2_TOL, config, rel_l2, top2_gap

pytestmark = pytest.mark.gpu


def _offsets(c):
    d, F, L, V = c["dim"], c["hidden_dim"], c["n_layers"], c["vocab_size"]
    kvd = c["n_kv_heads"] * (d // c["n_heads"])
    o = {"E": 0}
    o["g_att"] = V * d
    o["Wq"] = o["g_att"] + L * d
    o["g_ffn"] = o["Wq"] + L * (d * d + 2 * kvd * d + d * d)
    o["W1"] = o["g_ffn"] + L * d
    o["g_final"] = o["W1"] + 3 * L * F * d
    o["Wcls"] = o["g_final"] + d
    return o


def test_noalloc_classifier_matches_forward_on_two_calls():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import llama_fp32_token_decode_b300 as l2

    # the 15M shape's classifier (d 288, V 32000) with one cheap layer
    cfg = config(dim=288, hidden_dim=96, n_layers=1, n_heads=6, vocab_size=32000, seq_len=4)
    blob = synth.make_blob(cfg, 41, std=0.05)
    o = _offsets(cfg)
    d, V = cfg["dim"], cfg["vocab_size"]
    blob[o["Wq"]:o["g_ffn"]] = 0.0
    blob[o["W1"]:o["g_final"]] = 0.0
    rng = np.random.default_rng(7)
    blob[o["g_final"]:o["g_final"] + d] = rng.uniform(0.5, 1.5, d).astype(np.float32)
    assert l2.l2_blob_floats(cfg) == blob.size

    dev = torch.device("cuda", 0)
    d_gain = torch.from_numpy(blob[o["g_final"]:o["g_final"] + d].copy()).to(dev)
    d_wcls = torch.from_numpy(blob[o["Wcls"]:o["Wcls"] + V * d].copy()).to(dev)
    d_token = torch.full((1,), -7, dtype=torch.int32, device=dev)
    d_logit = torch.full((1,), float("nan"), dtype=torch.float32, device=dev)

    import oracle
    om = oracle.Model(cfg, blob)
    with l2.Decoder(cfg, blob) as dec:
        for tok in (17, 29001):
            ref = dec.forward([tok], [0])[0]
            # the closed form of this model, computed by the oracle (its pin:
            # zero layer weights leave logits = Wcls . rmsnorm(E[tok]))
            want_lg = om.forward(tok, 0)
            assert rel_l2(ref, want_lg) <= REL_L2_TOL
            d_x = torch.from_numpy(blob[tok * d:(tok + 1) * d].copy()).to(dev)
            rc = l2.l2_classify_greedy_noalloc(d_x, d_gain, d_wcls, d, V, cfg["norm_eps"],
                                               d_token, d_logit)
            assert rc == l2.L2_OK
            torch.cuda.synchronize()
            want = int(np.argmax(ref))
            assert int(d_token.item()) == want, (tok, int(d_token.item()), want)
            got = float(d_logit.item())
            assert abs(got - float(ref[want])) <= REL_L2_TOL * abs(float(ref[want])), (got, ref[want])
            # and against the oracle directly, where its top-2 gap decides the token
            if top2_gap(want_lg) > GAP_TOL:
                assert int(d_token.item()) == int(np.argmax(want_lg))
            o_want = float(want_lg[int(d_token.item())])
            assert abs(got - o_want) <= REL_L2_TOL * abs(o_want), (got, o_want)
    om.close()

    # sizes beyond the fixed scratch are rejected before any device work
    rc = l2.l2_classify_greedy_noalloc(d_gain, d_gain, d_wcls, d, l2.L2_NOALLOC_MAX_VOCAB + 1,
                                       1e-5, d_token)
    assert rc == l2.L2_EINVAL
