"""Failure detection on the GPU, without faulting it.

* Bounded waits. Every wait of a decode kernel on a bulk-copy completion gives
  up after a bounded number of SM clock cycles, records the timeout in the
  handle's device error word, and the call returns L2_ETIMEOUT.
  l2_watchdog_check runs that same bounded wait on an mbarrier that nothing
  arrives at (no copy in flight) with a short limit: it must give up, the call
  must return L2_ETIMEOUT, and the handle must stay usable.
* Device inputs. The *_device calls take token ids and positions that the host
  never sees. An id outside [0, V) or a position outside its range is clamped
  on the device (every access stays in bounds) and reported as L2_EINVAL by
  l2_status; a synchronous call starts from a clear error word.
"""
import numpy as np
import pytest

import synth
from parity_util import REL_L2_TOL, config, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def l2():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import llama_fp32_token_decode_b300 as m
    return m


def _model(cfg, seed=3):
    return synth.make_blob(cfg, seed, std=0.05)


def test_bounded_wait_gives_up_and_handle_stays_usable(l2):
    cfg = config()
    blob = _model(cfg)
    with l2.Decoder(cfg, blob) as dec:
        before = dec.forward([5], [0])[0]
        for limit in (1, 2_000_000):          # one cycle, then about a millisecond
            assert l2.l2_watchdog_check(dec.h, limit) == l2.L2_ETIMEOUT
            assert "bounded device wait" in l2.l2_last_error(dec.h)
        assert l2.l2_status(dec.h) == l2.L2_OK   # the word was cleared
        after = dec.forward([5], [0])[0]         # the next call runs normally
        assert rel_l2(after, before) == 0.0
        assert l2.l2_watchdog_check(dec.h, 0) == l2.L2_EINVAL


def test_bad_device_token_is_reported_not_decoded(l2):
    import torch
    cfg = config(max_batch=4)
    V = cfg["vocab_size"]
    blob = _model(cfg)
    dev = torch.device("cuda")
    s = torch.cuda.Stream()
    with l2.Decoder(cfg, blob) as dec:
        # batch 1, device forward: token V and token -1
        d_pos = torch.zeros(1, dtype=torch.int32, device=dev)
        for bad in (V, -1):
            d_tok = torch.tensor([bad], dtype=torch.int32, device=dev)
            l2.l2_forward_device(dec.h, d_tok, d_pos, 1, None, s)
            assert l2.l2_status(dec.h, s) == l2.L2_EINVAL
            assert "outside" in l2.l2_last_error(dec.h)
        # a good device call after the report: clear word, L2_OK
        d_tok = torch.tensor([7], dtype=torch.int32, device=dev)
        l2.l2_forward_device(dec.h, d_tok, d_pos, 1, None, s)
        assert l2.l2_status(dec.h, s) == l2.L2_OK
        # device position beyond seq_len
        d_badpos = torch.tensor([cfg["seq_len"]], dtype=torch.int32, device=dev)
        l2.l2_forward_device(dec.h, d_tok, d_badpos, 1, None, s)
        assert l2.l2_status(dec.h, s) == l2.L2_EINVAL
        # generation from a device prompt whose third id is out of range: the
        # bad id is consumed at position 2 and reported
        prompt = torch.tensor([5, 9, V + 3, 11], dtype=torch.int32, device=dev)
        d_out = torch.zeros(4, dtype=torch.int32, device=dev)
        l2.l2_generate_device(dec.h, prompt, 4, 4, d_out, s)
        assert l2.l2_status(dec.h, s) == l2.L2_EINVAL
        good = torch.tensor([5, 9, 13, 11], dtype=torch.int32, device=dev)
        l2.l2_generate_device(dec.h, good, 4, 4, d_out, s)
        assert l2.l2_status(dec.h, s) == l2.L2_OK
        # batched device forward: one of three rows out of range
        d_tok3 = torch.tensor([1, V, 2], dtype=torch.int32, device=dev)
        d_pos3 = torch.zeros(3, dtype=torch.int32, device=dev)
        l2.l2_forward_device(dec.h, d_tok3, d_pos3, 3, None, s)
        assert l2.l2_status(dec.h, s) == l2.L2_EINVAL
        # batched device generation with a bad prompt id in sequence 1
        d_prompts = torch.tensor([4, 5, -2, 6, 7], dtype=torch.int32, device=dev)
        lens = np.array([2, 2, 1], np.int32)
        d_bout = torch.zeros((3, 3), dtype=torch.int32, device=dev)
        l2.l2_generate_batch_device(dec.h, d_prompts, lens, 3, d_bout, s)
        assert l2.l2_status(dec.h, s) == l2.L2_EINVAL
        # a synchronous call starts clear and is unaffected
        lg = dec.forward([1, 2], [0, 0])
        assert np.all(np.isfinite(lg))
        assert l2.l2_status(dec.h) == l2.L2_OK


def test_bad_device_prompt_in_prefill_generation(l2):
    import torch
    cfg = config(max_prefill=8)
    V = cfg["vocab_size"]
    blob = _model(cfg)
    dev = torch.device("cuda")
    s = torch.cuda.Stream()
    with l2.Decoder(cfg, blob) as dec:
        prompt = torch.tensor([5, 9, 2 * V, 11], dtype=torch.int32, device=dev)
        d_out = torch.zeros(3, dtype=torch.int32, device=dev)
        l2.l2_generate_prefill_device(dec.h, prompt, 4, 3, d_out, s)
        assert l2.l2_status(dec.h, s) == l2.L2_EINVAL
        prompt[2] = 13
        l2.l2_generate_prefill_device(dec.h, prompt, 4, 3, d_out, s)
        assert l2.l2_status(dec.h, s) == l2.L2_OK
