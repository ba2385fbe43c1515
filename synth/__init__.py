"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

Nothing here computes any part of the decode step. The module draws random-init
weights and prompt ids (generator defined in ``synth.c``). It also names the
workloads: model shapes and run lengths of the llama2.c pages, with seeds.

Workloads (shapes from the llama2.c pages; trained weights and the TinyStories
data are not available, so weights are N(0, 0.02) and prompts are uniform ids):
  * ``15m``  dim 288, 6 layers, 6 heads -- the model of the 新智元 article's
    paragraph before "感受魔力" and of the introduction of
    "llama2.c｜Baby LLaMA-openAI维基百科".
  * ``44m``  dim 512, 8 layers, 8 heads, context 1024 -- "训练示例" on the
    openai.wiki page.
  * ``110m`` dim 768, 12 layers, 12 heads, context 1024.
  * ``7b``   dim 4096, 32 layers, 32 heads, hidden 11008, context 2048 -- the
    smallest Meta checkpoint that both pages call slow for the C engine.
  * ``batched`` the 44m shape, 256 independent sequences.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")

STREAM_WEIGHTS = 0x57454947  # "WEIG"
STREAM_PROMPT = 0x50524F4D  # "PROM"
STREAM_LENGTHS = 0x4C454E53  # "LENS"
STREAM_BATCH_PROMPT = 0x42505254  # "BPRT"

WEIGHT_STD = 0.02
PROMPT_ID_LO = 3  # ids 0..2 are the special tokens of a Llama tokenizer

_BASE = dict(n_kv_heads=None, vocab_size=32000, rope_theta=10000.0, norm_eps=1e-5,
             shared_classifier=0, max_batch=1)

WORKLOADS = {
    "15m": dict(dim=288, hidden_dim=768, n_layers=6, n_heads=6, seq_len=256, seed=0,
                prompt="bos", n_prompt=1, steps=256),
    "44m": dict(dim=512, hidden_dim=1376, n_layers=8, n_heads=8, seq_len=1024, seed=1,
                prompt="random", n_prompt=32, steps=992),
    "110m": dict(dim=768, hidden_dim=2048, n_layers=12, n_heads=12, seq_len=1024, seed=2,
                 prompt="bos", n_prompt=1, steps=1024),
    "7b": dict(dim=4096, hidden_dim=11008, n_layers=32, n_heads=32, seq_len=2048, seed=3,
               prompt="random", n_prompt=64, steps=256),
    "batched": dict(dim=512, hidden_dim=1376, n_layers=8, n_heads=8, seq_len=1024, seed=4,
                    prompt="batch", batch=256, len_lo=1, len_hi=128, steps=512,
                    max_batch=256),
}

CONFIG_KEYS = ("dim", "hidden_dim", "n_layers", "n_heads", "n_kv_heads", "vocab_size",
               "seq_len", "rope_theta", "norm_eps", "shared_classifier", "max_batch")


def workload(name: str) -> dict:
    """Full description of a named workload (model config + run + seed)."""
    w = dict(_BASE)
    w.update(WORKLOADS[name])
    if w["n_kv_heads"] is None:
        w["n_kv_heads"] = w["n_heads"]
    w["name"] = name
    return w


def model_config(w: dict) -> dict:
    """The model-config part of a workload, keyed like the C config struct."""
    return {k: w[k] for k in CONFIG_KEYS if k in w}


def _lib():
    global _LIB
    try:
        return _LIB
    except NameError:
        pass
    if not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        build()
    lib = ctypes.CDLL(_LIB_PATH)
    lib.synth_mix64.restype = ctypes.c_uint64
    lib.synth_mix64.argtypes = [ctypes.c_uint64]
    lib.synth_word.restype = ctypes.c_uint64
    lib.synth_word.argtypes = [ctypes.c_uint64] * 3
    lib.synth_uniform.restype = ctypes.c_double
    lib.synth_uniform.argtypes = [ctypes.c_uint64] * 3
    lib.synth_normal.restype = ctypes.c_double
    lib.synth_normal.argtypes = [ctypes.c_uint64] * 3
    lib.synth_fill_normal.restype = ctypes.c_int
    lib.synth_fill_normal.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                      ctypes.c_size_t, ctypes.c_double, ctypes.c_void_p,
                                      ctypes.c_int]
    lib.synth_fill_ids.restype = ctypes.c_int
    lib.synth_fill_ids.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                   ctypes.c_size_t, ctypes.c_int32, ctypes.c_int32,
                                   ctypes.c_void_p]
    _LIB = lib
    return lib


def build() -> str:
    """Compile libsynth.so in place (gcc, no fast-math)."""
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fno-fast-math", "-fPIC", "-shared", "-pthread",
                           _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def mix64(z: int) -> int:
    return int(_lib().synth_mix64(z & 0xFFFFFFFFFFFFFFFF))


def uniform(seed: int, stream: int, k: int) -> float:
    return float(_lib().synth_uniform(seed, stream, k))


def normal(seed: int, stream: int, k: int) -> float:
    return float(_lib().synth_normal(seed, stream, k))


def blob_segments(cfg: dict):
    """(name, n_floats, is_gain) for each tensor of the documented blob order."""
    d, F, L, V = cfg["dim"], cfg["hidden_dim"], cfg["n_layers"], cfg["vocab_size"]
    kvd = cfg["n_kv_heads"] * (d // cfg["n_heads"])
    segs = [("E", V * d, False), ("g_att", L * d, True), ("Wq", L * d * d, False),
            ("Wk", L * kvd * d, False), ("Wv", L * kvd * d, False), ("Wo", L * d * d, False),
            ("g_ffn", L * d, True), ("W1", L * F * d, False), ("W2", L * d * F, False),
            ("W3", L * F * d, False), ("g_final", d, True)]
    if not cfg.get("shared_classifier", 0):
        segs.append(("Wcls", V * d, False))
    return segs


def blob_floats(cfg: dict) -> int:
    return sum(n for _, n, _ in blob_segments(cfg))


def make_blob(cfg: dict, seed: int, out: np.ndarray | None = None, threads: int | None = None,
              std: float = WEIGHT_STD) -> np.ndarray:
    """Random-init fp32 blob: weight element k (global index in blob order) is
    std * normal(seed, WEIGHTS, k); norm gains are 1.0 and draw nothing."""
    n = blob_floats(cfg)
    if out is None:
        out = np.empty(n, dtype=np.float32)
    assert out.dtype == np.float32 and out.size == n and out.flags["C_CONTIGUOUS"]
    threads = threads or os.cpu_count() or 1
    lib = _lib()
    off = 0
    base = out.ctypes.data
    for _, cnt, is_gain in blob_segments(cfg):
        if is_gain:
            out[off:off + cnt] = 1.0
        else:
            lib.synth_fill_normal(seed, STREAM_WEIGHTS, off, cnt, std, base + 4 * off, threads)
        off += cnt
    return out


def fill_ids(seed: int, stream: int, k0: int, n: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    if n:
        rc = _lib().synth_fill_ids(seed, stream, k0, n, lo, hi, out.ctypes.data)
        if rc != 0:
            raise ValueError("empty id range")
    return out


def prompt_ids(seed: int, n: int, vocab: int) -> np.ndarray:
    """n prompt ids uniform in [3, vocab)."""
    return fill_ids(seed, STREAM_PROMPT, 0, n, PROMPT_ID_LO, vocab)


def batch_lengths(seed: int, batch: int, lo: int, hi: int) -> np.ndarray:
    """Prompt lengths uniform in [lo, hi] (inclusive)."""
    return fill_ids(seed, STREAM_LENGTHS, 0, batch, lo, hi + 1)


def batch_prompts(seed: int, lens, vocab: int, stride: int = 1 << 16) -> np.ndarray:
    """Concatenated prompts; sequence b draws counters b*stride + i."""
    parts = [fill_ids(seed, STREAM_BATCH_PROMPT, b * stride, int(n), PROMPT_ID_LO, vocab)
             for b, n in enumerate(lens)]
    return np.concatenate(parts) if parts else np.empty(0, dtype=np.int32)


def prompt(w: dict) -> np.ndarray:
    """Prompt of a batch-1 workload: token id 1 ("bos") or random ids."""
    if w["prompt"] == "bos":
        return np.ones(w["n_prompt"], dtype=np.int32)
    return prompt_ids(w["seed"], w["n_prompt"], w["vocab_size"])


def batch_inputs(w: dict):
    """(lens[B], concatenated prompts) of a batched workload."""
    lens = batch_lengths(w["seed"], w["batch"], w["len_lo"], w["len_hi"])
    return lens, batch_prompts(w["seed"], lens, w["vocab_size"])
