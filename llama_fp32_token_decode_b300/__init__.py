"""Python binding of libl2decode.so (include/l2decode.h), fp32 Llama-2 decode on B300.

Argument marshalling only: every step of the decode path runs in the library's
CUDA kernels. There is no CPU fallback; importing this package fails loudly when
the library has not been built (``python llama_fp32_token_decode_b300/build.py``).
Functions keep the C names: l2_create, l2_create_from_device, l2_forward, l2_forward_device,
l2_generate, l2_generate_device, l2_generate_batch, l2_generate_batch_device,
l2_generate_batch_sample, l2_generate_batch_sample_device, l2_generate_batch_prefill,
l2_generate_batch_prefill_device, l2_prefill, l2_generate_prefill, l2_generate_prefill_device, l2_generate_sample,
l2_generate_sample_device, l2_reset, l2_destroy,
l2_last_error, l2_blob_floats, l2_time_kernel, l2_kernel_bytes, l2_layer_kernels,
l2_classify_greedy_noalloc, l2_gemm_tf32x3, l2_status, l2_watchdog_check.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libl2decode.so")

L2_OK, L2_EINVAL, L2_ENOMEM, L2_ECUDA, L2_ETIMEOUT, L2_EBLOB = 0, -1, -2, -3, -4, -5
ERROR_NAMES = {L2_EINVAL: "L2_EINVAL", L2_ENOMEM: "L2_ENOMEM", L2_ECUDA: "L2_ECUDA",
               L2_ETIMEOUT: "L2_ETIMEOUT", L2_EBLOB: "L2_EBLOB"}

# kinds of l2_time_kernel / l2_kernel_bytes
KERNEL_KINDS = ("qkv_rope", "attention", "wo_residual", "w13_swiglu", "w2_residual",
                "classifier_argmax", "b_qkv_gemm", "b_attention", "b_wo_gemm", "b_w13_gemm",
                "b_w2_gemm", "b_classifier_gemm", "b_embedding", "b_advance",
                "attention_block", "ffn_block")

EXPORTS = ("l2_blob_floats", "l2_create", "l2_create_from_device", "l2_forward", "l2_forward_device", "l2_generate",
           "l2_generate_device", "l2_generate_batch", "l2_generate_batch_device",
           "l2_generate_batch_sample", "l2_generate_batch_sample_device",
           "l2_generate_batch_prefill", "l2_generate_batch_prefill_device", "l2_prefill",
           "l2_generate_prefill", "l2_generate_prefill_device", "l2_generate_sample",
           "l2_generate_sample_device", "l2_reset", "l2_destroy",
           "l2_last_error", "l2_time_kernel", "l2_kernel_bytes", "l2_layer_kernels",
           "l2_classify_greedy_noalloc",
           "l2_gemm_tf32x3", "l2_status", "l2_watchdog_check")

L2_NOALLOC_MAX_VOCAB = 262144


class L2Config(ctypes.Structure):
    _fields_ = [("dim", ctypes.c_int32), ("hidden_dim", ctypes.c_int32),
                ("n_layers", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("vocab_size", ctypes.c_int32),
                ("seq_len", ctypes.c_int32), ("rope_theta", ctypes.c_float),
                ("norm_eps", ctypes.c_float), ("max_batch", ctypes.c_int32),
                ("shared_classifier", ctypes.c_int32), ("max_prefill", ctypes.c_int32),
                ("rolling_positions", ctypes.c_int32), ("layer_kernels", ctypes.c_int32)]


class L2Error(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERROR_NAMES.get(code, code)}: {msg}")
        self.code = code


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with "
                      "`python llama_fp32_token_decode_b300/build.py` (nvcc, sm_103a)")

_lib = ctypes.CDLL(LIB_PATH)
_P = ctypes.c_void_p
_I = ctypes.c_int32
_CFG = ctypes.POINTER(L2Config)
_SIG = {
    "l2_blob_floats": (ctypes.c_size_t, [_CFG]),
    "l2_create": (ctypes.c_int, [_CFG, _P, ctypes.c_size_t, ctypes.POINTER(_P)]),
    "l2_create_from_device": (ctypes.c_int, [_CFG, _P, ctypes.c_size_t, ctypes.POINTER(_P)]),
    "l2_forward": (ctypes.c_int, [_P, _P, _P, _I, _P]),
    "l2_forward_device": (ctypes.c_int, [_P, _P, _P, _I, _P, _P]),
    "l2_generate": (ctypes.c_int, [_P, _P, _I, _I, _P]),
    "l2_generate_device": (ctypes.c_int, [_P, _P, _I, _I, _P, _P]),
    "l2_generate_batch": (ctypes.c_int, [_P, _P, _P, _I, _I, _P]),
    "l2_generate_batch_device": (ctypes.c_int, [_P, _P, _P, _I, _I, _P, _P]),
    "l2_generate_batch_prefill": (ctypes.c_int, [_P, _P, _P, _I, _I, _P]),
    "l2_generate_batch_prefill_device": (ctypes.c_int, [_P, _P, _P, _I, _I, _P, _P]),
    "l2_generate_batch_sample": (ctypes.c_int, [_P, _P, _P, _I, _I, ctypes.c_float,
                                                ctypes.c_float, _P, _P]),
    "l2_generate_batch_sample_device": (ctypes.c_int, [_P, _P, _P, _I, _I, ctypes.c_float,
                                                       ctypes.c_float, _P, _P, _P]),
    "l2_prefill": (ctypes.c_int, [_P, _P, _I, _I, _P]),
    "l2_generate_sample": (ctypes.c_int, [_P, _P, _I, _I, ctypes.c_float, ctypes.c_float, _P, _P]),
    "l2_generate_sample_device": (ctypes.c_int, [_P, _P, _I, _I, ctypes.c_float, ctypes.c_float,
                                                 _P, _P, _P]),
    "l2_generate_prefill": (ctypes.c_int, [_P, _P, _I, _I, _P]),
    "l2_generate_prefill_device": (ctypes.c_int, [_P, _P, _I, _I, _P, _P]),
    "l2_reset": (ctypes.c_int, [_P, _I]),
    "l2_destroy": (None, [_P]),
    "l2_last_error": (ctypes.c_char_p, [_P]),
    "l2_time_kernel": (ctypes.c_int, [_P, _I, _I, _I, _P, ctypes.POINTER(ctypes.c_float)]),
    "l2_kernel_bytes": (ctypes.c_double, [_P, _I, _I]),
    "l2_layer_kernels": (ctypes.c_int32, [_P]),
    "l2_gemm_tf32x3": (ctypes.c_int, [_P, _P, _P, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_float),
                                      _P]),
    "l2_classify_greedy_noalloc": (ctypes.c_int, [_P, _P, _P, _I, _I, ctypes.c_float, _P, _P,
                                                  _P]),
    "l2_status": (ctypes.c_int, [_P, _P]),
    "l2_watchdog_check": (ctypes.c_int, [_P, ctypes.c_int64]),
}
for _name, (_res, _args) in _SIG.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args


def make_config(cfg: dict) -> L2Config:
    return L2Config(cfg["dim"], cfg["hidden_dim"], cfg["n_layers"], cfg["n_heads"],
                    cfg.get("n_kv_heads") or cfg["n_heads"], cfg["vocab_size"], cfg["seq_len"],
                    cfg.get("rope_theta", 10000.0), cfg.get("norm_eps", 1e-5),
                    cfg.get("max_batch", 1), cfg.get("shared_classifier", 0),
                    cfg.get("max_prefill", 0), cfg.get("rolling_positions", 0),
                    cfg.get("layer_kernels", 0))


def _check(rc: int, h=None):
    if rc != L2_OK:
        raise L2Error(rc, l2_last_error(h))


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(t) -> int:
    """Device pointer of a torch tensor (or an int address)."""
    return t if isinstance(t, int) else t.data_ptr()


def l2_blob_floats(cfg: dict) -> int:
    return int(_lib.l2_blob_floats(ctypes.byref(make_config(cfg))))


def l2_create(cfg: dict, blob: np.ndarray):
    blob = np.ascontiguousarray(blob, dtype=np.float32)
    h = _P()
    c = make_config(cfg)
    _check(_lib.l2_create(ctypes.byref(c), blob.ctypes.data, blob.size, ctypes.byref(h)))
    return h


def l2_create_from_device(cfg: dict, d_blob, n_floats: int):
    """d_blob: device pointer (int) or a CUDA float32 torch tensor."""
    h = _P()
    c = make_config(cfg)
    _check(_lib.l2_create_from_device(ctypes.byref(c), _ptr(d_blob), n_floats, ctypes.byref(h)))
    return h


def l2_destroy(h) -> None:
    _lib.l2_destroy(h)


def l2_last_error(h=None) -> str:
    s = _lib.l2_last_error(h)
    return s.decode() if s else ""


def l2_reset(h, seq: int = -1) -> None:
    _check(_lib.l2_reset(h, seq), h)


def l2_forward(h, tokens, pos, vocab_size: int, want_logits: bool = True):
    tokens, pos = _i32(tokens).ravel(), _i32(pos).ravel()
    B = tokens.size
    if pos.size != B:
        raise ValueError("tokens and pos differ in length")
    out = np.empty((B, vocab_size), np.float32) if want_logits else None
    _check(_lib.l2_forward(h, tokens.ctypes.data, pos.ctypes.data, B,
                           out.ctypes.data if want_logits else None), h)
    return out


def l2_forward_device(h, d_tokens, d_pos, B: int, d_logits=None, stream=None) -> None:
    _check(_lib.l2_forward_device(h, _ptr(d_tokens), _ptr(d_pos), B,
                                  _ptr(d_logits) if d_logits is not None else None,
                                  _stream(stream)), h)


def l2_generate(h, prompt, steps: int) -> np.ndarray:
    prompt = _i32(prompt).ravel()
    out = np.empty(steps, np.int32)
    _check(_lib.l2_generate(h, prompt.ctypes.data, prompt.size, steps, out.ctypes.data), h)
    return out


def l2_generate_device(h, d_prompt, n_prompt: int, steps: int, d_out, stream=None) -> None:
    _check(_lib.l2_generate_device(h, _ptr(d_prompt), n_prompt, steps, _ptr(d_out),
                                   _stream(stream)), h)


def l2_prefill(h, tokens, pos0: int, vocab_size: int, want_logits: bool = True):
    """One causal prefill pass of sequence 0; returns logits [n][V] (or None)."""
    tokens = _i32(tokens).ravel()
    out = np.empty((tokens.size, vocab_size), np.float32) if want_logits else None
    _check(_lib.l2_prefill(h, tokens.ctypes.data, tokens.size, pos0,
                           out.ctypes.data if want_logits else None), h)
    return out


def l2_generate_prefill(h, prompt, steps: int) -> np.ndarray:
    prompt = _i32(prompt).ravel()
    out = np.empty(steps, np.int32)
    _check(_lib.l2_generate_prefill(h, prompt.ctypes.data, prompt.size, steps, out.ctypes.data),
           h)
    return out


def l2_generate_prefill_device(h, d_prompt, n_prompt: int, steps: int, d_out,
                               stream=None) -> None:
    _check(_lib.l2_generate_prefill_device(h, _ptr(d_prompt), n_prompt, steps, _ptr(d_out),
                                           _stream(stream)), h)


def l2_generate_sample(h, prompt, steps: int, temperature: float, topp: float,
                       uniforms) -> np.ndarray:
    prompt = _i32(prompt).ravel()
    u = np.ascontiguousarray(uniforms, dtype=np.float32).ravel()
    if u.size < steps:
        raise ValueError("need one uniform number per generated token")
    out = np.empty(steps, np.int32)
    _check(_lib.l2_generate_sample(h, prompt.ctypes.data, prompt.size, steps, temperature, topp,
                                   u.ctypes.data, out.ctypes.data), h)
    return out


def l2_generate_sample_device(h, d_prompt, n_prompt: int, steps: int, temperature: float,
                              topp: float, d_uniforms, d_out, stream=None) -> None:
    _check(_lib.l2_generate_sample_device(h, _ptr(d_prompt), n_prompt, steps, temperature, topp,
                                          _ptr(d_uniforms), _ptr(d_out), _stream(stream)), h)


def l2_generate_batch(h, prompts, lens, steps: int) -> np.ndarray:
    prompts, lens = _i32(prompts).ravel(), _i32(lens).ravel()
    out = np.empty((lens.size, steps), np.int32)
    _check(_lib.l2_generate_batch(h, prompts.ctypes.data, lens.ctypes.data, lens.size, steps,
                                  out.ctypes.data), h)
    return out


def l2_generate_batch_device(h, d_prompts, lens, steps: int, d_out, stream=None) -> None:
    """d_prompts, d_out: device buffers; lens: host lengths."""
    lens = _i32(lens).ravel()
    _check(_lib.l2_generate_batch_device(h, _ptr(d_prompts), lens.ctypes.data, lens.size, steps,
                                         _ptr(d_out), _stream(stream)), h)


def l2_generate_batch_prefill(h, prompts, lens, steps: int) -> np.ndarray:
    prompts, lens = _i32(prompts).ravel(), _i32(lens).ravel()
    out = np.empty((lens.size, steps), np.int32)
    _check(_lib.l2_generate_batch_prefill(h, prompts.ctypes.data, lens.ctypes.data, lens.size,
                                          steps, out.ctypes.data), h)
    return out


def l2_generate_batch_prefill_device(h, d_prompts, lens, steps: int, d_out, stream=None) -> None:
    """d_prompts, d_out: device buffers; lens: host lengths."""
    lens = _i32(lens).ravel()
    _check(_lib.l2_generate_batch_prefill_device(h, _ptr(d_prompts), lens.ctypes.data,
                                                 lens.size, steps, _ptr(d_out),
                                                 _stream(stream)), h)


def l2_generate_batch_sample(h, prompts, lens, steps: int, temperature: float, topp: float,
                             uniforms) -> np.ndarray:
    """uniforms: [B][steps] (sequence b's k-th draw at [b][k])."""
    prompts, lens = _i32(prompts).ravel(), _i32(lens).ravel()
    u = np.ascontiguousarray(uniforms, dtype=np.float32).ravel()
    if u.size < lens.size * steps:
        raise ValueError("need one uniform number per sequence and generated token")
    out = np.empty((lens.size, steps), np.int32)
    _check(_lib.l2_generate_batch_sample(h, prompts.ctypes.data, lens.ctypes.data, lens.size,
                                         steps, temperature, topp, u.ctypes.data,
                                         out.ctypes.data), h)
    return out


def l2_generate_batch_sample_device(h, d_prompts, lens, steps: int, temperature: float,
                                    topp: float, d_uniforms, d_out, stream=None) -> None:
    """d_prompts, d_uniforms, d_out: device buffers; lens: host lengths."""
    lens = _i32(lens).ravel()
    _check(_lib.l2_generate_batch_sample_device(h, _ptr(d_prompts), lens.ctypes.data, lens.size,
                                                steps, temperature, topp, _ptr(d_uniforms),
                                                _ptr(d_out), _stream(stream)), h)


def l2_status(h, stream=None) -> int:
    """Return code of the device work queued by the *_device calls (waits for
    `stream`); no exception, so that tests can compare codes."""
    return int(_lib.l2_status(h, _stream(stream)))


def l2_watchdog_check(h, spin_cycles: int) -> int:
    """Runs one bounded device wait that nothing completes; returns the C code
    (L2_ETIMEOUT when the wait gave up as designed)."""
    return int(_lib.l2_watchdog_check(h, int(spin_cycles)))


def l2_time_kernel(h, kind: int, pos: int, iters: int, stream=None) -> float:
    ms = ctypes.c_float()
    _check(_lib.l2_time_kernel(h, kind, pos, iters, _stream(stream), ctypes.byref(ms)), h)
    return float(ms.value)


def l2_kernel_bytes(h, kind: int, pos: int) -> float:
    return float(_lib.l2_kernel_bytes(h, kind, pos))


def l2_layer_kernels(h) -> int:
    return int(_lib.l2_layer_kernels(h))


def l2_gemm_tf32x3(d_A, d_W, d_C, M: int, N: int, K: int, iters: int = 0, stream=None):
    """C = A W^T through the 3xTF32 tensor-core kernel (device buffers). Returns
    the mean ms of `iters` timed launches (None when iters == 0)."""
    ms = ctypes.c_float()
    rc = _lib.l2_gemm_tf32x3(_ptr(d_A), _ptr(d_W), _ptr(d_C), M, N, K, iters,
                             ctypes.byref(ms) if iters else None, _stream(stream))
    if rc != L2_OK:
        raise L2Error(rc, "l2_gemm_tf32x3 failed")
    return float(ms.value) if iters else None


def l2_classify_greedy_noalloc(d_x, d_gain, d_wcls, dim: int, vocab: int, norm_eps: float,
                               d_token, d_logit=None, stream=None) -> int:
    """Greedy token of one hidden state; device buffers (torch tensors or ints).
    Returns the C return code (no exception: the call has no error text)."""
    return int(_lib.l2_classify_greedy_noalloc(
        _ptr(d_x), _ptr(d_gain), _ptr(d_wcls), dim, vocab, norm_eps, _ptr(d_token),
        _ptr(d_logit) if d_logit is not None else None, _stream(stream)))


def _stream(stream):
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream  # torch.cuda.Stream


class Decoder:
    """Owns one handle; methods forward to the C calls of the same names."""

    def __init__(self, cfg: dict, blob=None, d_blob=None):
        self.cfg = dict(cfg)
        if d_blob is not None:
            self.h = l2_create_from_device(cfg, d_blob, l2_blob_floats(cfg))
        else:
            self.h = l2_create(cfg, blob)

    def close(self):
        if getattr(self, "h", None):
            l2_destroy(self.h)
            self.h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        self.close()

    def forward(self, tokens, pos, want_logits: bool = True):
        return l2_forward(self.h, tokens, pos, self.cfg["vocab_size"], want_logits)

    def generate(self, prompt, steps: int) -> np.ndarray:
        return l2_generate(self.h, prompt, steps)

    def prefill(self, tokens, pos0: int = 0, want_logits: bool = True):
        return l2_prefill(self.h, tokens, pos0, self.cfg["vocab_size"], want_logits)

    def generate_prefill(self, prompt, steps: int) -> np.ndarray:
        return l2_generate_prefill(self.h, prompt, steps)

    def generate_sample(self, prompt, steps: int, temperature: float, topp: float,
                        uniforms) -> np.ndarray:
        return l2_generate_sample(self.h, prompt, steps, temperature, topp, uniforms)

    def generate_batch(self, prompts, lens, steps: int) -> np.ndarray:
        return l2_generate_batch(self.h, prompts, lens, steps)

    def generate_batch_prefill(self, prompts, lens, steps: int) -> np.ndarray:
        return l2_generate_batch_prefill(self.h, prompts, lens, steps)

    def generate_batch_sample(self, prompts, lens, steps: int, temperature: float, topp: float,
                              uniforms) -> np.ndarray:
        return l2_generate_batch_sample(self.h, prompts, lens, steps, temperature, topp, uniforms)

    def reset(self, seq: int = -1) -> None:
        l2_reset(self.h, seq)
