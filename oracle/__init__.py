"""TEST INFRASTRUCTURE ONLY: ctypes view of the plain C oracle (oracle.c).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product library never does, and the
oracle never touches the product library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
CFLAGS = ["-O2", "-fno-fast-math", "-ffp-contract=off", "-std=c99", "-fPIC", "-shared"]


class OracleConfig(ctypes.Structure):
    _fields_ = [("dim", ctypes.c_int32), ("hidden_dim", ctypes.c_int32),
                ("n_layers", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("vocab_size", ctypes.c_int32),
                ("seq_len", ctypes.c_int32), ("rope_theta", ctypes.c_float),
                ("norm_eps", ctypes.c_float), ("shared_classifier", ctypes.c_int32),
                ("rolling_cache", ctypes.c_int32)]


def build() -> str:
    """Compile liboracle.so in place (single-threaded, no contraction)."""
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_LIB = None


def lib():
    global _LIB
    if _LIB is not None:
        return _LIB
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest:
        build()
    _LIB = load(_LIB_PATH)
    return _LIB


def load(path: str):
    """Load a compiled oracle library and declare its signatures."""
    L = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32 = ctypes.c_int32
    L.oracle_blob_floats.restype = ctypes.c_size_t
    L.oracle_blob_floats.argtypes = [ctypes.POINTER(OracleConfig)]
    L.oracle_model_new.restype = P
    L.oracle_model_new.argtypes = [ctypes.POINTER(OracleConfig), P, ctypes.c_size_t]
    L.oracle_model_free.restype = None
    L.oracle_model_free.argtypes = [P]
    L.oracle_forward.restype = ctypes.c_int
    L.oracle_forward.argtypes = [P, i32, i32, P, P]
    L.oracle_generate.restype = ctypes.c_int
    L.oracle_generate.argtypes = [P, P, i32, i32, P, P]
    L.oracle_rmsnorm.restype = None
    L.oracle_rmsnorm.argtypes = [P, P, P, i32, ctypes.c_float]
    L.oracle_matvec.restype = None
    L.oracle_matvec.argtypes = [P, P, P, i32, i32]
    L.oracle_rope.restype = None
    L.oracle_rope.argtypes = [P, i32, i32, i32, ctypes.c_float]
    L.oracle_softmax.restype = None
    L.oracle_softmax.argtypes = [P, i32]
    L.oracle_attention_head.restype = None
    L.oracle_attention_head.argtypes = [P, P, P, P, i32, i32, i32]
    L.oracle_swiglu.restype = None
    L.oracle_swiglu.argtypes = [P, P, P, i32]
    L.oracle_argmax.restype = i32
    L.oracle_argmax.argtypes = [P, i32]
    L.oracle_sample.restype = i32
    L.oracle_sample.argtypes = [P, i32, ctypes.c_float, ctypes.c_float, ctypes.c_float, P]
    L.oracle_generate_sampled.restype = ctypes.c_int
    L.oracle_generate_sampled.argtypes = [P, P, i32, i32, ctypes.c_float, ctypes.c_float, P, P, P]
    return L


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def make_config(cfg: dict) -> OracleConfig:
    return OracleConfig(cfg["dim"], cfg["hidden_dim"], cfg["n_layers"], cfg["n_heads"],
                        cfg.get("n_kv_heads") or cfg["n_heads"], cfg["vocab_size"],
                        cfg["seq_len"], cfg.get("rope_theta", 10000.0),
                        cfg.get("norm_eps", 1e-5), cfg.get("shared_classifier", 0),
                        cfg.get("rolling_cache", 0))


def blob_floats(cfg: dict) -> int:
    c = make_config(cfg)
    return int(lib().oracle_blob_floats(ctypes.byref(c)))


class Model:
    """Oracle model over a blob (kept alive by this object) with its own KV cache."""

    def __init__(self, cfg: dict, blob: np.ndarray):
        self.cfg = dict(cfg)
        self._c = make_config(cfg)
        self.blob = blob if (blob.dtype == np.float32 and blob.flags["C_CONTIGUOUS"]) else _f32(blob)
        self._lib = lib()
        self._h = self._lib.oracle_model_new(ctypes.byref(self._c), self.blob.ctypes.data,
                                             self.blob.size)
        if not self._h:
            raise ValueError("oracle rejected the config or the blob size")

    def close(self):
        if getattr(self, "_h", None):
            self._lib.oracle_model_free(self._h)
            self._h = None

    __del__ = close

    def forward(self, token: int, pos: int, trace: bool = False):
        V, d, L = self.cfg["vocab_size"], self.cfg["dim"], self.cfg["n_layers"]
        logits = np.empty(V, dtype=np.float32)
        xt = np.empty((L + 1, d), dtype=np.float32) if trace else None
        rc = self._lib.oracle_forward(self._h, int(token), int(pos), logits.ctypes.data,
                                      xt.ctypes.data if trace else None)
        if rc != 0:
            raise ValueError(f"oracle_forward rejected token={token} pos={pos}")
        return (logits, xt) if trace else logits

    def generate(self, prompt, steps: int, trace: bool = False):
        prompt = np.ascontiguousarray(prompt, dtype=np.int32)
        out = np.empty(steps, dtype=np.int32)
        n_fwd = prompt.size + steps - 1
        lt = np.empty((n_fwd, self.cfg["vocab_size"]), dtype=np.float32) if trace else None
        rc = self._lib.oracle_generate(self._h, prompt.ctypes.data, prompt.size, steps,
                                       out.ctypes.data, lt.ctypes.data if trace else None)
        if rc != 0:
            raise ValueError("oracle_generate rejected its arguments")
        return (out, lt) if trace else out


    def generate_sampled(self, prompt, steps: int, temperature: float, topp: float, uniforms):
        """(tokens[steps], margins[steps]) drawn with oracle_sample."""
        prompt = np.ascontiguousarray(prompt, dtype=np.int32)
        u = _f32(uniforms)
        if u.size < steps:
            raise ValueError("need one uniform number per generated token")
        out = np.empty(steps, dtype=np.int32)
        mg = np.empty(steps, dtype=np.float32)
        rc = self._lib.oracle_generate_sampled(self._h, prompt.ctypes.data, prompt.size, steps,
                                               temperature, topp, u.ctypes.data, out.ctypes.data,
                                               mg.ctypes.data)
        if rc != 0:
            raise ValueError("oracle_generate_sampled rejected its arguments")
        return out, mg


# Building blocks (numpy in, numpy out).

def rmsnorm(x, g, eps: float = 1e-5) -> np.ndarray:
    x, g = _f32(x), _f32(g)
    out = np.empty_like(x)
    lib().oracle_rmsnorm(out.ctypes.data, x.ctypes.data, g.ctypes.data, x.size, eps)
    return out


def matvec(W, x) -> np.ndarray:
    W, x = _f32(W), _f32(x)
    rows, cols = W.shape
    y = np.empty(rows, dtype=np.float32)
    lib().oracle_matvec(y.ctypes.data, W.ctypes.data, x.ctypes.data, rows, cols)
    return y


def rope(v, n_heads: int, head_dim: int, pos: int, theta: float = 10000.0) -> np.ndarray:
    v = _f32(v).copy()
    lib().oracle_rope(v.ctypes.data, n_heads, head_dim, pos, theta)
    return v


def softmax(s) -> np.ndarray:
    s = _f32(s).copy()
    lib().oracle_softmax(s.ctypes.data, s.size)
    return s


def attention_head(q, k_rows, v_rows) -> np.ndarray:
    """q [hd]; k_rows, v_rows [n_pos][hd] (contiguous, stride hd)."""
    q, k_rows, v_rows = _f32(q), _f32(k_rows), _f32(v_rows)
    n_pos, hd = k_rows.shape
    out = np.empty(hd, dtype=np.float32)
    lib().oracle_attention_head(out.ctypes.data, q.ctypes.data, k_rows.ctypes.data,
                                v_rows.ctypes.data, hd, hd, n_pos)
    return out


def swiglu(h1, h3) -> np.ndarray:
    h1, h3 = _f32(h1), _f32(h3)
    out = np.empty_like(h1)
    lib().oracle_swiglu(out.ctypes.data, h1.ctypes.data, h3.ctypes.data, h1.size)
    return out


def argmax(v) -> int:
    v = _f32(v)
    return int(lib().oracle_argmax(v.ctypes.data, v.size))


def sample(logits, temperature: float, topp: float, u: float):
    """(token, margin) drawn from logits with oracle_sample."""
    v = _f32(logits)
    mg = ctypes.c_float()
    t = lib().oracle_sample(v.ctypes.data, v.size, temperature, topp, u, ctypes.byref(mg))
    return int(t), float(mg.value)
