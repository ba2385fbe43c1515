"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every symbol the header declares, agrees with the documented blob size, and
rejects bad arguments before touching the device."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def l2():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "l2build", os.path.join(ROOT, "llama_fp32_token_decode_b300", "build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    b.build()
    import llama_fp32_token_decode_b300 as m
    return m


def _declared():
    txt = open(os.path.join(ROOT, "include", "l2decode.h")).read()
    return sorted(set(re.findall(r"L2_API\s+[\w\s\*]+?\b(l2_\w+)\s*\(", txt)))


def test_header_declares_and_library_exports_every_symbol(l2):
    names = _declared()
    assert len(names) >= 12
    lib = ctypes.CDLL(l2.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(l2.EXPORTS) == names


def test_blob_size_agrees_with_generator_and_oracle(l2):
    import oracle
    import synth
    for name in synth.WORKLOADS:
        cfg = synth.model_config(synth.workload(name))
        n = l2.l2_blob_floats(cfg)
        assert n == synth.blob_floats(cfg) == oracle.blob_floats(cfg), name
        tied = dict(cfg, shared_classifier=1)
        assert l2.l2_blob_floats(tied) == n - cfg["vocab_size"] * cfg["dim"]


def test_workload_blob_sizes_match_the_shapes():
    import synth
    # untied 15M-shape model: 24.4M floats (97.6 MB)
    assert synth.blob_floats(synth.model_config(synth.workload("15m"))) == 24407712
    # 7B shape: 6.74 G floats (26.95 GB)
    n7 = synth.blob_floats(synth.model_config(synth.workload("7b")))
    assert abs(n7 * 4 / 1e9 - 26.95) < 0.01


BAD = [dict(dim=0), dict(dim=65), dict(n_heads=5), dict(n_kv_heads=3), dict(dim=60, n_heads=20),
       dict(hidden_dim=162), dict(max_batch=0), dict(max_batch=4096), dict(seq_len=-1),
       dict(dim=66, n_heads=2), dict(shared_classifier=2), dict(norm_eps=-1.0)]


@pytest.mark.parametrize("bad", BAD)
def test_invalid_config_rejected(l2, bad):
    from parity_util import config
    cfg = config(**bad)
    assert l2.l2_blob_floats(cfg) == 0
    with pytest.raises(l2.L2Error) as e:
        l2.l2_create(cfg, np.zeros(16, np.float32))
    assert e.value.code == l2.L2_EINVAL
    assert "invalid config" in l2.l2_last_error(None)


def test_blob_size_mismatch(l2):
    from parity_util import config
    cfg = config()
    n = l2.l2_blob_floats(cfg)
    with pytest.raises(l2.L2Error) as e:
        l2.l2_create(cfg, np.zeros(n - 1, np.float32))
    assert e.value.code == l2.L2_EBLOB


def test_null_handle_rejected(l2):
    lib = l2._lib
    assert lib.l2_forward(None, None, None, 1, None) == l2.L2_EINVAL
    assert lib.l2_generate(None, None, 1, 1, None) == l2.L2_EINVAL
    assert lib.l2_generate_batch(None, None, None, 1, 1, None) == l2.L2_EINVAL
    assert lib.l2_reset(None, -1) == l2.L2_EINVAL
    assert lib.l2_kernel_bytes(None, 0, 0) == 0.0
    lib.l2_destroy(None)


def test_create_without_device_reports_cuda_error(l2):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    from parity_util import config
    cfg = config()
    with pytest.raises(l2.L2Error) as e:
        l2.l2_create(cfg, np.zeros(l2.l2_blob_floats(cfg), np.float32))
    assert e.value.code in (l2.L2_ECUDA, l2.L2_ENOMEM)


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "l2decode.h"

int main(void) {
    /* the 15M workload shape, untied classifier */
    l2_config c;
    memset(&c, 0, sizeof c);
    c.dim = 288; c.hidden_dim = 768; c.n_layers = 6; c.n_heads = 6; c.n_kv_heads = 6;
    c.vocab_size = 32000; c.seq_len = 256; c.rope_theta = 10000.0f; c.norm_eps = 1e-5f;
    c.max_batch = 1;
    printf("%zu\n", l2_blob_floats(&c));
    l2_handle* h = (l2_handle*)&c;  /* must be overwritten with NULL on failure */
    c.dim = 65;                       /* not a multiple of n_heads */
    int rc = l2_create(&c, NULL, 0, &h);
    printf("%d %d\n", rc, h == NULL);
    printf("%s\n", l2_last_error(NULL));
    printf("%d\n", l2_reset(NULL, -1));
    l2_destroy(NULL);
    return 0;
}
"""


@pytest.mark.parametrize("lang", ["c", "c++"])
def test_header_is_plain_c_and_links_from_c(l2, tmp_path, lang):
    # a C (and a C++) consumer compiles against the header alone with strict
    # warnings, links the in-tree library and calls its host-only paths
    import subprocess
    src = tmp_path / ("main.c" if lang == "c" else "main.cpp")
    src.write_text(C_PROGRAM)
    exe = tmp_path / "main"
    lib_dir = os.path.dirname(l2.LIB_PATH)
    cc = ["gcc", "-std=c99"] if lang == "c" else ["g++", "-std=c++17"]
    cmd = cc + ["-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                str(src), "-o", str(exe), "-L", lib_dir, "-l:libl2decode.so",
                "-Wl,-rpath," + lib_dir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    lines = r.stdout.splitlines()
    assert int(lines[0]) == 24407712
    assert lines[1] == f"{l2.L2_EINVAL} 1"
    assert "invalid config" in lines[2]
    assert int(lines[3]) == l2.L2_EINVAL
