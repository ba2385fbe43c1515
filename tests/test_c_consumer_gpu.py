"""A C program decodes through the library's C ABI on the GPU.

Every other GPU test reaches the library through the Python binding (ctypes):
the same ABI, but not the way a C caller uses it. Here a C99 program compiled
against include/l2decode.h alone creates a handle from a host blob, runs a
greedy generation and teacher-forced forwards, and writes the tokens and
logits to a file; they must match the oracle (logits within relative L2
1e-4, tokens equal up to the oracle's first near-tie).
"""
import os
import subprocess

import numpy as np
import pytest

import synth
from parity_util import REL_L2_TOL, config, first_near_tie, oracle_run, rel_l2

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_PROGRAM = r"""
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include "l2decode.h"

int main(int argc, char** argv) {
    if (argc != 3) return 2;
    l2_config c;
    memset(&c, 0, sizeof c);
    c.dim = 64; c.hidden_dim = 160; c.n_layers = 2; c.n_heads = 4; c.n_kv_heads = 4;
    c.vocab_size = 1000; c.seq_len = 32; c.rope_theta = 10000.0f; c.norm_eps = 1e-5f;
    c.max_batch = 1;
    const size_t n = l2_blob_floats(&c);
    float* blob = (float*)malloc(n * sizeof(float));
    FILE* f = fopen(argv[1], "rb");
    if (!blob || !f || fread(blob, sizeof(float), n, f) != n) return 3;
    fclose(f);
    l2_handle* h = NULL;
    int rc = l2_create(&c, blob, n, &h);
    free(blob);  /* the handle keeps its own copy */
    if (rc != L2_OK) {
        fprintf(stderr, "create: %d %s\n", rc, l2_last_error(NULL));
        return 4;
    }
    const int32_t prompt[4] = {5, 9, 13, 2};
    int32_t out[20];
    rc = l2_generate(h, prompt, 4, 20, out);
    if (rc != L2_OK) {
        fprintf(stderr, "generate: %d %s\n", rc, l2_last_error(h));
        return 5;
    }
    float* lg = (float*)malloc(4 * 1000 * sizeof(float));
    for (int32_t p = 0; p < 4 && lg; ++p) {
        rc = l2_forward(h, &prompt[p], &p, 1, lg + (size_t)p * 1000);
        if (rc != L2_OK) {
            fprintf(stderr, "forward: %d %s\n", rc, l2_last_error(h));
            return 6;
        }
    }
    f = fopen(argv[2], "wb");
    if (!f || !lg) return 7;
    fwrite(out, sizeof(int32_t), 20, f);
    fwrite(lg, sizeof(float), 4 * 1000, f);
    fclose(f);
    free(lg);
    l2_destroy(h);
    return 0;
}
"""


def test_c_program_decodes_through_the_abi(tmp_path):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import llama_fp32_token_decode_b300 as l2
    cfg = config(dim=64, hidden_dim=160, n_layers=2, n_heads=4, vocab_size=1000, seq_len=32)
    blob = synth.make_blob(cfg, 61, std=0.05)
    assert blob.size == l2.l2_blob_floats(cfg)
    blob_path = tmp_path / "blob.f32"
    blob.tofile(blob_path)
    src = tmp_path / "decode.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "decode"
    lib_dir = os.path.dirname(l2.LIB_PATH)
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I",
                        os.path.join(ROOT, "include"), str(src), "-o", str(exe), "-L", lib_dir,
                        "-l:libl2decode.so", "-Wl,-rpath," + lib_dir],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out_path = tmp_path / "out.bin"
    r = subprocess.run([str(exe), str(blob_path), str(out_path)], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, (r.returncode, r.stderr)
    raw = np.fromfile(out_path, dtype=np.uint8)
    tokens = raw[:80].view(np.int32)
    logits = raw[80:].view(np.float32).reshape(4, 1000)
    prompt = np.array([5, 9, 13, 2], np.int32)
    toks, consumed, trace = oracle_run(cfg, blob, prompt, 20)
    for p in range(4):
        e = rel_l2(logits[p], trace[p])
        assert e <= REL_L2_TOL, f"pos {p}: rel-L2 {e:.3e}"
    k = first_near_tie(trace, len(prompt))
    n = min(k + 1, 20)
    np.testing.assert_array_equal(tokens[:n], toks[:n])
