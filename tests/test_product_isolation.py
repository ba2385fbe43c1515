"""The product path never touches the oracle (CPU, static).

The oracle is test infrastructure: the package under
llama_fp32_token_decode_b300/ (Python binding, build script, CUDA sources)
must not import, load or link anything under oracle/, and the oracle's C
sources must not include the package's headers (the two share no code)."""
import os
import re
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "llama_fp32_token_decode_b300")


def _files(top, exts):
    for d, _, names in os.walk(top):
        if "__pycache__" in d:
            continue
        for n in names:
            if n.endswith(exts):
                yield os.path.join(d, n)


def test_package_sources_do_not_reach_the_oracle():
    pat = re.compile(r"\boracle\b|liboracle|oracle\.h")
    hits = []
    for f in _files(PKG, (".py", ".cu", ".cuh", ".h", ".c", ".cpp")):
        for i, line in enumerate(open(f, encoding="utf-8"), 1):
            if pat.search(line):
                hits.append(f"{os.path.relpath(f, ROOT)}:{i}: {line.strip()}")
    assert not hits, "\n".join(hits)


def test_oracle_sources_do_not_include_the_package():
    pat = re.compile(r"#\s*include\s*[<\"](?!std|math|string|stdio|stdlib|stddef|float|limits)")
    for f in _files(os.path.join(ROOT, "oracle"), (".c", ".h")):
        for line in open(f, encoding="utf-8"):
            m = pat.search(line)
            if m:
                assert "l2decode" not in line and "l2_internal" not in line, line
                assert "csrc" not in line, line


def test_built_library_does_not_link_the_oracle():
    lib = os.path.join(PKG, "libl2decode.so")
    if not os.path.exists(lib):
        import pytest
        pytest.skip("library not built")
    out = subprocess.run(["ldd", lib], capture_output=True, text=True).stdout
    assert "oracle" not in out and "synth" not in out, out
