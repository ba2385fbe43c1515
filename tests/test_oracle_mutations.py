"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a private copy of oracle.c (on the CPU, in a
temporary directory), builds it, swaps it in for the real oracle, and runs the
pin functions of test_oracle_components / test_oracle_model. At least one pin
must fail for every mutant; the unmodified source must pass them all.
"""
import os
import subprocess

import pytest

import oracle
import test_oracle_components as comp
import test_oracle_model as model
import test_oracle_sampling as samp

SRC = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()

MUTANTS = {
    "eps_outside_root": [("ss = ss / (float)n + eps;\n    const float inv = 1.0f / sqrtf(ss);",
                          "ss = ss / (float)n;\n    const float inv = 1.0f / (sqrtf(ss) + eps);")],
    "rmsnorm_drops_gain": [("out[i] = g[i] * (inv * x[i]);", "out[i] = inv * x[i];")],
    "matvec_transposed": [("acc += w[c] * x[c];", "acc += W[(size_t)c * (size_t)rows + r] * x[c];")],
    "rope_sign": [("p[0] = a * c - b * s;", "p[0] = a * c + b * s;")],
    "rope_frequency": [("-2.0 * (double)i / (double)head_dim", "-1.0 * (double)i / (double)head_dim")],
    "rope_on_q_only": [("oracle_rope(m->k, c->n_kv_heads, hd, pos, c->rope_theta);", "")],
    "softmax_no_max_shift": [("s[i] = expf(s[i] - mx);", "s[i] = expf(s[i]);")],
    "attention_unscaled": [("s[t] = dot / scale_div;", "s[t] = dot;")],
    "attention_skips_current_position": [("int32_t n_pos = pos + 1;",
                                          "int32_t n_pos = pos > 0 ? pos : 1;")],
    "kv_written_to_slot_zero": [("memcpy(kc + slot * kvd", "memcpy(kc + 0 * kvd")],
    "values_written_to_slot_zero": [("memcpy(vc + slot * kvd", "memcpy(vc + 0 * kvd")],
    "gqa_head_map_modulo": [("const int32_t kvh = h / group;",
                             "const int32_t kvh = h % c->n_kv_heads;")],
    "gate_up_swapped": [("const float z = h1[i];\n        hb[i] = (z / (1.0f + expf(-z))) * h3[i];",
                         "const float z = h3[i];\n        hb[i] = (z / (1.0f + expf(-z))) * h1[i];")],
    "attention_residual_dropped": [("oracle_matvec(m->y, m->wo + (size_t)l * d * d, m->att, d, d);\n"
                                    "        for (int32_t i = 0; i < d; ++i) m->x[i] += m->y[i];",
                                    "oracle_matvec(m->y, m->wo + (size_t)l * d * d, m->att, d, d);\n"
                                    "        for (int32_t i = 0; i < d; ++i) m->x[i] = m->y[i];")],
    "wo_of_layer_zero": [("m->wo + (size_t)l * d * d", "m->wo")],
    "ffn_norm_uses_attention_gain": [("m->g_ffn + (size_t)l * d", "m->g_att + (size_t)l * d")],
    "final_gain_skipped": [("oracle_rmsnorm(m->xb, m->x, m->g_final, d, c->norm_eps);",
                            "oracle_rmsnorm(m->xb, m->x, m->g_ffn, d, c->norm_eps);")],
    "final_norm_skipped": [("oracle_rmsnorm(m->xb, m->x, m->g_final, d, c->norm_eps);\n"
                            "    oracle_matvec(logits_out, m->wcls, m->xb,",
                            "oracle_rmsnorm(m->xb, m->x, m->g_final, d, c->norm_eps);\n"
                            "    oracle_matvec(logits_out, m->wcls, m->x,")],
    "argmax_last_tie": [("if (v[i] > v[best]) best = i;", "if (v[i] >= v[best]) best = i;")],
    "generate_feeds_prompt_late": [("token = (pos + 1 < n_prompt) ? prompt[pos + 1] : best;",
                                    "token = (pos < n_prompt) ? prompt[pos] : best;")],
    "rolling_rope_at_slot": [("oracle_rope(m->q, c->n_heads, hd, pos, c->rope_theta);",
                              "oracle_rope(m->q, c->n_heads, hd, pos % c->seq_len, c->rope_theta);"),
                             ("oracle_rope(m->k, c->n_kv_heads, hd, pos, c->rope_theta);",
                              "oracle_rope(m->k, c->n_kv_heads, hd, pos % c->seq_len, c->rope_theta);")],
    "rolling_slot_not_wrapped": [("const size_t slot = (size_t)pos % S;",
                                  "const size_t slot = (size_t)pos % S == 0 && pos > 0 ? S - 1 : (size_t)pos % S;")],
    "sample_temperature_multiplies": [("p[i] = expf((logits[i] - mx) / temperature);",
                                       "p[i] = expf((logits[i] - mx) * temperature);")],
    "sample_nucleus_drops_last": [("            if (cum >= target) {\n                v = s[k].p;",
                                   "            if (cum >= target) {\n                v = s[k > 0 ? k - 1 : 0].p;")],
    "sample_walks_rank_order": [("        if (p[i] < v) continue;\n        last = i;",
                                 "        if (p[i] < v) continue;\n        if (i == 0 && n > 1 && p[1] > p[0]) continue;\n        last = i;")],
    "sample_r_over_total": [("const float r = u * mass;", "const float r = u * total;")],
    "sample_prompt_positions": [("const int32_t k = pos - (n_prompt - 1);\n        float mg",
                                 "const int32_t k = pos - n_prompt + 1 > 0 ? pos - n_prompt + 1 : 0;\n        if (pos == n_prompt - 1) continue;\n        float mg")],
}


def _pins():
    fns = [getattr(comp, n) for n in dir(comp)
           if n.startswith("test_") and n != "test_argmax_last_and_first"]
    fns += [lambda: comp.test_argmax_last_and_first(n) for n in (1, 2, 31999)]
    fns += [model.test_handworked_two_layer_model, model.test_zero_layer_weights_closed_form,
            model.test_generate_feeds_prompt_then_greedy]
    fns += [getattr(samp, n) for n in dir(samp) if n.startswith("test_")]
    for p in model.test_incremental_decode_equals_full_causal_recompute.pytestmark[0].args[1]:
        fns.append(lambda p=p: model.test_incremental_decode_equals_full_causal_recompute(p))
    for p in model.test_rolling_cache_equals_windowed_full_recompute.pytestmark[0].args[1]:
        fns.append(lambda p=p: model.test_rolling_cache_equals_windowed_full_recompute(p))
    return fns


def _run_pins_with(lib_path):
    saved = oracle._LIB
    oracle._LIB = oracle.load(lib_path)
    failures = 0
    try:
        for fn in _pins():
            try:
                fn()
            except (AssertionError, ValueError):
                failures += 1
    finally:
        oracle._LIB = saved
    return failures


def _build(tmp_path, src, name):
    c = tmp_path / f"{name}.c"
    c.write_text(src)
    so = tmp_path / f"lib{name}.so"
    subprocess.check_call(["gcc", *oracle.CFLAGS, "-I", os.path.dirname(oracle.__file__),
                           str(c), "-o", str(so), "-lm"])
    return str(so)


def test_unmodified_source_passes_every_pin(tmp_path):
    assert _run_pins_with(_build(tmp_path, SRC, "clean")) == 0


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    src = SRC
    for old, new in MUTANTS[name]:
        assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
        src = src.replace(old, new)
    assert _run_pins_with(_build(tmp_path, src, name)) > 0, f"no pin caught {name}"
