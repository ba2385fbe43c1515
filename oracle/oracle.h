/*
 * oracle.h -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded C statement of one Llama-2 fp32 decode step,
 * written from the llama2.c pages. Only the test suite, the package's smoke
 * check and the benchmark's CPU-baseline leg may load it. The CUDA library
 * never includes, links or calls anything here, and nothing here comes from
 * the CUDA library.
 *
 * Sources (page titles as published):
 *  [P2] 新智元 article on llama2.c (m.greenbasetech.com), the paragraph before
 *       "感受魔力": a Llama 2 architecture is trained in PyTorch, its weights
 *       are saved as a raw binary file and a ~500-line C file runs it in fp32.
 *  [P4] "llama2.c｜Baby LLaMA-openAI维基百科" (openai.wiki), introduction:
 *       the Llama-2 architecture is hard-coded, fp32 only, one pure-C
 *       inference file; model shapes dim 288 / 6 layers / 6 heads and, under
 *       "训练示例", dim 512 / 8 layers / 8 heads / context 1024.
 *       "未排序的待办事项": the KV cache bounds decoding to max_seq_len.
 * The pages name the architecture but never write its formulas out. Each
 * function below states the reading it takes of "Llama 2 architecture".
 *
 * Parity status: every function here is pinned by the tests under
 * tests/test_oracle_*.py (closed forms, invariants, a hand-worked model and a
 * brute-force full causal recompute); see the header of oracle.c.
 */
#ifndef L2_ORACLE_H
#define L2_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int32_t dim, hidden_dim, n_layers, n_heads, n_kv_heads, vocab_size, seq_len;
    float rope_theta, norm_eps;
    int32_t shared_classifier; /* 1: the classifier is the embedding table */
    int32_t rolling_cache;     /* 1: positions beyond seq_len keep the last seq_len */
} oracle_config;

typedef struct oracle_model oracle_model;

/* Number of floats in a weight blob for cfg (layout in oracle.c). */
size_t oracle_blob_floats(const oracle_config* cfg);

/* Maps blob (caller keeps it alive) and allocates a zeroed KV cache. NULL on a
 * bad config or size mismatch. */
oracle_model* oracle_model_new(const oracle_config* cfg, const float* blob, size_t blob_floats);
void oracle_model_free(oracle_model* m);

/* One decode step: token at position pos, writes KV slot pos, reads slots
 * 0..pos. With rolling_cache (decoding beyond seq_len, a to-do item of the
 * openai.wiki page, "未排序的待办事项"): position pos (any pos >= 0) writes
 * slot pos % seq_len and attends, in position order, over positions
 * max(0, pos - seq_len + 1) .. pos; RoPE uses the absolute position. logits_out: [vocab]. x_trace (nullable): [n_layers + 1][dim], the
 * residual stream after the embedding and after each layer. Returns 0, or -1
 * on a token or position out of range. */
int oracle_forward(oracle_model* m, int32_t token, int32_t pos, float* logits_out,
                   float* x_trace);

/* Greedy decode: forwards at pos 0 .. n_prompt + steps - 2; out_tokens[k] is
 * the argmax at pos n_prompt - 1 + k. logits_trace (nullable):
 * [n_prompt + steps - 1][vocab]. Returns 0 or -1. */
int oracle_generate(oracle_model* m, const int32_t* prompt, int32_t n_prompt, int32_t steps,
                    int32_t* out_tokens, float* logits_trace);

/* Sampling instead of greedy (see oracle.c for the rule): the token drawn
 * from logits[n] at the given temperature and top-p with the uniform number
 * u in [0, 1); margin_out (nullable) receives how close the draw was to a
 * decision boundary, relative to the nucleus mass. */
int32_t oracle_sample(const float* logits, int32_t n, float temperature, float topp, float u,
                      float* margin_out);

/* oracle_generate drawing every generated token with oracle_sample and
 * uniforms[k] (k = 0 .. steps-1); margins_out (nullable): [steps]. */
int oracle_generate_sampled(oracle_model* m, const int32_t* prompt, int32_t n_prompt,
                            int32_t steps, float temperature, float topp, const float* uniforms,
                            int32_t* out_tokens, float* margins_out);

/* Building blocks, exported so that tests can pin each one. */
void oracle_rmsnorm(float* out, const float* x, const float* g, int32_t n, float eps);
void oracle_matvec(float* y, const float* W, const float* x, int32_t rows, int32_t cols);
void oracle_rope(float* v, int32_t n_heads, int32_t head_dim, int32_t pos, float theta);
void oracle_softmax(float* s, int32_t n);
void oracle_attention_head(float* out, const float* q, const float* k_cache, const float* v_cache,
                           int32_t row_stride, int32_t head_dim, int32_t n_pos);
void oracle_swiglu(float* hb, const float* h1, const float* h3, int32_t n);
int32_t oracle_argmax(const float* v, int32_t n);

#ifdef __cplusplus
}
#endif
#endif
