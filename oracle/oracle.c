/*
 * oracle.c -- TEST INFRASTRUCTURE ONLY (see oracle.h). Plain C99, one thread,
 * fp32 storage and fp32 accumulation in sequential loop order, because the
 * pages fix fp32 for the engine ([P2] paragraph before "感受魔力"; [P4]
 * introduction, "坚持使用fp32"). Build with
 *   gcc -O2 -fno-fast-math -ffp-contract=off -fPIC -shared oracle.c -lm
 * so that no multiply-add is contracted and no operation is reordered.
 *
 * Blob layout (the pages say only "raw binary file"; this is the documented
 * order the boundary also reads), fp32, contiguous:
 *   E[V][d], g_att[L][d], Wq[L][d][d], Wk[L][kvd][d], Wv[L][kvd][d],
 *   Wo[L][d][d], g_ffn[L][d], W1[L][F][d], W2[L][d][F], W3[L][F][d],
 *   g_final[d], Wcls[V][d] (absent when the classifier is shared with E).
 * Every matrix is row-major [out][in] and acts as y = W x.
 *
 * Readings of what the pages leave open (each also listed in the design notes):
 *  - RMSNorm: out_i = g_i * (x_i / sqrt(mean(x^2) + eps)), eps inside the root.
 *  - RoPE: adjacent pairs (2i, 2i+1) of each head, angle pos * theta^(-2i/hd),
 *    angle, cosine and sine in double, rounded to float before the rotation.
 *  - Attention: scores (q . k) / sqrt(hd) over positions 0..pos (causal),
 *    max-subtracted softmax, weighted sum of values; query head h reads kv
 *    head h / (n_heads / n_kv_heads).
 *  - FFN: hb = silu(W1 x) * (W3 x), silu(z) = z / (1 + exp(-z)); W1 is the
 *    gate, W3 the up projection, W2 the down projection.
 *  - Greedy: the lowest index wins a tie.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

struct oracle_model {
    oracle_config c;
    int32_t hd, kvd;
    /* views into the caller's blob */
    const float *emb, *g_att, *wq, *wk, *wv, *wo, *g_ffn, *w1, *w2, *w3, *g_final, *wcls;
    /* KV cache [L][S][kvd] each */
    float *k_cache, *v_cache;
    /* run state */
    float *x, *xb, *q, *k, *v, *att, *y, *h1, *h3, *hb, *scores;
    /* rolling cache: the attended window's K and V rows in position order [S][kvd] */
    float *kwin, *vwin;
};

static int config_ok(const oracle_config* c) {
    if (c->dim <= 0 || c->hidden_dim <= 0 || c->n_layers <= 0 || c->n_heads <= 0 ||
        c->n_kv_heads <= 0 || c->vocab_size <= 0 || c->seq_len <= 0)
        return 0;
    if (c->dim % c->n_heads != 0) return 0;
    if (c->n_heads % c->n_kv_heads != 0) return 0;
    if ((c->dim / c->n_heads) % 2 != 0) return 0;
    return 1;
}

size_t oracle_blob_floats(const oracle_config* c) {
    if (!config_ok(c)) return 0;
    const size_t d = (size_t)c->dim, F = (size_t)c->hidden_dim, L = (size_t)c->n_layers;
    const size_t V = (size_t)c->vocab_size;
    const size_t kvd = (size_t)c->n_kv_heads * (d / (size_t)c->n_heads);
    size_t n = V * d;                          /* E */
    n += L * d;                                /* g_att */
    n += L * d * d + 2 * L * kvd * d;          /* Wq, Wk, Wv */
    n += L * d * d;                            /* Wo */
    n += L * d;                                /* g_ffn */
    n += 3 * L * F * d;                        /* W1, W2, W3 */
    n += d;                                    /* g_final */
    if (!c->shared_classifier) n += V * d;     /* Wcls */
    return n;
}

oracle_model* oracle_model_new(const oracle_config* c, const float* blob, size_t blob_floats) {
    if (!config_ok(c) || blob == NULL || blob_floats != oracle_blob_floats(c)) return NULL;
    oracle_model* m = (oracle_model*)calloc(1, sizeof(oracle_model));
    if (!m) return NULL;
    m->c = *c;
    m->hd = c->dim / c->n_heads;
    m->kvd = c->n_kv_heads * m->hd;
    const size_t d = (size_t)c->dim, F = (size_t)c->hidden_dim, L = (size_t)c->n_layers;
    const size_t V = (size_t)c->vocab_size, kvd = (size_t)m->kvd;
    const float* p = blob;
    m->emb = p;     p += V * d;
    m->g_att = p;   p += L * d;
    m->wq = p;      p += L * d * d;
    m->wk = p;      p += L * kvd * d;
    m->wv = p;      p += L * kvd * d;
    m->wo = p;      p += L * d * d;
    m->g_ffn = p;   p += L * d;
    m->w1 = p;      p += L * F * d;
    m->w2 = p;      p += L * d * F;
    m->w3 = p;      p += L * F * d;
    m->g_final = p; p += d;
    m->wcls = c->shared_classifier ? m->emb : p;

    const size_t cache = L * (size_t)c->seq_len * kvd;
    m->k_cache = (float*)calloc(cache, sizeof(float));
    m->v_cache = (float*)calloc(cache, sizeof(float));
    m->x = (float*)calloc(d, sizeof(float));
    m->xb = (float*)calloc(d, sizeof(float));
    m->q = (float*)calloc(d, sizeof(float));
    m->k = (float*)calloc(kvd, sizeof(float));
    m->v = (float*)calloc(kvd, sizeof(float));
    m->att = (float*)calloc(d, sizeof(float));
    m->y = (float*)calloc(d, sizeof(float));
    m->h1 = (float*)calloc(F, sizeof(float));
    m->h3 = (float*)calloc(F, sizeof(float));
    m->hb = (float*)calloc(F, sizeof(float));
    m->scores = (float*)calloc((size_t)c->seq_len, sizeof(float));
    m->kwin = (float*)calloc((size_t)c->seq_len * kvd, sizeof(float));
    m->vwin = (float*)calloc((size_t)c->seq_len * kvd, sizeof(float));
    if (!m->k_cache || !m->v_cache || !m->x || !m->xb || !m->q || !m->k || !m->v || !m->att ||
        !m->y || !m->h1 || !m->h3 || !m->hb || !m->scores || !m->kwin || !m->vwin) {
        oracle_model_free(m);
        return NULL;
    }
    return m;
}

void oracle_model_free(oracle_model* m) {
    if (!m) return;
    free(m->k_cache); free(m->v_cache);
    free(m->x); free(m->xb); free(m->q); free(m->k); free(m->v); free(m->att); free(m->y);
    free(m->h1); free(m->h3); free(m->hb); free(m->scores);
    free(m->kwin); free(m->vwin);
    free(m);
}

/* RMSNorm of the Llama 2 architecture named in [P2]/[P4]:
 * out_i = g_i * (x_i / sqrt(sum(x^2) / n + eps)). */
void oracle_rmsnorm(float* out, const float* x, const float* g, int32_t n, float eps) {
    float ss = 0.0f;
    for (int32_t i = 0; i < n; ++i) ss += x[i] * x[i];
    ss = ss / (float)n + eps;
    const float inv = 1.0f / sqrtf(ss);
    for (int32_t i = 0; i < n; ++i) out[i] = g[i] * (inv * x[i]);
}

/* y = W x with W row-major [rows][cols]: the fp32 projection of the engine. */
void oracle_matvec(float* y, const float* W, const float* x, int32_t rows, int32_t cols) {
    for (int32_t r = 0; r < rows; ++r) {
        const float* w = W + (size_t)r * (size_t)cols;
        float acc = 0.0f;
        for (int32_t c = 0; c < cols; ++c) acc += w[c] * x[c];
        y[r] = acc;
    }
}

/* Rotary position embedding on n_heads heads of head_dim each: the pair
 * (v[2i], v[2i+1]) of every head turns by pos * theta^(-2i/head_dim). */
void oracle_rope(float* v, int32_t n_heads, int32_t head_dim, int32_t pos, float theta) {
    for (int32_t i = 0; i < head_dim / 2; ++i) {
        const double freq = pow((double)theta, -2.0 * (double)i / (double)head_dim);
        const double angle = (double)pos * freq;
        const float c = (float)cos(angle), s = (float)sin(angle);
        for (int32_t h = 0; h < n_heads; ++h) {
            float* p = v + (size_t)h * (size_t)head_dim + 2 * i;
            const float a = p[0], b = p[1];
            p[0] = a * c - b * s;
            p[1] = a * s + b * c;
        }
    }
}

/* Softmax in place: subtract the maximum, exponentiate, divide by the sum. */
void oracle_softmax(float* s, int32_t n) {
    float mx = s[0];
    for (int32_t i = 1; i < n; ++i)
        if (s[i] > mx) mx = s[i];
    float sum = 0.0f;
    for (int32_t i = 0; i < n; ++i) {
        s[i] = expf(s[i] - mx);
        sum += s[i];
    }
    for (int32_t i = 0; i < n; ++i) s[i] = s[i] / sum;
}

/* One head of causal attention over cached positions 0 .. n_pos-1:
 * out = sum_t softmax_t((q . k_t) / sqrt(hd)) v_t. k_cache / v_cache point at
 * the head's first element of position 0; row_stride is the distance between
 * positions (kvd). */
void oracle_attention_head(float* out, const float* q, const float* k_cache, const float* v_cache,
                           int32_t row_stride, int32_t head_dim, int32_t n_pos) {
    float* s = (float*)malloc((size_t)n_pos * sizeof(float));
    if (!s) return;
    const float scale_div = sqrtf((float)head_dim);
    for (int32_t t = 0; t < n_pos; ++t) {
        const float* k = k_cache + (size_t)t * (size_t)row_stride;
        float dot = 0.0f;
        for (int32_t i = 0; i < head_dim; ++i) dot += q[i] * k[i];
        s[t] = dot / scale_div;
    }
    oracle_softmax(s, n_pos);
    for (int32_t i = 0; i < head_dim; ++i) out[i] = 0.0f;
    for (int32_t t = 0; t < n_pos; ++t) {
        const float* v = v_cache + (size_t)t * (size_t)row_stride;
        for (int32_t i = 0; i < head_dim; ++i) out[i] += s[t] * v[i];
    }
    free(s);
}

/* SwiGLU gate: hb_i = silu(h1_i) * h3_i, silu(z) = z / (1 + exp(-z)). */
void oracle_swiglu(float* hb, const float* h1, const float* h3, int32_t n) {
    for (int32_t i = 0; i < n; ++i) {
        const float z = h1[i];
        hb[i] = (z / (1.0f + expf(-z))) * h3[i];
    }
}

/* Greedy choice of the next token; the lowest index wins a tie. */
int32_t oracle_argmax(const float* v, int32_t n) {
    int32_t best = 0;
    for (int32_t i = 1; i < n; ++i)
        if (v[i] > v[best]) best = i;
    return best;
}

/* Sampling instead of the greedy choice. The pages print sampled stories and
 * mention the engine's "C sampling code" (openai.wiki, "未排序的待办事项")
 * without giving its rule; the reading taken here:
 *   temperature <= 0: the greedy choice (lowest index of the largest logit);
 *   otherwise p_i = expf((l_i - max_j l_j) / temperature) in fp32, total =
 *   their sum; with 0 < topp < 1 the nucleus is the smallest set of highest
 *   p (sorted by p, ties by lower index) whose sum reaches topp * total,
 *   widened to every token whose p equals the last one taken; otherwise the
 *   nucleus is every token. With r = u * (sum of p over the nucleus), the
 *   sampled token is the first nucleus member, in increasing index order,
 *   whose running sum exceeds r (the last member if none does).
 * u in [0, 1) is the uniform random number of this draw, supplied by the
 * caller. Sums are sequential fp32. margin_out (nullable) receives the
 * smallest distance, relative to the nucleus mass, between a running sum and
 * the value it was compared with (r, or topp * total): a decision with a tiny
 * margin can flip under a different summation order. */
typedef struct {
    float p;
    int32_t i;
} prob_index;

static int by_p_desc(const void* a, const void* b) {
    const prob_index* x = (const prob_index*)a;
    const prob_index* y = (const prob_index*)b;
    if (x->p > y->p) return -1;
    if (x->p < y->p) return 1;
    return (x->i > y->i) - (x->i < y->i);
}

int32_t oracle_sample(const float* logits, int32_t n, float temperature, float topp, float u,
                      float* margin_out) {
    if (margin_out) *margin_out = 1.0f;
    if (!(temperature > 0.0f)) return oracle_argmax(logits, n);
    float mx = logits[0];
    for (int32_t i = 1; i < n; ++i)
        if (logits[i] > mx) mx = logits[i];
    float* p = (float*)malloc(sizeof(float) * (size_t)n);
    float total = 0.0f;
    for (int32_t i = 0; i < n; ++i) {
        p[i] = expf((logits[i] - mx) / temperature);
        total += p[i];
    }
    float v = 0.0f;  /* nucleus: p >= v */
    float margin = 1.0f;
    if (topp > 0.0f && topp < 1.0f) {
        prob_index* s = (prob_index*)malloc(sizeof(prob_index) * (size_t)n);
        for (int32_t i = 0; i < n; ++i) {
            s[i].p = p[i];
            s[i].i = i;
        }
        qsort(s, (size_t)n, sizeof(prob_index), by_p_desc);
        const float target = topp * total;
        float cum = 0.0f;
        v = s[n - 1].p;
        for (int32_t k = 0; k < n; ++k) {
            const float before = cum;
            cum += s[k].p;
            if (cum >= target) {
                v = s[k].p;
                margin = fminf(cum - target, target - before) / total;
                break;
            }
        }
        free(s);
    }
    float mass = 0.0f;
    for (int32_t i = 0; i < n; ++i)
        if (p[i] >= v) mass += p[i];
    const float r = u * mass;
    float cum = 0.0f;
    int32_t pick = -1, last = 0;
    for (int32_t i = 0; i < n; ++i) {
        if (p[i] < v) continue;
        last = i;
        const float before = cum;
        cum += p[i];
        if (cum > r) {
            pick = i;
            margin = fminf(margin, fminf(cum - r, r - before) / mass);
            break;
        }
    }
    if (pick < 0) {
        pick = last;
        margin = 0.0f;
    }
    free(p);
    if (margin_out) *margin_out = margin;
    return pick;
}

/* oracle_generate with sampling: the token chosen at position p >= n_prompt-1
 * is oracle_sample(logits, temperature, topp, uniforms[p - (n_prompt - 1)]).
 * margins_out (nullable): [steps], the margin of each draw. */
int oracle_generate_sampled(oracle_model* m, const int32_t* prompt, int32_t n_prompt,
                            int32_t steps, float temperature, float topp, const float* uniforms,
                            int32_t* out_tokens, float* margins_out) {
    const oracle_config* c = &m->c;
    if (n_prompt < 1 || steps < 1) return -1;
    if (!c->rolling_cache && n_prompt + steps - 1 > c->seq_len) return -1;
    float* logits = (float*)malloc(sizeof(float) * (size_t)c->vocab_size);
    int32_t token = prompt[0];
    for (int32_t pos = 0; pos < n_prompt + steps - 1; ++pos) {
        if (oracle_forward(m, token, pos, logits, NULL) != 0) {
            free(logits);
            return -1;
        }
        if (pos + 1 < n_prompt) {
            token = prompt[pos + 1];
            continue;
        }
        const int32_t k = pos - (n_prompt - 1);
        float mg = 1.0f;
        const int32_t pick =
            oracle_sample(logits, c->vocab_size, temperature, topp, uniforms[k], &mg);
        out_tokens[k] = pick;
        if (margins_out) margins_out[k] = mg;
        token = pick;
    }
    free(logits);
    return 0;
}

/* The decode step, in the order the Llama-2 architecture applies it. */
int oracle_forward(oracle_model* m, int32_t token, int32_t pos, float* logits_out,
                   float* x_trace) {
    const oracle_config* c = &m->c;
    if (token < 0 || token >= c->vocab_size || pos < 0) return -1;
    if (!c->rolling_cache && pos >= c->seq_len) return -1;
    const int32_t d = c->dim, F = c->hidden_dim, hd = m->hd, kvd = m->kvd;
    const int32_t group = c->n_heads / c->n_kv_heads;
    const size_t S = (size_t)c->seq_len;

    /* embedding row */
    memcpy(m->x, m->emb + (size_t)token * (size_t)d, (size_t)d * sizeof(float));
    if (x_trace) memcpy(x_trace, m->x, (size_t)d * sizeof(float));

    for (int32_t l = 0; l < c->n_layers; ++l) {
        /* attention block */
        oracle_rmsnorm(m->xb, m->x, m->g_att + (size_t)l * d, d, c->norm_eps);
        oracle_matvec(m->q, m->wq + (size_t)l * d * d, m->xb, d, d);
        oracle_matvec(m->k, m->wk + (size_t)l * kvd * d, m->xb, kvd, d);
        oracle_matvec(m->v, m->wv + (size_t)l * kvd * d, m->xb, kvd, d);
        oracle_rope(m->q, c->n_heads, hd, pos, c->rope_theta);
        oracle_rope(m->k, c->n_kv_heads, hd, pos, c->rope_theta);

        float* kc = m->k_cache + (size_t)l * S * (size_t)kvd;
        float* vc = m->v_cache + (size_t)l * S * (size_t)kvd;
        const size_t slot = (size_t)pos % S;  /* == pos unless the cache rolls */
        memcpy(kc + slot * kvd, m->k, (size_t)kvd * sizeof(float));
        memcpy(vc + slot * kvd, m->v, (size_t)kvd * sizeof(float));

        /* the attended positions, oldest first */
        const float* ka = kc;
        const float* va = vc;
        int32_t n_pos = pos + 1;
        if ((size_t)pos >= S) {  /* rolling: the last S positions, gathered in order */
            for (size_t j = 0; j < S; ++j) {
                const size_t src = ((size_t)pos + 1 + j) % S;
                memcpy(m->kwin + j * kvd, kc + src * kvd, (size_t)kvd * sizeof(float));
                memcpy(m->vwin + j * kvd, vc + src * kvd, (size_t)kvd * sizeof(float));
            }
            ka = m->kwin;
            va = m->vwin;
            n_pos = (int32_t)S;
        }
        for (int32_t h = 0; h < c->n_heads; ++h) {
            const int32_t kvh = h / group;
            oracle_attention_head(m->att + (size_t)h * hd, m->q + (size_t)h * hd,
                                  ka + (size_t)kvh * hd, va + (size_t)kvh * hd, kvd, hd, n_pos);
        }
        oracle_matvec(m->y, m->wo + (size_t)l * d * d, m->att, d, d);
        for (int32_t i = 0; i < d; ++i) m->x[i] += m->y[i];

        /* feed-forward block */
        oracle_rmsnorm(m->xb, m->x, m->g_ffn + (size_t)l * d, d, c->norm_eps);
        oracle_matvec(m->h1, m->w1 + (size_t)l * F * d, m->xb, F, d);
        oracle_matvec(m->h3, m->w3 + (size_t)l * F * d, m->xb, F, d);
        oracle_swiglu(m->hb, m->h1, m->h3, F);
        oracle_matvec(m->y, m->w2 + (size_t)l * d * F, m->hb, d, F);
        for (int32_t i = 0; i < d; ++i) m->x[i] += m->y[i];

        if (x_trace) memcpy(x_trace + (size_t)(l + 1) * d, m->x, (size_t)d * sizeof(float));
    }

    oracle_rmsnorm(m->xb, m->x, m->g_final, d, c->norm_eps);
    oracle_matvec(logits_out, m->wcls, m->xb, c->vocab_size, d);
    return 0;
}

/* The generation loop of the single-file engine: one forward per position;
 * prompt positions are fed from the prompt, later ones from the previous
 * greedy choice; no stop token. */
int oracle_generate(oracle_model* m, const int32_t* prompt, int32_t n_prompt, int32_t steps,
                    int32_t* out_tokens, float* logits_trace) {
    const oracle_config* c = &m->c;
    if (n_prompt < 1 || steps < 1) return -1;
    if (!c->rolling_cache && n_prompt + steps - 1 > c->seq_len) return -1;
    float* logits = (float*)malloc((size_t)c->vocab_size * sizeof(float));
    if (!logits) return -1;
    int32_t token = prompt[0];
    const int32_t n_fwd = n_prompt + steps - 1;
    for (int32_t pos = 0; pos < n_fwd; ++pos) {
        if (oracle_forward(m, token, pos, logits, NULL) != 0) {
            free(logits);
            return -1;
        }
        if (logits_trace)
            memcpy(logits_trace + (size_t)pos * c->vocab_size, logits,
                   (size_t)c->vocab_size * sizeof(float));
        const int32_t best = oracle_argmax(logits, c->vocab_size);
        if (pos >= n_prompt - 1) out_tokens[pos - (n_prompt - 1)] = best;
        token = (pos + 1 < n_prompt) ? prompt[pos + 1] : best;
    }
    free(logits);
    return 0;
}
