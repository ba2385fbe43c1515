// api.cu -- the C ABI of include/l2decode.h: handle lifetime, validation,
// weight upload + layout pass, per-forward CUDA graphs, and the decode loops.
//
// Decode loop (llama2.c pages: `./run out/model.bin` streams one token per
// forward in the single-file fp32 engine, 新智元 article "使用指南" and
// openai.wiki "模型推理"): the token and position of each forward live on the
// device. The classifier's last CTA writes the next token and advances the
// position, so a generation is `n_prompt + steps - 1` replays of one captured
// forward graph with no host round trip in between: one copy in, one copy out.
#include <cuda_runtime.h>
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <string>
#include <vector>

#include "l2_internal.cuh"

using namespace l2;

struct l2_handle {
    l2_config cfg{};
    int dev = 0, num_sms = 0;
    int hd = 0, kvd = 0;
    int pmax = 0;                    // batch-1 positions 0 .. pmax-1 (> seq_len: rolling cache)

    float* weights = nullptr;
    float *emb = nullptr, *g_att = nullptr, *g_ffn = nullptr, *g_final = nullptr;
    float *wqkv = nullptr, *wo = nullptr, *w13 = nullptr, *w2 = nullptr, *wcls = nullptr;
    size_t weight_floats = 0;

    float* kv = nullptr;             // K caches then V caches
    float *k_cache = nullptr, *v_cache = nullptr;
    size_t cache_layer = 0;          // floats of one layer of one sequence
    size_t cache_seq = 0;            // floats of one sequence (all layers)

    float* act = nullptr;            // activations block
    float *x = nullptr, *q = nullptr, *att = nullptr, *hb = nullptr, *logits = nullptr;
    float2* rope = nullptr;
    L2State* st = nullptr;
    int* ibuf = nullptr;             // prompt [S] + out [S] + uniforms [S]
    int *d_prompt = nullptr, *d_out = nullptr;
    float* d_uniforms = nullptr;     // sampling: one uniform number per generated token

    MatvecPlan p_qkv{}, p_wo{}, p_w13{}, p_w2{}, p_cls{};
    int nsplit = 1;
    uint64_t policy = 0;

    // two kernels per layer (fused_small.cu): Wo per head, W2 transposed, and
    // the fixed-point residual buffers P[2], M[2] of d entries each
    bool fused = false;
    FAttnArgs fattn{};
    FFfnArgs fffn{};
    int ffn_grid = 0;
    float* fw = nullptr;               // wo_h [L][H][d][hd], then w2t [L][F][d]
    long long* fx = nullptr;           // P0, P1, M0, M1

    // batched path (max_batch > 1): weights as tf32 (hi, lo) pairs, [Mcap][...]
    // activation rows, per-sequence state and the GEMM operand maps
    int mcap = 0;
    int rows = 0;                      // max(max_batch, max_prefill): row buffers of the GEMM path
    int a_rows = 128;                  // rows of the GEMMs' A tiles: 64 when rows <= 64
    // 64-row handles whose QKV / W1W3 / classifier launches are drained: the
    // *_hi copy holds W * g in fp32 (no lo copy), split in shared memory
    bool conv_qkv = false, conv_wo = false, conv_w13 = false, conv_w2 = false, conv_cls = false;
    float* bw = nullptr;
    float *qkv_hi = nullptr, *qkv_lo = nullptr, *wo_hi = nullptr, *wo_lo = nullptr;
    float *w13_hi = nullptr, *w13_lo = nullptr, *w2_hi = nullptr, *w2_lo = nullptr;
    float *cls_hi = nullptr, *cls_lo = nullptr;
    float* bact = nullptr;
    // bx: residual rows; xn_hi / xn_lo: the same rows as a tf32 pair, the A
    // operand of the norm-folded QKV, W1/W3 and classifier GEMMs
    float *bx = nullptr, *xn_hi = nullptr, *xn_lo = nullptr, *bq = nullptr;
    float *att_hi = nullptr, *att_lo = nullptr, *hb_hi = nullptr, *hb_lo = nullptr;
    float* blogits = nullptr;
    int* bst = nullptr;
    int *b_pos = nullptr, *b_token = nullptr, *b_active = nullptr, *b_len = nullptr;
    int *b_poff = nullptr, *b_last = nullptr, *b_prompts = nullptr, *b_out = nullptr;
    int* b_seq = nullptr;              // KV cache of each row (prefill: all 0)
    int* b_rmap = nullptr;             // batched prefill: (sequence, position) of each prompt row
    unsigned long long* b_keys = nullptr;
    // sums of squares of the rows entering a folded RMSNorm, [Mcap][ss_stride]:
    // ss_att (from the embedding gather or W2, read by QKV and the classifier)
    // and ss_ffn (from Wo, read by W1/W3)
    float *ss_att = nullptr, *ss_ffn = nullptr;
    int ss_stride = 0;
    GemmMaps m_qkv{}, m_wo{}, m_w13{}, m_w2{}, m_cls{};
    GemmPlan gp_qkv{64, 1, 2}, gp_wo{64, 1, 2}, gp_w13{64, 1, 2}, gp_w2{64, 1, 2}, gp_cls{128, 1, 2};
    GemmOccupancy gocc{};
    cudaGraphExec_t bgraph = nullptr;  // one batched generation step
    int bgraph_M = 0, bgraph_steps = 0;
    cudaGraphExec_t bgraph_s = nullptr;  // the same with sampling
    int bgraph_s_M = 0, bgraph_s_steps = 0;
    SampleParams* d_sparams = nullptr;   // batched sampling parameters
    float* b_uniforms = nullptr;         // [max_batch][seq_len] host-path uniforms

    cudaStream_t stream = nullptr;
    cudaGraphExec_t fwd1 = nullptr;  // one forward
    cudaGraphExec_t fwdN = nullptr;  // kGraphBatch forwards
    cudaGraphExec_t fwd1s = nullptr; // one forward + the sampler (captured on first use)
    cudaGraphExec_t fwdNs = nullptr; // kGraphBatch of them
    cudaEvent_t ev0 = nullptr, ev1 = nullptr;
    std::string err;
};

namespace {

constexpr int kGraphBatch = 8;
thread_local std::string g_create_error;

int fail(l2_handle* h, int code, const std::string& msg) {
    if (h)
        h->err = msg;
    else
        g_create_error = msg;
    return code;
}

int cuda_fail(l2_handle* h, cudaError_t e, const char* what) {
    const int code = (e == cudaErrorMemoryAllocation) ? L2_ENOMEM : L2_ECUDA;
    return fail(h, code, std::string(what) + ": " + cudaGetErrorString(e));
}

#define L2_CUDA(h, call)                                         \
    do {                                                         \
        cudaError_t e_ = (call);                                 \
        if (e_ != cudaSuccess) return cuda_fail((h), e_, #call); \
    } while (0)

size_t align64(size_t n) { return (n + 63) & ~static_cast<size_t>(63); }

bool config_valid(const l2_config* c, std::string* why) {
    auto bad = [&](const char* m) {
        if (why) *why = m;
        return false;
    };
    if (!c) return bad("config is NULL");
    if (c->dim <= 0 || c->hidden_dim <= 0 || c->n_layers <= 0 || c->n_heads <= 0 ||
        c->n_kv_heads <= 0 || c->vocab_size <= 0 || c->seq_len <= 0 || c->max_batch <= 0)
        return bad("every size must be positive");
    if (c->dim % c->n_heads != 0) return bad("dim must be a multiple of n_heads");
    if (c->n_heads % c->n_kv_heads != 0) return bad("n_heads must be a multiple of n_kv_heads");
    const int hd = c->dim / c->n_heads;
    if (hd % 2 != 0) return bad("head_dim must be even (RoPE pairs)");
    if (hd > 256) return bad("head_dim must be <= 256");
    if (c->dim % 4 != 0 || c->hidden_dim % 4 != 0) return bad("dim and hidden_dim must be multiples of 4");
    if (c->dim > 16384 || c->hidden_dim > 32768) return bad("dim <= 16384 and hidden_dim <= 32768");
    if (c->vocab_size > (1 << 24)) return bad("vocab_size <= 2^24");
    if (c->seq_len > (1 << 20)) return bad("seq_len <= 2^20");
    if (c->max_batch > 1024) return bad("max_batch <= 1024");
    if (c->max_prefill < 0 || c->max_prefill > 1024) return bad("0 <= max_prefill <= 1024");
    if (c->rolling_positions < 0 || c->rolling_positions > (1 << 24))
        return bad("0 <= rolling_positions <= 2^24");
    if (!(c->norm_eps >= 0.0f) || !(c->rope_theta > 0.0f)) return bad("norm_eps >= 0 and rope_theta > 0");
    if (c->shared_classifier != 0 && c->shared_classifier != 1) return bad("shared_classifier is 0 or 1");
    if (c->layer_kernels != 0 && c->layer_kernels != 2 && c->layer_kernels != 5)
        return bad("layer_kernels is 0, 2 or 5");
    return true;
}

__global__ void init_state_kernel(L2State* st, int pos, int token, const int* d_token,
                                  const int* d_pos, int vocab, int seq_len, int n_prompt, int mode,
                                  const int* prompt, int* out, int reset_err) {
    const int p_in = d_pos ? d_pos[0] : pos;
    // the token is checked (and clamped) where it is consumed, by the layer-0
    // QKV kernel's embedding read; a device position outside [0, seq_len) is
    // reported here and clamped, since the RoPE table and the cache slot
    // index depend on it
    const int t = d_token ? d_token[0] : (prompt && mode >= 1 ? prompt[0] : token);
    const int p = min(max(p_in, 0), seq_len - 1);
    (void)vocab;
    st->pos = p;
    st->token = t;
    st->n_prompt = n_prompt;
    st->mode = mode;
    st->prompt = prompt;
    st->out_tokens = out;
    st->argmax_key = 0ull;
    st->cls_done = 0u;
    if (reset_err) st->err = 0;
    if (p != p_in) atomicOr(&st->err, ERR_BAD_INPUT);
}

MatvecArgs base_args(l2_handle* h) {
    MatvecArgs a{};
    a.eps = h->cfg.norm_eps;
    a.d = h->cfg.dim;
    a.kvd = h->kvd;
    a.head_dim = h->hd;
    a.seq_len = h->cfg.seq_len;
    a.vocab = h->cfg.vocab_size;
    a.rope = h->rope;
    a.st = h->st;
    a.l2_policy = h->policy;
    return a;
}

// Launches kernel `kind` of layer l on stream s (kind as in l2_time_kernel).
void fused_layer_args(const l2_handle* h, size_t l, FAttnArgs* a, FFfnArgs* f);
// 64-bit words of the two-kernel path's residual buffers: two output rows of
// the FFN block in kFfnCopies copies each, two of the attention block.
inline size_t fx_words(size_t d) { return (2 * kFfnCopies + 2) * d; }

cudaError_t launch_kind(l2_handle* h, int kind, int l, cudaStream_t s) {
    const l2_config& c = h->cfg;
    const size_t d = c.dim, F = c.hidden_dim, kvd = h->kvd;
    if (kind == 14 || kind == 15) {  // the two-kernels-per-layer blocks
        FAttnArgs fa;
        FFfnArgs ff;
        fused_layer_args(h, static_cast<size_t>(l), &fa, &ff);
        return kind == 14 ? launch_fattn(fa, s, true) : launch_fffn(ff, h->ffn_grid, s, true);
    }
    MatvecArgs a = base_args(h);
    switch (kind) {
        case 0:
            a.W = h->wqkv + static_cast<size_t>(l) * (d + 2 * kvd) * d;
            a.plan = h->p_qkv;
            a.src = h->x;
            a.gain = h->g_att + l * d;
            a.emb = (l == 0) ? h->emb : nullptr;
            a.x_init = (l == 0) ? h->x : nullptr;
            a.q_out = h->q;
            a.k_cache = h->k_cache + l * h->cache_layer;
            a.v_cache = h->v_cache + l * h->cache_layer;
            return launch_matvec(EPI_QKV_ROPE, a, s, true);
        case 1: {
            AttnArgs t{};
            t.q = h->q;
            t.k_cache = h->k_cache + l * h->cache_layer;
            t.v_cache = h->v_cache + l * h->cache_layer;
            t.att = h->att;
            t.n_heads = c.n_heads;
            t.n_kv_heads = c.n_kv_heads;
            t.head_dim = h->hd;
            t.seq_len = c.seq_len;
            t.nsplit = h->nsplit;
            t.st = h->st;
            return launch_attention(t, s, true);
        }
        case 2:
            a.W = h->wo + static_cast<size_t>(l) * d * d;
            a.plan = h->p_wo;
            a.src = h->att;
            a.out = h->x;
            return launch_matvec(EPI_RESIDUAL, a, s, true);
        case 3:
            a.W = h->w13 + static_cast<size_t>(l) * 2 * F * d;
            a.plan = h->p_w13;
            a.src = h->x;
            a.gain = h->g_ffn + l * d;
            a.out = h->hb;
            return launch_matvec(EPI_SWIGLU, a, s, true);
        case 4:
            a.W = h->w2 + static_cast<size_t>(l) * d * F;
            a.plan = h->p_w2;
            a.src = h->hb;
            a.out = h->x;
            return launch_matvec(EPI_RESIDUAL, a, s, true);
        case 5:
            a.W = h->wcls;
            a.plan = h->p_cls;
            a.src = h->x;
            a.gain = h->g_final;
            a.out = h->logits;
            return launch_matvec(EPI_CLASSIFIER, a, s, true);
        default:
            return cudaErrorInvalidValue;
    }
}

// Two kernels per layer: the attention block and the FFN block, the residual
// in fixed point (P[l % 2] enters layer l, M[l % 2] after its attention).
void fused_layer_args(const l2_handle* h, size_t l, FAttnArgs* a, FFfnArgs* f) {
    const l2_config& c = h->cfg;
    const size_t d = c.dim, F = c.hidden_dim, kvd = h->kvd, L = c.n_layers;
    // P[b]: kFfnCopies copies of d (the FFN blocks' output), M[b]: one copy
    const size_t R = kFfnCopies;
    long long* P[2] = {h->fx, h->fx + R * d};
    long long* M[2] = {h->fx + 2 * R * d, h->fx + 2 * R * d + d};
    *a = h->fattn;
    a->wqkv = h->wqkv + l * (d + 2 * kvd) * d;
    a->wo_h = h->fw + l * d * d;
    a->g_att = h->g_att + l * d;
    a->x_in = l == 0 ? nullptr : P[l % 2];
    a->x_mid = M[l % 2];
    a->x_zero = P[(l + 1) % 2];
    a->k_cache = h->k_cache + l * h->cache_layer;
    a->v_cache = h->v_cache + l * h->cache_layer;
    *f = h->fffn;
    f->w13 = h->w13 + l * 2 * F * d;
    f->w2t = h->fw + L * d * d + l * F * d;
    f->g_ffn = h->g_ffn + l * d;
    f->x_mid = M[l % 2];
    f->x_out = P[(l + 1) % 2];
    f->x_zero = M[(l + 1) % 2];
}

cudaError_t enqueue_forward_fused(l2_handle* h, cudaStream_t s) {
    const size_t d = h->cfg.dim, L = h->cfg.n_layers;
    for (size_t l = 0; l < L; ++l) {
        FAttnArgs a;
        FFfnArgs f;
        fused_layer_args(h, l, &a, &f);
        cudaError_t e = launch_fattn(a, s, true);
        if (e != cudaSuccess) return e;
        if ((e = launch_fffn(f, h->ffn_grid, s, true)) != cudaSuccess) return e;
    }
    // classifier on the last residual; it also clears the next forward's M[0]
    long long* P[2] = {h->fx, h->fx + kFfnCopies * d};
    long long* M0 = h->fx + 2 * kFfnCopies * d;
    MatvecArgs a = base_args(h);
    a.W = h->wcls;
    a.plan = h->p_cls;
    a.src = h->x;
    a.src_fixed = P[L % 2];
    a.gain = h->g_final;
    a.out = h->logits;
    a.zero_fixed = M0;
    a.zero_n = static_cast<int>(d);
    return launch_matvec(EPI_CLASSIFIER, a, s, true);
}

cudaError_t enqueue_forward(l2_handle* h, cudaStream_t s) {
    if (h->fused) return enqueue_forward_fused(h, s);
    for (int l = 0; l < h->cfg.n_layers; ++l)
        for (int k = 0; k < 5; ++k) {
            cudaError_t e = launch_kind(h, k, l, s);
            if (e != cudaSuccess) return e;
        }
    return launch_kind(h, 5, 0, s);
}

int capture(l2_handle* h, int n_forwards, cudaGraphExec_t* out, bool sample = false) {
    cudaGraph_t g = nullptr;
    L2_CUDA(h, cudaStreamBeginCapture(h->stream, cudaStreamCaptureModeThreadLocal));
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < n_forwards && e == cudaSuccess; ++i) {
        e = enqueue_forward(h, h->stream);
        if (e == cudaSuccess && sample)
            e = launch_sample(SampleArgs{h->st, h->logits, h->cfg.vocab_size}, h->stream, true);
    }
    cudaError_t e2 = cudaStreamEndCapture(h->stream, &g);
    if (e != cudaSuccess) {
        if (g) cudaGraphDestroy(g);
        return cuda_fail(h, e, "kernel launch during capture");
    }
    if (e2 != cudaSuccess) return cuda_fail(h, e2, "cudaStreamEndCapture");
    e = cudaGraphInstantiate(out, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaGraphInstantiate");
    return L2_OK;
}

// Synchronous calls clear the device error word before their work and report
// it after; the *_device calls leave it accumulating for l2_status.
cudaError_t clear_device_error(l2_handle* h, cudaStream_t s) {
    return cudaMemsetAsync(&h->st->err, 0, sizeof(int), s);
}

// Return code for the bits of the device error word.
int status_of(l2_handle* h, int err) {
    if (err & (ERR_TIMEOUT_TMA | ERR_BAD_PLAN))
        return fail(h, L2_ETIMEOUT, "a bounded device wait gave up (bulk-copy completion)");
    if (err & ERR_BAD_INPUT)
        return fail(h, L2_EINVAL,
                    "a device token id outside [0, vocab_size) or position outside its range "
                    "(it was clamped, so the results are not those of the input)");
    return L2_OK;
}

int check_device_error(l2_handle* h) {
    int err = 0;
    L2_CUDA(h, cudaMemcpy(&err, &h->st->err, sizeof(int), cudaMemcpyDeviceToHost));
    return status_of(h, err);
}

// ---------------------------------------------------------------- batched path

// Kernel kinds of a batched step (l2_time_kernel numbers them 6 + kind).
enum BKind : int {
    BK_QKV = 0, BK_ATTN = 1, BK_WO = 2, BK_W13 = 3, BK_W2 = 4, BK_CLS = 5,
    BK_EMB = 6,  // embedding gather: residual rows, their tf32 pair, sums of squares
    BK_ADVANCE = 7,
    BK_SAMPLE_ADVANCE = 8,  // the advance of a generation with sampling
};

// Partial sums of squares a residual GEMM with this plan writes per row.
int ss_slots(const GemmPlan& p, int N) { return 2 * ((N + p.bn - 1) / p.bn); }

// Launches one kernel of a batched step for layer l on M rows.
cudaError_t launch_bkind(l2_handle* h, int kind, int l, int row0, int M, int mode, int steps,
                         bool want_logits, cudaStream_t s, bool prefill = false) {
    const l2_config& c = h->cfg;
    const int d = c.dim, F = c.hidden_dim, V = c.vocab_size;
    GemmArgs g{};
    g.row0 = row0;
    g.M = M;
    g.err = &h->st->err;
    g.layer = l;
    g.a_rows = h->a_rows;
    // tile width fixed at create (it is the weight maps' box); K split for this M
    auto plan = [&](const GemmPlan& p, int N, int K) {
        return plan_split(h->gocc, p.bn, M, N, K, h->a_rows);
    };
    switch (kind) {
        case BK_EMB: {
            BNormArgs n{};
            n.row0 = row0;
            n.x = h->bx;
            n.emb = h->emb;
            n.token = h->b_token;
            n.xn_hi = h->xn_hi;
            n.xn_lo = h->xn_lo;
            n.ss_out = h->ss_att;
            n.ss_stride = h->ss_stride;
            n.d = d;
            n.vocab = V;
            n.pos = h->b_pos;
            n.pmax = h->pmax;
            n.err = &h->st->err;
            return launch_brmsnorm(n, M, s, true);
        }
        case BK_QKV:
            g.N = d + 2 * h->kvd;
            g.K = d;
            g.q = h->bq;
            g.k_cache = h->k_cache + l * h->cache_layer;
            g.v_cache = h->v_cache + l * h->cache_layer;
            g.rope = h->rope;
            g.pos = h->b_pos;
            g.active = h->b_active;
            g.seq = prefill ? h->b_seq : nullptr;
            g.d = d;
            g.kvd = h->kvd;
            g.head_dim = h->hd;
            g.seq_len = c.seq_len;
            g.rope_positions = h->pmax;
            g.cache_seq = h->cache_seq;
            g.ss_in = h->ss_att;  // attention RMSNorm (gain in the weights)
            g.conv = h->conv_qkv ? 1 : 0;
            g.ss_count = l == 0 ? 1 : ss_slots(h->gp_w2, d);
            g.ss_stride = h->ss_stride;
            g.eps = c.norm_eps;
            return launch_gemm(GEPI_QKV_ROPE, plan(h->gp_qkv, g.N, g.K), h->m_qkv, g, s, true);
        case BK_ATTN: {
            BAttnArgs t{};
            t.row0 = row0;
            t.q = h->bq;
            t.k_cache = h->k_cache + l * h->cache_layer;
            t.v_cache = h->v_cache + l * h->cache_layer;
            t.att_hi = h->att_hi;
            t.att_lo = h->att_lo;
            t.pos = h->b_pos;
            t.active = h->b_active;
            t.seq = prefill ? h->b_seq : nullptr;
            t.d = d;
            t.n_heads = c.n_heads;
            t.n_kv_heads = c.n_kv_heads;
            t.head_dim = h->hd;
            t.seq_len = c.seq_len;
            t.cache_seq = h->cache_seq;
            // Launched after the QKV GEMM has drained, not overlapped with it:
            // with programmatic dependent launch its CTAs took SM slots while
            // the GEMM's CTAs still held them, landed unevenly and ran beside
            // the GEMM's shared-memory configuration (measured: the 256-row
            // step 0.53 -> 0.50 s without the overlap; the Wo GEMM after it
            // keeps the overlap, which measured better).
            return launch_battn(t, M, s, false);
        }
        case BK_WO:
            g.N = d;
            g.K = d;
            g.out = h->bx;
            g.ldc = d;
            g.x_hi = h->xn_hi;  // the W1/W3 GEMM's rows and their sums of squares
            g.x_lo = h->xn_lo;
            g.ss_out = h->ss_ffn;
            g.ss_stride = h->ss_stride;
            g.conv = h->conv_wo ? 1 : 0;  // fp32 Wo split in shared memory (no gain)
            return launch_gemm(GEPI_RESIDUAL, plan(h->gp_wo, g.N, g.K), h->m_wo, g, s, true);
        case BK_W13:
            g.N = 2 * F;
            g.K = d;
            g.out_hi = h->hb_hi;
            g.out_lo = h->hb_lo;
            g.ss_in = h->ss_ffn;  // FFN RMSNorm (gain in the weights)
            g.conv = h->conv_w13 ? 1 : 0;
            g.ss_count = ss_slots(h->gp_wo, d);
            g.ss_stride = h->ss_stride;
            g.eps = c.norm_eps;
            return launch_gemm(GEPI_SWIGLU, plan(h->gp_w13, g.N, g.K), h->m_w13, g, s, true);
        case BK_W2:
            g.N = d;
            g.K = F;
            g.out = h->bx;
            g.ldc = d;
            g.x_hi = h->xn_hi;  // the next QKV (or classifier) GEMM's rows and sums of squares
            g.x_lo = h->xn_lo;
            g.ss_out = h->ss_att;
            g.ss_stride = h->ss_stride;
            g.conv = h->conv_w2 ? 1 : 0;  // fp32 W2 split in shared memory (no gain)
            return launch_gemm(GEPI_RESIDUAL, plan(h->gp_w2, g.N, g.K), h->m_w2, g, s, true);
        case BK_CLS:
            g.layer = 0;
            g.N = V;
            g.K = d;
            g.out = want_logits ? h->blogits : nullptr;
            g.ldc = V;
            g.argmax_keys = h->b_keys;
            g.ss_in = h->ss_att;  // final RMSNorm (gain in the weights)
            g.conv = h->conv_cls ? 1 : 0;
            g.ss_count = ss_slots(h->gp_w2, d);
            g.ss_stride = h->ss_stride;
            g.eps = c.norm_eps;
            return launch_gemm(GEPI_ARGMAX, plan(h->gp_cls, g.N, g.K), h->m_cls, g, s, true);
        case BK_SAMPLE_ADVANCE: {
            BSampleArgs a{};
            a.row0 = row0;
            a.steps = steps;
            a.vocab = V;
            a.params = h->d_sparams;
            a.logits = h->blogits;
            a.keys = h->b_keys;
            a.last = h->b_last;
            a.pos = h->b_pos;
            a.token = h->b_token;
            a.active = h->b_active;
            a.len = h->b_len;
            a.poff = h->b_poff;
            a.prompts = h->b_prompts;
            a.out = h->b_out;
            return launch_bsample(a, M, s, true);
        }
        case BK_ADVANCE: {
            BAdvanceArgs a{};
            a.row0 = row0;
            a.M = M;
            a.mode = mode;
            a.steps = steps;
            a.keys = h->b_keys;
            a.last = h->b_last;
            a.pos = h->b_pos;
            a.token = h->b_token;
            a.active = h->b_active;
            a.len = h->b_len;
            a.poff = h->b_poff;
            a.prompts = h->b_prompts;
            a.out = h->b_out;
            return launch_badvance(a, s, true);
        }
        default:
            return cudaErrorInvalidValue;
    }
}

// Kernels of one lockstep step of rows [row0, row0 + M), in order: the
// embedding gather, then per layer the QKV GEMM (attention RMSNorm folded in;
// RoPE + KV append), attention, Wo GEMM + residual, W1/W3 GEMM (FFN RMSNorm
// folded in; SwiGLU), W2 GEMM + residual; the classifier GEMM (final RMSNorm
// folded in) with the per-row argmax; and the per-sequence advance.
// `prefill`: every row is a position of sequence 0 (cache 0, row positions
// in b_pos) instead of a sequence of its own.
cudaError_t enqueue_rows(l2_handle* h, int row0, int M, int mode, int steps, bool want_logits,
                         cudaStream_t s, bool prefill = false, bool sample = false) {
    if (sample) want_logits = true;  // the sampler reads every row's logits
    cudaError_t e = launch_bkind(h, BK_EMB, 0, row0, M, mode, steps, want_logits, s, prefill);
    for (int l = 0; l < h->cfg.n_layers && e == cudaSuccess; ++l) {
        const int seq[] = {BK_QKV, BK_ATTN, BK_WO, BK_W13, BK_W2};
        for (int i = 0; i < 5 && e == cudaSuccess; ++i)
            e = launch_bkind(h, seq[i], l, row0, M, mode, steps, want_logits, s, prefill);
    }
    if (e == cudaSuccess) e = launch_bkind(h, BK_CLS, 0, row0, M, mode, steps, want_logits, s, prefill);
    if (e == cudaSuccess)
        e = launch_bkind(h, sample ? BK_SAMPLE_ADVANCE : BK_ADVANCE, 0, row0, M, mode, steps,
                         want_logits, s, prefill);
    return e;
}

// Prefill rows [0, n): token tokens[r] at position pos0 + r of cache 0.
__global__ void prefill_setup_kernel(int n, int pos0, const int* tokens, int vocab, int* b_token,
                                     int* b_pos, int* b_seq, int* b_active,
                                     unsigned long long* keys, L2State* st) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= n) return;
    b_token[r] = tokens[r];  // checked and clamped by the embedding gather
    b_pos[r] = pos0 + r;
    b_seq[r] = 0;
    b_active[r] = 1;
    keys[r] = 0ull;
}

// After a prefill of positions 0..n-1: the argmax of position n-1 is the first
// generated token; the batch-1 decode state continues at position n.
__global__ void prefill_handoff_kernel(L2State* st, const int* last, int n, const int* prompt,
                                       int* out) {
    const int idx = last[n - 1];
    out[0] = idx;
    st->pos = n;
    st->token = idx;
    st->n_prompt = n;
    st->mode = 1;
    st->prompt = prompt;
    st->out_tokens = out;
    st->last_argmax = idx;
    st->argmax_key = 0ull;
    st->cls_done = 0u;
}

// One lockstep step of M sequences (rows [0, M)) on stream s.
cudaError_t enqueue_bstep(l2_handle* h, int M, int mode, int steps, bool want_logits,
                          cudaStream_t s) {
    return enqueue_rows(h, 0, M, mode, steps, want_logits, s);
}

// Rows [0, M): active, keys cleared; for generation, pos 0 and the first prompt token.
__global__ void binit_kernel(int M, int mode, int* pos, int* token, int* active,
                             const int* len, const int* poff, const int* prompts,
                             unsigned long long* keys, L2State* st) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= M) return;
    active[b] = 1;
    keys[b] = 0ull;
    if (mode == 1) {
        pos[b] = 0;
        token[b] = prompts[poff[b]];
    }
}

// Timing set-up: rows [0, M) active at position pos with token 1.
__global__ void bset_kernel(int M, int pos, int* b_pos, int* token, int* active,
                            unsigned long long* keys, L2State* st) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= M) return;
    b_pos[b] = pos;
    token[b] = 1;
    active[b] = 1;
    keys[b] = 0ull;
}

// Allocates the batched path's buffers, splits the laid-out weights into tf32
// pairs and builds the GEMM operand maps.
int setup_batched(l2_handle* h) {
    const l2_config& c = h->cfg;
    const size_t d = c.dim, F = c.hidden_dim, L = c.n_layers, V = c.vocab_size, S = c.seq_len;
    const size_t kvd = h->kvd, B = c.max_batch;
    const size_t RW = static_cast<size_t>(h->rows);  // row capacity (>= B)
    h->mcap = static_cast<int>((RW + 127) / 128 * 128);
    const size_t Mc = h->mcap;
    size_t off = 0;
    auto take = [&](size_t n) {
        const size_t o = off;
        off += align64(n);
        return o;
    };
    const size_t n_qkv = L * (d + 2 * kvd) * d, n_wo = L * d * d, n_w13 = L * 2 * F * d;
    const size_t n_w2 = L * d * F, n_cls = V * d;
    cudaStream_t s = h->stream;
    L2_CUDA(h, prepare_gemm(&h->gocc));
    const int Mb = static_cast<int>(RW);
    // at most 64 rows per GEMM (a prefill-only handle): 64-row A tiles, so the
    // shared-memory ring holds more weight bytes and the A operand is read once
    h->a_rows = RW <= 64 ? 64 : 128;
    const int ar = h->a_rows;
    h->gp_qkv = plan_gemm(h->gocc, Mb, static_cast<int>(d + 2 * kvd), static_cast<int>(d), 256, ar);
    // Wo and W2 write the per-row sums of squares of the next norm: tiles <= 128
    h->gp_wo = plan_gemm(h->gocc, Mb, static_cast<int>(d), static_cast<int>(d), 128, ar);
    h->gp_w13 = plan_gemm(h->gocc, Mb, static_cast<int>(2 * F), static_cast<int>(d), 256, ar);
    h->gp_w2 = plan_gemm(h->gocc, Mb, static_cast<int>(d), static_cast<int>(F), 128, ar);
    h->gp_cls = plan_gemm(h->gocc, Mb, static_cast<int>(V), static_cast<int>(d), 256, ar);
    // 64-row handles whose launches are drained split fp32 weights in shared
    // memory: no tf32 pair copy for them (Wo, W2: the weights themselves;
    // QKV, W1/W3, classifier: W * g in fp32 in the hi buffer)
    h->conv_qkv = ar == 64 && gemm_drained(h->gp_qkv, static_cast<int>(d));
    h->conv_wo = ar == 64 && gemm_drained(h->gp_wo, static_cast<int>(d));
    h->conv_w13 = ar == 64 && gemm_drained(h->gp_w13, static_cast<int>(d));
    h->conv_w2 = ar == 64 && gemm_drained(h->gp_w2, static_cast<int>(F));
    h->conv_cls = ar == 64 && gemm_drained(h->gp_cls, static_cast<int>(d));
    const size_t o_qh = take(n_qkv), o_ql = h->conv_qkv ? 0 : take(n_qkv);
    const size_t o_oh = h->conv_wo ? 0 : take(n_wo), o_ol = h->conv_wo ? 0 : take(n_wo);
    const size_t o_uh = take(n_w13), o_ul = h->conv_w13 ? 0 : take(n_w13);
    const size_t o_dh = h->conv_w2 ? 0 : take(n_w2), o_dl = h->conv_w2 ? 0 : take(n_w2);
    const size_t o_ch = take(n_cls), o_cl = h->conv_cls ? 0 : take(n_cls);
    L2_CUDA(h, cudaMalloc(&h->bw, off * sizeof(float)));
    // buffers that are not allocated alias one of the same size that is, so
    // that every tensor map stays valid; their launches never read them
    h->qkv_hi = h->bw + o_qh;
    h->qkv_lo = h->conv_qkv ? h->qkv_hi : h->bw + o_ql;
    h->wo_hi = h->conv_wo ? h->wo : h->bw + o_oh;
    h->wo_lo = h->conv_wo ? h->wo : h->bw + o_ol;
    h->w13_hi = h->bw + o_uh;
    h->w13_lo = h->conv_w13 ? h->w13_hi : h->bw + o_ul;
    h->w2_hi = h->conv_w2 ? h->w2 : h->bw + o_dh;
    h->w2_lo = h->conv_w2 ? h->w2 : h->bw + o_dl;
    h->cls_hi = h->bw + o_ch;
    h->cls_lo = h->conv_cls ? h->cls_hi : h->bw + o_cl;
    // the GEMMs that consume a normalised row carry the RMSNorm gain in their
    // weights (W[n][k] * g[k]); the row scale is applied in their epilogue
    if (h->conv_qkv)
        L2_CUDA(h, launch_scale_gain(h->wqkv, h->g_att, d, d + 2 * kvd, L, h->qkv_hi, s));
    else
        L2_CUDA(h, launch_split_tf32_gain(h->wqkv, h->g_att, d, d + 2 * kvd, L, h->qkv_hi, h->qkv_lo, s));
    if (!h->conv_wo) L2_CUDA(h, launch_split_tf32(h->wo, h->wo_hi, h->wo_lo, n_wo, s));
    if (h->conv_w13)
        L2_CUDA(h, launch_scale_gain(h->w13, h->g_ffn, d, 2 * F, L, h->w13_hi, s));
    else
        L2_CUDA(h, launch_split_tf32_gain(h->w13, h->g_ffn, d, 2 * F, L, h->w13_hi, h->w13_lo, s));
    if (!h->conv_w2) L2_CUDA(h, launch_split_tf32(h->w2, h->w2_hi, h->w2_lo, n_w2, s));
    if (h->conv_cls)
        L2_CUDA(h, launch_scale_gain(h->wcls, h->g_final, d, V, 1, h->cls_hi, s));
    else
        L2_CUDA(h, launch_split_tf32_gain(h->wcls, h->g_final, d, V, 1, h->cls_hi, h->cls_lo, s));

    off = 0;
    const size_t o_x = take(Mc * d), o_nh = take(Mc * d), o_nl = take(Mc * d), o_q = take(Mc * d);
    const size_t o_ah = take(Mc * d), o_al = take(Mc * d), o_hh = take(Mc * F), o_hl = take(Mc * F);
    const size_t o_lg = take(RW * V);
    // two slots per N tile of >= 64 columns, rounded up to whole 16-byte groups
    h->ss_stride = static_cast<int>((2 * ((d + 63) / 64) + 3) / 4 * 4);
    const size_t o_ssa = take(Mc * h->ss_stride), o_ssf = take(Mc * h->ss_stride);
    const size_t o_bu = take(B * static_cast<size_t>(h->pmax));
    L2_CUDA(h, cudaMalloc(&h->bact, off * sizeof(float)));
    L2_CUDA(h, cudaMemsetAsync(h->bact, 0, off * sizeof(float), s));
    h->bx = h->bact + o_x; h->xn_hi = h->bact + o_nh; h->xn_lo = h->bact + o_nl;
    h->bq = h->bact + o_q; h->att_hi = h->bact + o_ah; h->att_lo = h->bact + o_al;
    h->hb_hi = h->bact + o_hh; h->hb_lo = h->bact + o_hl; h->blogits = h->bact + o_lg;
    h->ss_att = h->bact + o_ssa; h->ss_ffn = h->bact + o_ssf;
    h->b_uniforms = h->bact + o_bu;

    off = 0;
    const size_t o_pos = take(Mc), o_tok = take(Mc), o_act = take(Mc), o_len = take(Mc);
    const size_t o_poff = take(Mc), o_last = take(Mc), o_pr = take(B * S);
    const size_t o_out = take(B * static_cast<size_t>(h->pmax));
    const size_t o_seq = take(Mc), o_keys = take(2 * Mc);
    const size_t o_sp = take((sizeof(SampleParams) + 3) / 4);
    const size_t o_rmap = take(2 * B * S);
    L2_CUDA(h, cudaMalloc(&h->bst, off * sizeof(int)));
    L2_CUDA(h, cudaMemsetAsync(h->bst, 0, off * sizeof(int), s));
    h->b_pos = h->bst + o_pos; h->b_token = h->bst + o_tok; h->b_active = h->bst + o_act;
    h->b_len = h->bst + o_len; h->b_poff = h->bst + o_poff; h->b_last = h->bst + o_last;
    h->b_prompts = h->bst + o_pr; h->b_out = h->bst + o_out;
    h->b_seq = h->bst + o_seq;
    h->b_keys = reinterpret_cast<unsigned long long*>(h->bst + o_keys);
    h->d_sparams = reinterpret_cast<SampleParams*>(h->bst + o_sp);
    h->b_rmap = h->bst + o_rmap;

    const long long D = d, FF = F, LL = L, MC = Mc;
    struct MapSpec { CUtensorMap* m; const float* p; long long inner, rows, layers; int box; };
    const MapSpec specs[] = {
        {&h->m_qkv.a_hi, h->xn_hi, D, MC, 1, ar}, {&h->m_qkv.a_lo, h->xn_lo, D, MC, 1, ar},
        {&h->m_qkv.b_hi, h->qkv_hi, D, D + 2 * static_cast<long long>(kvd), LL, h->gp_qkv.bn},
        {&h->m_qkv.b_lo, h->qkv_lo, D, D + 2 * static_cast<long long>(kvd), LL, h->gp_qkv.bn},
        {&h->m_wo.a_hi, h->att_hi, D, MC, 1, ar}, {&h->m_wo.a_lo, h->att_lo, D, MC, 1, ar},
        {&h->m_wo.b_hi, h->wo_hi, D, D, LL, h->gp_wo.bn}, {&h->m_wo.b_lo, h->wo_lo, D, D, LL, h->gp_wo.bn},
        {&h->m_w13.a_hi, h->xn_hi, D, MC, 1, ar}, {&h->m_w13.a_lo, h->xn_lo, D, MC, 1, ar},
        {&h->m_w13.b_hi, h->w13_hi, D, 2 * FF, LL, h->gp_w13.bn},
        {&h->m_w13.b_lo, h->w13_lo, D, 2 * FF, LL, h->gp_w13.bn},
        {&h->m_w2.a_hi, h->hb_hi, FF, MC, 1, ar}, {&h->m_w2.a_lo, h->hb_lo, FF, MC, 1, ar},
        {&h->m_w2.b_hi, h->w2_hi, FF, D, LL, h->gp_w2.bn}, {&h->m_w2.b_lo, h->w2_lo, FF, D, LL, h->gp_w2.bn},
        {&h->m_cls.a_hi, h->xn_hi, D, MC, 1, ar}, {&h->m_cls.a_lo, h->xn_lo, D, MC, 1, ar},
        {&h->m_cls.b_hi, h->cls_hi, D, static_cast<long long>(V), 1, h->gp_cls.bn},
        {&h->m_cls.b_lo, h->cls_lo, D, static_cast<long long>(V), 1, h->gp_cls.bn},
        // W in fp32 (times the folded gain), for the 64-row launches that
        // split it in shared memory
        {&h->m_qkv.b_raw, h->qkv_hi, D, D + 2 * static_cast<long long>(kvd), LL, h->gp_qkv.bn},
        {&h->m_wo.b_raw, h->wo, D, D, LL, h->gp_wo.bn},
        {&h->m_w13.b_raw, h->w13_hi, D, 2 * FF, LL, h->gp_w13.bn},
        {&h->m_w2.b_raw, h->w2, FF, D, LL, h->gp_w2.bn},
        {&h->m_cls.b_raw, h->cls_hi, D, static_cast<long long>(V), 1, h->gp_cls.bn},
    };
    for (const MapSpec& m : specs) {
        cudaError_t e = make_gemm_map(m.m, m.p, m.inner, m.rows, m.layers, m.box);
        if (e != cudaSuccess) return cuda_fail(h, e, "tensor map (cuTensorMapEncodeTiled)");
    }
    L2_CUDA(h, cudaStreamSynchronize(s));
    return L2_OK;
}

int upload(l2_handle* h, const float* blob, cudaMemcpyKind kind) {
    const l2_config& c = h->cfg;
    const size_t d = c.dim, F = c.hidden_dim, L = c.n_layers, V = c.vocab_size, kvd = h->kvd;
    const size_t o_gatt = V * d, o_wq = o_gatt + L * d, o_wk = o_wq + L * d * d;
    const size_t o_wv = o_wk + L * kvd * d, o_wo = o_wv + L * kvd * d, o_gffn = o_wo + L * d * d;
    const size_t o_w1 = o_gffn + L * d, o_w2 = o_w1 + L * F * d, o_w3 = o_w2 + L * d * F;
    const size_t o_gfin = o_w3 + L * F * d, o_wcls = o_gfin + d;
    cudaStream_t s = h->stream;
    const size_t fs = sizeof(float);
    auto h2d = [&](float* dst, size_t off, size_t n) {
        return cudaMemcpyAsync(dst, blob + off, n * fs, kind, s);
    };
    L2_CUDA(h, h2d(h->emb, 0, V * d));
    L2_CUDA(h, h2d(h->g_att, o_gatt, L * d));
    L2_CUDA(h, h2d(h->g_ffn, o_gffn, L * d));
    L2_CUDA(h, h2d(h->g_final, o_gfin, d));
    for (size_t l = 0; l < L; ++l) {
        float* dst = h->wqkv + l * (d + 2 * kvd) * d;
        L2_CUDA(h, h2d(dst, o_wq + l * d * d, d * d));
        L2_CUDA(h, h2d(dst + d * d, o_wk + l * kvd * d, kvd * d));
        L2_CUDA(h, h2d(dst + (d + kvd) * d, o_wv + l * kvd * d, kvd * d));
    }
    L2_CUDA(h, h2d(h->wo, o_wo, L * d * d));
    L2_CUDA(h, h2d(h->w2, o_w2, L * d * F));
    if (!c.shared_classifier) L2_CUDA(h, h2d(h->wcls, o_wcls, V * d));
    // W1/W3 interleave through a per-layer staging buffer
    float* stage = nullptr;
    L2_CUDA(h, cudaMalloc(&stage, 2 * F * d * fs));
    int rc = L2_OK;
    for (size_t l = 0; l < L && rc == L2_OK; ++l) {
        cudaError_t e = h2d(stage, o_w1 + l * F * d, F * d);
        if (e == cudaSuccess) e = h2d(stage + F * d, o_w3 + l * F * d, F * d);
        if (e == cudaSuccess)
            e = launch_interleave_rows(h->w13 + l * 2 * F * d, stage, stage + F * d,
                                       static_cast<long long>(F), static_cast<int>(d), s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) rc = cuda_fail(h, e, "weight upload / layout pass");
    }
    cudaFree(stage);
    if (rc != L2_OK) return rc;
    L2_CUDA(h, cudaStreamSynchronize(s));
    return L2_OK;
}

void free_all(l2_handle* h) {
    cudaFree(h->fw);
    cudaFree(h->fx);
    h->fw = nullptr;
    h->fx = nullptr;
    if (h->fwd1) cudaGraphExecDestroy(h->fwd1);
    if (h->fwdN) cudaGraphExecDestroy(h->fwdN);
    if (h->fwd1s) cudaGraphExecDestroy(h->fwd1s);
    if (h->fwdNs) cudaGraphExecDestroy(h->fwdNs);
    h->fwd1s = h->fwdNs = nullptr;
    if (h->bgraph) cudaGraphExecDestroy(h->bgraph);
    if (h->bgraph_s) cudaGraphExecDestroy(h->bgraph_s);
    h->bgraph_s = nullptr;
    cudaFree(h->bw);
    cudaFree(h->bact);
    cudaFree(h->bst);
    h->bgraph = nullptr;
    h->bw = h->bact = nullptr;
    h->bst = nullptr;
    if (h->ev0) cudaEventDestroy(h->ev0);
    if (h->ev1) cudaEventDestroy(h->ev1);
    if (h->stream) cudaStreamDestroy(h->stream);
    cudaFree(h->weights);
    cudaFree(h->kv);
    cudaFree(h->act);
    h->fwd1 = h->fwdN = nullptr;
    h->ev0 = h->ev1 = nullptr;
    h->stream = nullptr;
    h->weights = h->kv = h->act = nullptr;
}

// Decides between five and two kernels per layer for the batch-1 forward and,
// for two, lays out Wo per head and W2 transposed and allocates the
// fixed-point residual buffers.
int setup_fused(l2_handle* h) {
    const l2_config& c = h->cfg;
    const size_t d = c.dim, F = c.hidden_dim, L = c.n_layers;
    if (c.layer_kernels == 5) return L2_OK;
    FAttnArgs& a = h->fattn;
    FFfnArgs& f = h->fffn;
    a.emb = h->emb;
    a.rope = h->rope;
    a.st = h->st;
    a.d = c.dim;
    a.kvd = h->kvd;
    a.hd = h->hd;
    a.H = c.n_heads;
    a.KVH = c.n_kv_heads;
    a.S = c.seq_len;
    a.vocab = c.vocab_size;
    a.eps = c.norm_eps;
    a.l2_policy = h->policy;
    f.err = &h->st->err;
    f.d = c.dim;
    f.F = c.hidden_dim;
    f.eps = c.norm_eps;
    f.l2_policy = h->policy;
    int optin = 0;
    L2_CUDA(h, cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->dev));
    const bool fits = plan_fused(a, f, h->num_sms, static_cast<size_t>(optin), &h->ffn_grid);
    if (c.layer_kernels == 2 && !fits)
        return fail(h, L2_EINVAL, "layer_kernels 2: the shape does not fit the two-kernel layer");
    if (c.layer_kernels == 0 &&
        (!fits || static_cast<double>(h->weight_floats) * 4.0 >= 2e9))
        return L2_OK;
    L2_CUDA(h, cudaMalloc(&h->fw, (L * d * d + L * F * d) * sizeof(float)));
    L2_CUDA(h, cudaMalloc(&h->fx, fx_words(d) * sizeof(long long)));
    L2_CUDA(h, cudaMemsetAsync(h->fx, 0, fx_words(d) * sizeof(long long), h->stream));
    L2_CUDA(h, launch_retile_heads(h->fw, h->wo, static_cast<int>(L), static_cast<int>(d), h->hd,
                                   h->stream));
    L2_CUDA(h, launch_transpose_layers(h->fw + L * d * d, h->w2, static_cast<int>(L),
                                       static_cast<int>(d), static_cast<int>(F), h->stream));
    L2_CUDA(h, prepare_fused(a, f));
    L2_CUDA(h, cudaStreamSynchronize(h->stream));
    h->fused = true;
    return L2_OK;
}

// Batched forward of M rows whose tokens and positions are already in
// b_token / b_pos (device values are clamped by the kernels).
int bforward(l2_handle* h, int M, bool want_logits, cudaStream_t s) {
    binit_kernel<<<(M + 127) / 128, 128, 0, s>>>(M, 0, h->b_pos, h->b_token, h->b_active,
                                                 h->b_len, h->b_poff, h->b_prompts, h->b_keys,
                                                 h->st);
    L2_CUDA(h, cudaGetLastError());
    L2_CUDA(h, enqueue_bstep(h, M, 0, 0, want_logits, s));
    return L2_OK;
}

int capture_bstep(l2_handle* h, int M, int steps, bool sample = false) {
    cudaGraphExec_t& gx = sample ? h->bgraph_s : h->bgraph;
    int& gM = sample ? h->bgraph_s_M : h->bgraph_M;
    int& gS = sample ? h->bgraph_s_steps : h->bgraph_steps;
    if (gx && gM == M && gS == steps) return L2_OK;
    if (gx) cudaGraphExecDestroy(gx);
    gx = nullptr;
    cudaGraph_t g = nullptr;
    L2_CUDA(h, cudaStreamBeginCapture(h->stream, cudaStreamCaptureModeThreadLocal));
    cudaError_t e = enqueue_rows(h, 0, M, 1, steps, false, h->stream, false, sample);
    cudaError_t e2 = cudaStreamEndCapture(h->stream, &g);
    if (e != cudaSuccess) {
        if (g) cudaGraphDestroy(g);
        return cuda_fail(h, e, "batched step launch during capture");
    }
    if (e2 != cudaSuccess) return cuda_fail(h, e2, "cudaStreamEndCapture");
    e = cudaGraphInstantiate(&gx, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaGraphInstantiate");
    gM = M;
    gS = steps;
    return L2_OK;
}

// One bounded wait that nothing completes: an mbarrier expecting one arrival
// that is never made, with no copy in flight. The wait gives up after `limit`
// SM clock cycles and records the timeout in the error word, exactly as the
// decode kernels' waits on bulk-copy completions do.
__global__ void watchdog_kernel(L2State* st, long long limit) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait_bounded(&bar, 0u, limit)) atomicOr(&st->err, ERR_TIMEOUT_TMA);
}

}  // namespace

extern "C" {

size_t l2_blob_floats(const l2_config* c) {
    if (!config_valid(c, nullptr)) return 0;
    const size_t d = c->dim, F = c->hidden_dim, L = c->n_layers, V = c->vocab_size;
    const size_t kvd = static_cast<size_t>(c->n_kv_heads) * (d / c->n_heads);
    size_t n = V * d + L * d + L * d * d + 2 * L * kvd * d + L * d * d + L * d + 3 * L * F * d + d;
    if (!c->shared_classifier) n += V * d;
    return n;
}

static int create_impl(const l2_config* cfg, const float* blob, size_t blob_floats, bool on_device,
                       l2_handle** out) {
    if (out) *out = nullptr;
    std::string why;
    if (!out) return fail(nullptr, L2_EINVAL, "out is NULL");
    if (!config_valid(cfg, &why)) return fail(nullptr, L2_EINVAL, "invalid config: " + why);
    if (!blob) return fail(nullptr, L2_EINVAL, "blob is NULL");
    if (blob_floats != l2_blob_floats(cfg))
        return fail(nullptr, L2_EBLOB, "blob size " + std::to_string(blob_floats) +
                                           " != expected " + std::to_string(l2_blob_floats(cfg)));
    l2_handle* h = new l2_handle();
    h->cfg = *cfg;
    auto bail = [&](int rc) {
        g_create_error = h->err;
        free_all(h);
        delete h;
        return rc;
    };
    cudaError_t e = cudaGetDevice(&h->dev);
    if (e != cudaSuccess) return bail(cuda_fail(h, e, "cudaGetDevice"));
    cudaDeviceProp prop;
    e = cudaGetDeviceProperties(&prop, h->dev);
    if (e != cudaSuccess) return bail(cuda_fail(h, e, "cudaGetDeviceProperties"));
    if (prop.major < 10) return bail(fail(h, L2_ECUDA, "needs a Blackwell (sm_10x) device"));
    h->num_sms = prop.multiProcessorCount;

    const l2_config& c = h->cfg;
    const size_t d = c.dim, F = c.hidden_dim, L = c.n_layers, V = c.vocab_size, S = c.seq_len;
    const size_t B = c.max_batch;
    h->hd = c.dim / c.n_heads;
    h->kvd = c.n_kv_heads * h->hd;
    h->pmax = c.rolling_positions > c.seq_len ? c.rolling_positions : c.seq_len;
    const size_t P = static_cast<size_t>(h->pmax);
    const size_t kvd = h->kvd;

    // plans. A matrix under 3 MB is streamed by half the SMs (one CTA each):
    // such a launch is a few microseconds of latency, not bandwidth, and the
    // next kernel's CTAs (launched early, programmatic dependent launch) then
    // find free SMs, become resident and request their first weight slots
    // while this one runs, instead of waiting for its CTAs to leave (measured:
    // 15M +6 %, 44M +2 %, 110M +3 % tok/s; the 7B shape's matrices are all
    // larger and keep every SM)
    auto sms_for = [&](size_t rows, size_t cols) {
        return 4.0 * static_cast<double>(rows) * static_cast<double>(cols) < 3e6
                   ? (h->num_sms + 1) / 2
                   : h->num_sms;
    };
    h->p_qkv = plan_matvec(static_cast<int>(d + 2 * kvd), static_cast<int>(d), 2,
                           sms_for(d + 2 * kvd, d));
    h->p_wo = plan_matvec(static_cast<int>(d), static_cast<int>(d), 1, sms_for(d, d));
    h->p_w13 = plan_matvec(static_cast<int>(2 * F), static_cast<int>(d), 2, sms_for(2 * F, d));
    h->p_w2 = plan_matvec(static_cast<int>(d), static_cast<int>(F), 1, sms_for(d, F));
    h->p_cls = plan_matvec(static_cast<int>(V), static_cast<int>(d), 1, sms_for(V, d));
    size_t smem_max = 0;
    for (const MatvecPlan* p : {&h->p_qkv, &h->p_wo, &h->p_w13, &h->p_w2, &h->p_cls})
        smem_max = p->smem_bytes > smem_max ? p->smem_bytes : smem_max;
    // the opt-in limit covers static + dynamic shared memory; keep 1 KB for the static part
    if (smem_max + 1024 > prop.sharedMemPerBlockOptin)
        return bail(fail(h, L2_EINVAL, "shape needs more shared memory than a CTA has"));
    if ((e = prepare_attention()) != cudaSuccess) return bail(cuda_fail(h, e, "attention setup"));
    h->nsplit = attn_nsplit(c.n_heads, c.seq_len, h->num_sms);
    while (h->nsplit > 1 && attn_cluster_ok(h->hd, h->nsplit, c.n_heads) < 1) h->nsplit >>= 1;

    // weights
    size_t off = 0;
    auto take = [&](size_t n) {
        const size_t o = off;
        off += align64(n);
        return o;
    };
    const size_t o_emb = take(V * d), o_ga = take(L * d), o_gf = take(L * d), o_gfin = take(d);
    const size_t o_qkv = take(L * (d + 2 * kvd) * d), o_wo = take(L * d * d);
    const size_t o_w13 = take(L * 2 * F * d), o_w2 = take(L * d * F);
    const size_t o_cls = c.shared_classifier ? o_emb : take(V * d);
    h->weight_floats = off;
    e = cudaMalloc(&h->weights, off * sizeof(float));
    if (e != cudaSuccess) return bail(cuda_fail(h, e, "cudaMalloc(weights)"));
    h->emb = h->weights + o_emb;
    h->g_att = h->weights + o_ga;
    h->g_ffn = h->weights + o_gf;
    h->g_final = h->weights + o_gfin;
    h->wqkv = h->weights + o_qkv;
    h->wo = h->weights + o_wo;
    h->w13 = h->weights + o_w13;
    h->w2 = h->weights + o_w2;
    h->wcls = h->weights + o_cls;

    // KV caches: [B][L][KVH][S][hd] for K, then the same for V
    h->cache_layer = static_cast<size_t>(c.n_kv_heads) * S * h->hd;
    h->cache_seq = L * h->cache_layer;
    e = cudaMalloc(&h->kv, 2 * B * h->cache_seq * sizeof(float));
    if (e != cudaSuccess) return bail(cuda_fail(h, e, "cudaMalloc(kv cache)"));
    h->k_cache = h->kv;
    h->v_cache = h->kv + B * h->cache_seq;

    // activations and state
    off = 0;
    const size_t o_x = take(d), o_q = take(d), o_att = take(d), o_hb = take(F);
    const size_t o_lg = take(B * V);
    const size_t o_rope = take(P * h->hd);  // float2 [positions][hd/2]
    const size_t o_st = take((sizeof(L2State) + 3) / 4), o_ib = take(3 * P);
    e = cudaMalloc(&h->act, off * sizeof(float));
    if (e != cudaSuccess) return bail(cuda_fail(h, e, "cudaMalloc(activations)"));
    h->x = h->act + o_x;
    h->q = h->act + o_q;
    h->att = h->act + o_att;
    h->hb = h->act + o_hb;
    h->logits = h->act + o_lg;
    h->rope = reinterpret_cast<float2*>(h->act + o_rope);
    h->st = reinterpret_cast<L2State*>(h->act + o_st);
    h->ibuf = reinterpret_cast<int*>(h->act + o_ib);
    h->d_prompt = h->ibuf;
    h->d_out = h->ibuf + P;
    h->d_uniforms = reinterpret_cast<float*>(h->ibuf + 2 * P);

    e = cudaStreamCreateWithFlags(&h->stream, cudaStreamNonBlocking);
    if (e != cudaSuccess) return bail(cuda_fail(h, e, "cudaStreamCreate"));
    if ((e = cudaEventCreate(&h->ev0)) != cudaSuccess || (e = cudaEventCreate(&h->ev1)) != cudaSuccess)
        return bail(cuda_fail(h, e, "cudaEventCreate"));
    if ((e = cudaMemsetAsync(h->act, 0, off * sizeof(float), h->stream)) != cudaSuccess ||
        (e = cudaMemsetAsync(h->kv, 0, 2 * B * h->cache_seq * sizeof(float), h->stream)) != cudaSuccess)
        return bail(cuda_fail(h, e, "cudaMemset"));

    // RoPE table: angle pos * theta^(-2i/hd) in double, rounded to float
    {
        std::vector<float2> tab(P * (h->hd / 2));
        for (size_t p = 0; p < P; ++p)
            for (int i = 0; i < h->hd / 2; ++i) {
                const double freq = pow(static_cast<double>(c.rope_theta), -2.0 * i / h->hd);
                const double ang = static_cast<double>(p) * freq;
                tab[p * (h->hd / 2) + i] = make_float2(static_cast<float>(cos(ang)),
                                                       static_cast<float>(sin(ang)));
            }
        e = cudaMemcpyAsync(h->rope, tab.data(), tab.size() * sizeof(float2),
                            cudaMemcpyHostToDevice, h->stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(h->stream);
        if (e != cudaSuccess) return bail(cuda_fail(h, e, "rope table upload"));
    }

    // L2 policy for the weight stream: keep small models resident in L2
    const double wbytes = static_cast<double>(h->weight_floats) * 4.0;
    if (wbytes < 100e6) {
        const float frac = 1.0f;
        uint32_t bits;
        memcpy(&bits, &frac, 4);
        h->policy = bits;  // evict_last, fraction 1
    } else {
        h->policy = 0;     // evict_first
    }

    if ((e = set_matvec_smem_limits()) != cudaSuccess)
        return bail(cuda_fail(h, e, "cudaFuncSetAttribute"));

    // weights: upload + layout pass (pin the caller's host blob when possible)
    int rc;
    if (on_device) {
        rc = upload(h, blob, cudaMemcpyDeviceToDevice);
    } else {
        const size_t bytes = blob_floats * sizeof(float);
        const bool pinned = cudaHostRegister(const_cast<float*>(blob), bytes,
                                             cudaHostRegisterReadOnly) == cudaSuccess;
        if (!pinned) cudaGetLastError();
        rc = upload(h, blob, cudaMemcpyHostToDevice);
        if (pinned) cudaHostUnregister(const_cast<float*>(blob));
    }
    if (rc != L2_OK) return bail(rc);
    h->rows = c.max_batch > c.max_prefill ? c.max_batch : c.max_prefill;
    if (h->rows > 1 && (rc = setup_batched(h)) != L2_OK) return bail(rc);
    if ((rc = setup_fused(h)) != L2_OK) return bail(rc);

    if ((rc = capture(h, 1, &h->fwd1)) != L2_OK) return bail(rc);
    if ((rc = capture(h, kGraphBatch, &h->fwdN)) != L2_OK) return bail(rc);
    e = cudaStreamSynchronize(h->stream);
    if (e != cudaSuccess) return bail(cuda_fail(h, e, "create sync"));
    *out = h;
    return L2_OK;
}

int l2_create(const l2_config* cfg, const float* blob, size_t blob_floats, l2_handle** out) {
    return create_impl(cfg, blob, blob_floats, false, out);
}

int l2_create_from_device(const l2_config* cfg, const float* d_blob, size_t blob_floats,
                          l2_handle** out) {
    return create_impl(cfg, d_blob, blob_floats, true, out);
}

void l2_destroy(l2_handle* h) {
    if (!h) return;
    cudaStreamSynchronize(h->stream);
    free_all(h);
    delete h;
}

const char* l2_last_error(const l2_handle* h) {
    return h ? h->err.c_str() : g_create_error.c_str();
}

int l2_reset(l2_handle* h, int32_t seq) {
    if (!h) return fail(nullptr, L2_EINVAL, "handle is NULL");
    const size_t B = h->cfg.max_batch;
    if (seq < -1 || seq >= static_cast<int32_t>(B)) return fail(h, L2_EINVAL, "seq out of range");
    if (seq == -1) {
        L2_CUDA(h, cudaMemsetAsync(h->kv, 0, 2 * B * h->cache_seq * sizeof(float), h->stream));
    } else {
        L2_CUDA(h, cudaMemsetAsync(h->k_cache + seq * h->cache_seq, 0, h->cache_seq * sizeof(float), h->stream));
        L2_CUDA(h, cudaMemsetAsync(h->v_cache + seq * h->cache_seq, 0, h->cache_seq * sizeof(float), h->stream));
    }
    L2_CUDA(h, cudaStreamSynchronize(h->stream));
    return L2_OK;
}

static int run_forwards(l2_handle* h, int n, cudaStream_t s, bool sample = false) {
    cudaGraphExec_t gN = sample ? h->fwdNs : h->fwdN, g1 = sample ? h->fwd1s : h->fwd1;
    while (n >= kGraphBatch) {
        L2_CUDA(h, cudaGraphLaunch(gN, s));
        n -= kGraphBatch;
    }
    for (; n > 0; --n) L2_CUDA(h, cudaGraphLaunch(g1, s));
    return L2_OK;
}

// Sampling parameters of a generation (the state already holds mode 2).
__global__ void init_sample_kernel(L2State* st, float temperature, float topp,
                                   const float* uniforms) {
    st->temperature = temperature;
    st->topp = topp;
    st->uniforms = uniforms;
}

static int generate_sample_impl(l2_handle* h, const int32_t* prompt, int32_t n_prompt,
                                int32_t steps, float temperature, float topp,
                                const float* uniforms, int32_t* out, bool on_device,
                                cudaStream_t stream) {
    if (!h) return fail(nullptr, L2_EINVAL, "handle is NULL");
    if (!prompt || !out || !uniforms) return fail(h, L2_EINVAL, "NULL prompt, uniforms or output");
    if (n_prompt < 1 || steps < 1 || static_cast<long long>(n_prompt) + steps - 1 > h->pmax)
        return fail(h, L2_EINVAL,
                    "need n_prompt >= 1, steps >= 1, n_prompt + steps - 1 <= seq_len (rolling: "
                    "rolling_positions)");
    if (!(temperature >= 0.0f) || !(topp > 0.0f && topp <= 1.0f))
        return fail(h, L2_EINVAL, "need temperature >= 0 and 0 < topp <= 1");
    if (!on_device) {
        for (int i = 0; i < n_prompt; ++i)
            if (prompt[i] < 0 || prompt[i] >= h->cfg.vocab_size)
                return fail(h, L2_EINVAL, "prompt id out of range");
        for (int i = 0; i < steps; ++i)
            if (!(uniforms[i] >= 0.0f && uniforms[i] < 1.0f))
                return fail(h, L2_EINVAL, "uniform numbers must lie in [0, 1)");
    }
    if (!h->fwd1s) {
        int rc = capture(h, 1, &h->fwd1s, true);
        if (rc == L2_OK) rc = capture(h, kGraphBatch, &h->fwdNs, true);
        if (rc != L2_OK) return rc;
    }
    cudaStream_t s = on_device ? stream : h->stream;
    const int32_t* d_prompt = prompt;
    const float* d_u = uniforms;
    int32_t* d_out = on_device ? out : h->d_out;
    if (!on_device) {
        L2_CUDA(h, cudaMemcpyAsync(h->d_prompt, prompt, sizeof(int32_t) * n_prompt,
                                   cudaMemcpyHostToDevice, s));
        L2_CUDA(h, cudaMemcpyAsync(h->d_uniforms, uniforms, sizeof(float) * steps,
                                   cudaMemcpyHostToDevice, s));
        d_prompt = h->d_prompt;
        d_u = h->d_uniforms;
    }
    init_state_kernel<<<1, 1, 0, s>>>(h->st, 0, 0, nullptr, nullptr, h->cfg.vocab_size,
                                      h->pmax, n_prompt, 2, d_prompt, d_out, 1);
    init_sample_kernel<<<1, 1, 0, s>>>(h->st, temperature, topp, d_u);
    L2_CUDA(h, cudaGetLastError());
    int rc = run_forwards(h, n_prompt + steps - 1, s, true);
    if (rc != L2_OK || on_device) return rc;
    L2_CUDA(h, cudaMemcpyAsync(out, h->d_out, sizeof(int32_t) * steps, cudaMemcpyDeviceToHost, s));
    L2_CUDA(h, cudaStreamSynchronize(s));
    return check_device_error(h);
}

int l2_generate_sample(l2_handle* h, const int32_t* prompt, int32_t n_prompt, int32_t steps,
                       float temperature, float topp, const float* uniforms,
                       int32_t* out_tokens) {
    return generate_sample_impl(h, prompt, n_prompt, steps, temperature, topp, uniforms,
                                out_tokens, false, nullptr);
}

int l2_generate_sample_device(l2_handle* h, const int32_t* d_prompt, int32_t n_prompt,
                              int32_t steps, float temperature, float topp,
                              const float* d_uniforms, int32_t* d_out, void* stream) {
    return generate_sample_impl(h, d_prompt, n_prompt, steps, temperature, topp, d_uniforms,
                                d_out, true, static_cast<cudaStream_t>(stream));
}

int l2_forward_device(l2_handle* h, const int32_t* d_tokens, const int32_t* d_pos, int32_t B,
                      float* d_logits, void* stream) {
    if (!h) return fail(nullptr, L2_EINVAL, "handle is NULL");
    if (B < 1 || B > h->cfg.max_batch) return fail(h, L2_EINVAL, "B out of range");
    if (!d_tokens || !d_pos) return fail(h, L2_EINVAL, "NULL token or position buffer");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (B > 1) {
        L2_CUDA(h, cudaMemcpyAsync(h->b_token, d_tokens, sizeof(int32_t) * B,
                                   cudaMemcpyDeviceToDevice, s));
        L2_CUDA(h, cudaMemcpyAsync(h->b_pos, d_pos, sizeof(int32_t) * B, cudaMemcpyDeviceToDevice,
                                   s));
        int rc = bforward(h, B, d_logits != nullptr, s);
        if (rc != L2_OK) return rc;
        if (d_logits)
            L2_CUDA(h, cudaMemcpyAsync(d_logits, h->blogits,
                                       sizeof(float) * B * static_cast<size_t>(h->cfg.vocab_size),
                                       cudaMemcpyDeviceToDevice, s));
        return L2_OK;
    }
    init_state_kernel<<<1, 1, 0, s>>>(h->st, 0, 0, d_tokens, d_pos, h->cfg.vocab_size,
                                      h->pmax, 0, 0, nullptr, nullptr, 0);
    L2_CUDA(h, cudaGetLastError());
    int rc = run_forwards(h, 1, s);
    if (rc != L2_OK) return rc;
    if (d_logits)
        L2_CUDA(h, cudaMemcpyAsync(d_logits, h->logits, sizeof(float) * h->cfg.vocab_size,
                                   cudaMemcpyDeviceToDevice, s));
    return L2_OK;
}

int l2_forward(l2_handle* h, const int32_t* tokens, const int32_t* pos, int32_t B,
               float* logits_out) {
    if (!h) return fail(nullptr, L2_EINVAL, "handle is NULL");
    if (!tokens || !pos) return fail(h, L2_EINVAL, "NULL tokens or positions");
    if (B < 1 || B > h->cfg.max_batch) return fail(h, L2_EINVAL, "B out of range");
    for (int b = 0; b < B; ++b) {
        if (tokens[b] < 0 || tokens[b] >= h->cfg.vocab_size) return fail(h, L2_EINVAL, "token out of range");
        if (pos[b] < 0 || pos[b] >= h->pmax)
            return fail(h, L2_EINVAL, "position out of range");
    }
    if (B > 1) {
        L2_CUDA(h, clear_device_error(h, h->stream));
        L2_CUDA(h, cudaMemcpyAsync(h->b_token, tokens, sizeof(int32_t) * B, cudaMemcpyHostToDevice,
                                   h->stream));
        L2_CUDA(h, cudaMemcpyAsync(h->b_pos, pos, sizeof(int32_t) * B, cudaMemcpyHostToDevice,
                                   h->stream));
        int rc = bforward(h, B, logits_out != nullptr, h->stream);
        if (rc != L2_OK) return rc;
        if (logits_out)
            L2_CUDA(h, cudaMemcpyAsync(logits_out, h->blogits,
                                       sizeof(float) * B * static_cast<size_t>(h->cfg.vocab_size),
                                       cudaMemcpyDeviceToHost, h->stream));
        L2_CUDA(h, cudaStreamSynchronize(h->stream));
        return check_device_error(h);
    }
    init_state_kernel<<<1, 1, 0, h->stream>>>(h->st, pos[0], tokens[0], nullptr, nullptr,
                                              h->cfg.vocab_size, h->pmax, 0, 0, nullptr,
                                              nullptr, 1);
    L2_CUDA(h, cudaGetLastError());
    int rc = run_forwards(h, 1, h->stream);
    if (rc != L2_OK) return rc;
    if (logits_out)
        L2_CUDA(h, cudaMemcpyAsync(logits_out, h->logits, sizeof(float) * h->cfg.vocab_size,
                                   cudaMemcpyDeviceToHost, h->stream));
    L2_CUDA(h, cudaStreamSynchronize(h->stream));
    return check_device_error(h);
}

int l2_generate_device(l2_handle* h, const int32_t* d_prompt, int32_t n_prompt, int32_t steps,
                       int32_t* d_out, void* stream) {
    if (!h) return fail(nullptr, L2_EINVAL, "handle is NULL");
    if (!d_prompt || !d_out) return fail(h, L2_EINVAL, "NULL prompt or output buffer");
    if (n_prompt < 1 || steps < 1 || static_cast<long long>(n_prompt) + steps - 1 > h->pmax)
        return fail(h, L2_EINVAL,
                    "need n_prompt >= 1, steps >= 1, n_prompt + steps - 1 <= seq_len (rolling: "
                    "rolling_positions)");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    init_state_kernel<<<1, 1, 0, s>>>(h->st, 0, 0, nullptr, nullptr, h->cfg.vocab_size,
                                      h->pmax, n_prompt, 1, d_prompt, d_out, 0);
    L2_CUDA(h, cudaGetLastError());
    return run_forwards(h, n_prompt + steps - 1, s);
}

int l2_generate(l2_handle* h, const int32_t* prompt, int32_t n_prompt, int32_t steps,
                int32_t* out_tokens) {
    if (!h) return fail(nullptr, L2_EINVAL, "handle is NULL");
    if (!prompt || !out_tokens) return fail(h, L2_EINVAL, "NULL prompt or output");
    if (n_prompt < 1 || steps < 1 || static_cast<long long>(n_prompt) + steps - 1 > h->pmax)
        return fail(h, L2_EINVAL,
                    "need n_prompt >= 1, steps >= 1, n_prompt + steps - 1 <= seq_len (rolling: "
                    "rolling_positions)");
    for (int i = 0; i < n_prompt; ++i)
        if (prompt[i] < 0 || prompt[i] >= h->cfg.vocab_size) return fail(h, L2_EINVAL, "prompt id out of range");
    L2_CUDA(h, cudaMemcpyAsync(h->d_prompt, prompt, sizeof(int32_t) * n_prompt,
                               cudaMemcpyHostToDevice, h->stream));
    init_state_kernel<<<1, 1, 0, h->stream>>>(h->st, 0, 0, nullptr, nullptr, h->cfg.vocab_size,
                                              h->pmax, n_prompt, 1, h->d_prompt, h->d_out, 1);
    L2_CUDA(h, cudaGetLastError());
    int rc = run_forwards(h, n_prompt + steps - 1, h->stream);
    if (rc != L2_OK) return rc;
    L2_CUDA(h, cudaMemcpyAsync(out_tokens, h->d_out, sizeof(int32_t) * steps,
                               cudaMemcpyDeviceToHost, h->stream));
    L2_CUDA(h, cudaStreamSynchronize(h->stream));
    return check_device_error(h);
}

__global__ void bparams_kernel(SampleParams* p, float temperature, float topp,
                               const float* uniforms) {
    p->temperature = temperature;
    p->topp = topp;
    p->uniforms = uniforms;
}

// sample: draw generated tokens (temperature, topp, uniforms [B][steps]) instead
// of the greedy choice.
static int generate_batch_impl(l2_handle* h, const int32_t* prompts, const int32_t* lens,
                               int32_t B, int32_t steps, int32_t* out_tokens, bool on_device,
                               cudaStream_t stream, bool sample = false,
                               float temperature = 0.0f, float topp = 1.0f,
                               const float* uniforms = nullptr) {
    if (!h) return fail(nullptr, L2_EINVAL, "handle is NULL");
    if (!prompts || !lens || !out_tokens) return fail(h, L2_EINVAL, "NULL prompts, lens or output");
    if (B < 1 || B > h->cfg.max_batch) return fail(h, L2_EINVAL, "B out of range");
    if (steps < 1) return fail(h, L2_EINVAL, "steps must be >= 1");
    const int S = h->cfg.seq_len, V = h->cfg.vocab_size;
    std::vector<int32_t> poff(B);
    long long total = 0;
    int max_len = 0;
    for (int b = 0; b < B; ++b) {
        if (lens[b] < 1 || lens[b] > S || static_cast<long long>(lens[b]) + steps - 1 > h->pmax)
            return fail(h, L2_EINVAL,
                        "need 1 <= lens[b] <= seq_len and lens[b] + steps - 1 <= seq_len "
                        "(rolling: rolling_positions)");
        poff[b] = static_cast<int32_t>(total);
        total += lens[b];
        max_len = lens[b] > max_len ? lens[b] : max_len;
    }
    if (!on_device)
        for (long long i = 0; i < total; ++i)
            if (prompts[i] < 0 || prompts[i] >= V) return fail(h, L2_EINVAL, "prompt id out of range");
    if (!on_device) L2_CUDA(h, clear_device_error(h, h->stream));
    if (sample) {
        if (!uniforms) return fail(h, L2_EINVAL, "NULL uniforms");
        if (!(temperature >= 0.0f) || !(topp > 0.0f && topp <= 1.0f))
            return fail(h, L2_EINVAL, "need temperature >= 0 and 0 < topp <= 1");
        if (!on_device)
            for (long long i = 0; i < static_cast<long long>(B) * steps; ++i)
                if (!(uniforms[i] >= 0.0f && uniforms[i] < 1.0f))
                    return fail(h, L2_EINVAL, "uniform numbers must lie in [0, 1)");
        if (h->cfg.max_batch == 1)
            return fail(h, L2_EINVAL,
                        "batched sampling needs max_batch > 1 (batch 1: l2_generate_sample)");
    }
    if (h->cfg.max_batch == 1)
        return on_device ? l2_generate_device(h, prompts, lens[0], steps, out_tokens, stream)
                         : l2_generate(h, prompts, lens[0], steps, out_tokens);
    cudaStream_t s = on_device ? stream : h->stream;
    if (sample) {
        const float* d_u = uniforms;
        if (!on_device) {
            L2_CUDA(h, cudaMemcpyAsync(h->b_uniforms, uniforms,
                                       sizeof(float) * static_cast<size_t>(B) * steps,
                                       cudaMemcpyHostToDevice, s));
            d_u = h->b_uniforms;
        }
        bparams_kernel<<<1, 1, 0, s>>>(h->d_sparams, temperature, topp, d_u);
        L2_CUDA(h, cudaGetLastError());
    }
    L2_CUDA(h, cudaMemcpyAsync(h->b_prompts, prompts, sizeof(int32_t) * total,
                               on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice, s));
    L2_CUDA(h, cudaMemcpyAsync(h->b_len, lens, sizeof(int32_t) * B, cudaMemcpyHostToDevice, s));
    L2_CUDA(h, cudaMemcpyAsync(h->b_poff, poff.data(), sizeof(int32_t) * B, cudaMemcpyHostToDevice,
                               s));
    binit_kernel<<<(B + 127) / 128, 128, 0, s>>>(B, 1, h->b_pos, h->b_token, h->b_active,
                                                 h->b_len, h->b_poff, h->b_prompts, h->b_keys,
                                                 h->st);
    L2_CUDA(h, cudaGetLastError());
    int rc = capture_bstep(h, B, steps, sample);
    if (rc != L2_OK) return rc;
    const int n = max_len + steps - 1;
    cudaGraphExec_t gx = sample ? h->bgraph_s : h->bgraph;
    for (int i = 0; i < n; ++i) L2_CUDA(h, cudaGraphLaunch(gx, s));
    L2_CUDA(h, cudaMemcpyAsync(out_tokens, h->b_out, sizeof(int32_t) * B * static_cast<size_t>(steps),
                               on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyDeviceToHost, s));
    if (on_device) return L2_OK;
    L2_CUDA(h, cudaStreamSynchronize(s));
    return check_device_error(h);
}

// Queues prefill rows [0, n) of cache 0 at positions pos0.. (tokens: device).
static int enqueue_prefill(l2_handle* h, const int32_t* d_tokens, int32_t n, int32_t pos0,
                           bool want_logits, cudaStream_t s) {
    prefill_setup_kernel<<<(n + 127) / 128, 128, 0, s>>>(n, pos0, d_tokens, h->cfg.vocab_size,
                                                         h->b_token, h->b_pos, h->b_seq,
                                                         h->b_active, h->b_keys, h->st);
    L2_CUDA(h, cudaGetLastError());
    L2_CUDA(h, enqueue_rows(h, 0, n, 0, 0, want_logits, s, true));
    return L2_OK;
}

static int prefill_checks(l2_handle* h, int32_t n, int32_t pos0) {
    if (h->rows < 2) return fail(h, L2_EINVAL, "handle has no prefill path (max_prefill and max_batch <= 1)");
    if (n < 1 || n > h->rows) return fail(h, L2_EINVAL, "prefill length outside [1, max(max_batch, max_prefill)]");
    if (pos0 < 0 || static_cast<long long>(pos0) + n > h->cfg.seq_len)
        return fail(h, L2_EINVAL, "prefill positions outside [0, seq_len)");
    return L2_OK;
}

int l2_prefill(l2_handle* h, const int32_t* tokens, int32_t n, int32_t pos0, float* logits_out) {
    if (!h) return fail(nullptr, L2_EINVAL, "handle is NULL");
    if (!tokens) return fail(h, L2_EINVAL, "NULL tokens");
    int rc = prefill_checks(h, n, pos0);
    if (rc != L2_OK) return rc;
    for (int i = 0; i < n; ++i)
        if (tokens[i] < 0 || tokens[i] >= h->cfg.vocab_size) return fail(h, L2_EINVAL, "token out of range");
    cudaStream_t s = h->stream;
    L2_CUDA(h, clear_device_error(h, s));
    L2_CUDA(h, cudaMemcpyAsync(h->d_prompt, tokens, sizeof(int32_t) * n, cudaMemcpyHostToDevice, s));
    if ((rc = enqueue_prefill(h, h->d_prompt, n, pos0, logits_out != nullptr, s)) != L2_OK) return rc;
    if (logits_out)
        L2_CUDA(h, cudaMemcpyAsync(logits_out, h->blogits,
                                   sizeof(float) * n * static_cast<size_t>(h->cfg.vocab_size),
                                   cudaMemcpyDeviceToHost, s));
    L2_CUDA(h, cudaStreamSynchronize(s));
    return check_device_error(h);
}

static int generate_prefill_impl(l2_handle* h, const int32_t* prompt, int32_t n_prompt,
                                 int32_t steps, int32_t* out, bool on_device, cudaStream_t stream) {
    if (!h) return fail(nullptr, L2_EINVAL, "handle is NULL");
    if (!prompt || !out) return fail(h, L2_EINVAL, "NULL prompt or output");
    if (n_prompt < 1 || steps < 1 || static_cast<long long>(n_prompt) + steps - 1 > h->pmax)
        return fail(h, L2_EINVAL,
                    "need n_prompt >= 1, steps >= 1, n_prompt + steps - 1 <= seq_len (rolling: "
                    "rolling_positions)");
    int rc = prefill_checks(h, n_prompt, 0);
    if (rc != L2_OK) return rc;
    cudaStream_t s = on_device ? stream : h->stream;
    const int32_t* d_prompt = prompt;
    int32_t* d_out = on_device ? out : h->d_out;
    if (!on_device) {
        for (int i = 0; i < n_prompt; ++i)
            if (prompt[i] < 0 || prompt[i] >= h->cfg.vocab_size)
                return fail(h, L2_EINVAL, "prompt id out of range");
        L2_CUDA(h, clear_device_error(h, s));
        L2_CUDA(h, cudaMemcpyAsync(h->d_prompt, prompt, sizeof(int32_t) * n_prompt,
                                   cudaMemcpyHostToDevice, s));
        d_prompt = h->d_prompt;
    }
    if ((rc = enqueue_prefill(h, d_prompt, n_prompt, 0, false, s)) != L2_OK) return rc;
    prefill_handoff_kernel<<<1, 1, 0, s>>>(h->st, h->b_last, n_prompt, d_prompt, d_out);
    L2_CUDA(h, cudaGetLastError());
    if ((rc = run_forwards(h, steps - 1, s)) != L2_OK) return rc;
    if (on_device) return L2_OK;
    L2_CUDA(h, cudaMemcpyAsync(out, h->d_out, sizeof(int32_t) * steps, cudaMemcpyDeviceToHost, s));
    L2_CUDA(h, cudaStreamSynchronize(s));
    return check_device_error(h);
}

// Batched prefill: rows [0, n) of a pass are prompt rows start .. start+n-1
// of the concatenated prompts; row r is sequence rmap[2 i] at position
// rmap[2 i + 1] (i = start + r) and writes that sequence's cache.
__global__ void bprefill_setup_kernel(int n, int start, const int* rmap, const int* prompts,
                                      const int* poff, int vocab, int* b_token, int* b_pos,
                                      int* b_seq, int* b_active, unsigned long long* keys,
                                      L2State* st) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= n) return;
    const int b = rmap[2 * (start + r)], p = rmap[2 * (start + r) + 1];
    b_token[r] = prompts[poff[b] + p];  // checked and clamped by the embedding gather
    b_pos[r] = p;
    b_seq[r] = b;
    b_active[r] = 1;
    keys[r] = 0ull;
}

// After a pass: the argmax of a sequence's last prompt position is its first
// generated token.
__global__ void bprefill_handoff_kernel(int n, int start, const int* rmap, const int* lens,
                                        const int* last, int steps, int* out) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= n) return;
    const int b = rmap[2 * (start + r)], p = rmap[2 * (start + r) + 1];
    if (p == lens[b] - 1) out[static_cast<size_t>(b) * steps] = last[r];
}

// Sequences continue in lockstep from their first generated token.
__global__ void bprefill_continue_kernel(int B, int steps, const int* lens, const int* out,
                                         int* pos, int* token, int* active,
                                         unsigned long long* keys) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    pos[b] = lens[b];
    token[b] = out[static_cast<size_t>(b) * steps];
    active[b] = steps > 1 ? 1 : 0;
    keys[b] = 0ull;
}

static int generate_batch_prefill_impl(l2_handle* h, const int32_t* prompts, const int32_t* lens,
                                       int32_t B, int32_t steps, int32_t* out_tokens,
                                       bool on_device, cudaStream_t stream) {
    if (!h) return fail(nullptr, L2_EINVAL, "handle is NULL");
    if (!prompts || !lens || !out_tokens) return fail(h, L2_EINVAL, "NULL prompts, lens or output");
    if (h->cfg.max_batch < 2) return fail(h, L2_EINVAL, "batched prefill needs max_batch > 1");
    if (B < 1 || B > h->cfg.max_batch) return fail(h, L2_EINVAL, "B out of range");
    if (steps < 1) return fail(h, L2_EINVAL, "steps must be >= 1");
    const int S = h->cfg.seq_len, V = h->cfg.vocab_size;
    std::vector<int32_t> poff(B), rmap;
    long long total = 0;
    for (int b = 0; b < B; ++b) {
        if (lens[b] < 1 || lens[b] > S || static_cast<long long>(lens[b]) + steps - 1 > h->pmax)
            return fail(h, L2_EINVAL,
                        "need 1 <= lens[b] <= seq_len and lens[b] + steps - 1 <= seq_len "
                        "(rolling: rolling_positions)");
        poff[b] = static_cast<int32_t>(total);
        total += lens[b];
    }
    if (!on_device)
        for (long long i = 0; i < total; ++i)
            if (prompts[i] < 0 || prompts[i] >= V) return fail(h, L2_EINVAL, "prompt id out of range");
    if (!on_device) L2_CUDA(h, clear_device_error(h, h->stream));
    rmap.reserve(2 * total);
    for (int b = 0; b < B; ++b)
        for (int p = 0; p < lens[b]; ++p) {
            rmap.push_back(b);
            rmap.push_back(p);
        }
    cudaStream_t s = on_device ? stream : h->stream;
    L2_CUDA(h, cudaMemcpyAsync(h->b_prompts, prompts, sizeof(int32_t) * total,
                               on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice, s));
    L2_CUDA(h, cudaMemcpyAsync(h->b_len, lens, sizeof(int32_t) * B, cudaMemcpyHostToDevice, s));
    L2_CUDA(h, cudaMemcpyAsync(h->b_poff, poff.data(), sizeof(int32_t) * B, cudaMemcpyHostToDevice,
                               s));
    L2_CUDA(h, cudaMemcpyAsync(h->b_rmap, rmap.data(), sizeof(int32_t) * rmap.size(),
                               cudaMemcpyHostToDevice, s));
    // passes of up to `rows` prompt rows, in order: a sequence's earlier
    // positions are in its cache before its later ones attend to them
    for (long long start = 0; start < total; start += h->rows) {
        const int n = static_cast<int>(total - start < h->rows ? total - start : h->rows);
        const int st0 = static_cast<int>(start);
        bprefill_setup_kernel<<<(n + 127) / 128, 128, 0, s>>>(n, st0, h->b_rmap, h->b_prompts,
                                                              h->b_poff, V, h->b_token, h->b_pos,
                                                              h->b_seq, h->b_active, h->b_keys,
                                                              h->st);
        L2_CUDA(h, cudaGetLastError());
        L2_CUDA(h, enqueue_rows(h, 0, n, 0, 0, false, s, true));
        bprefill_handoff_kernel<<<(n + 127) / 128, 128, 0, s>>>(n, st0, h->b_rmap, h->b_len,
                                                                h->b_last, steps, h->b_out);
        L2_CUDA(h, cudaGetLastError());
    }
    bprefill_continue_kernel<<<(B + 127) / 128, 128, 0, s>>>(B, steps, h->b_len, h->b_out,
                                                             h->b_pos, h->b_token, h->b_active,
                                                             h->b_keys);
    L2_CUDA(h, cudaGetLastError());
    if (steps > 1) {
        int rc = capture_bstep(h, B, steps);
        if (rc != L2_OK) return rc;
        for (int i = 0; i < steps - 1; ++i) L2_CUDA(h, cudaGraphLaunch(h->bgraph, s));
    }
    L2_CUDA(h, cudaMemcpyAsync(out_tokens, h->b_out, sizeof(int32_t) * B * static_cast<size_t>(steps),
                               on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyDeviceToHost, s));
    if (on_device) return L2_OK;
    L2_CUDA(h, cudaStreamSynchronize(s));
    return check_device_error(h);
}

int l2_generate_batch_prefill(l2_handle* h, const int32_t* prompts, const int32_t* lens, int32_t B,
                              int32_t steps, int32_t* out_tokens) {
    return generate_batch_prefill_impl(h, prompts, lens, B, steps, out_tokens, false, nullptr);
}

int l2_generate_batch_prefill_device(l2_handle* h, const int32_t* d_prompts, const int32_t* lens,
                                     int32_t B, int32_t steps, int32_t* d_out, void* stream) {
    return generate_batch_prefill_impl(h, d_prompts, lens, B, steps, d_out, true,
                                       static_cast<cudaStream_t>(stream));
}

int l2_generate_prefill(l2_handle* h, const int32_t* prompt, int32_t n_prompt, int32_t steps,
                        int32_t* out_tokens) {
    return generate_prefill_impl(h, prompt, n_prompt, steps, out_tokens, false, nullptr);
}

int l2_generate_prefill_device(l2_handle* h, const int32_t* d_prompt, int32_t n_prompt,
                               int32_t steps, int32_t* d_out, void* stream) {
    return generate_prefill_impl(h, d_prompt, n_prompt, steps, d_out, true,
                                 static_cast<cudaStream_t>(stream));
}

int l2_generate_batch(l2_handle* h, const int32_t* prompts, const int32_t* lens, int32_t B,
                      int32_t steps, int32_t* out_tokens) {
    return generate_batch_impl(h, prompts, lens, B, steps, out_tokens, false, nullptr);
}

int l2_generate_batch_device(l2_handle* h, const int32_t* d_prompts, const int32_t* lens,
                             int32_t B, int32_t steps, int32_t* d_out, void* stream) {
    return generate_batch_impl(h, d_prompts, lens, B, steps, d_out, true,
                               static_cast<cudaStream_t>(stream));
}

int l2_generate_batch_sample(l2_handle* h, const int32_t* prompts, const int32_t* lens, int32_t B,
                             int32_t steps, float temperature, float topp, const float* uniforms,
                             int32_t* out_tokens) {
    return generate_batch_impl(h, prompts, lens, B, steps, out_tokens, false, nullptr, true,
                               temperature, topp, uniforms);
}

int l2_generate_batch_sample_device(l2_handle* h, const int32_t* d_prompts, const int32_t* lens,
                                    int32_t B, int32_t steps, float temperature, float topp,
                                    const float* d_uniforms, int32_t* d_out, void* stream) {
    return generate_batch_impl(h, d_prompts, lens, B, steps, d_out, true,
                               static_cast<cudaStream_t>(stream), true, temperature, topp,
                               d_uniforms);
}

int l2_time_kernel(l2_handle* h, int32_t kind, int32_t pos, int32_t iters, void* stream,
                   float* ms) {
    if (!h) return fail(nullptr, L2_EINVAL, "handle is NULL");
    if (kind < 0 || kind > 15 || iters < 1 || !ms || pos < 0 || pos >= h->cfg.seq_len)
        return fail(h, L2_EINVAL, "bad kind, iters, pos or output");
    // a prefill-only handle (max_batch 1, max_prefill > 1) times the GEMMs that
    // touch no KV cache (Wo, W1/W3, W2) on its max_prefill rows
    const bool prefill_gemm = kind >= 8 && kind <= 10 && h->cfg.max_batch < 2 && h->rows > 1;
    if (kind >= 6 && kind <= 13 && h->cfg.max_batch < 2 && !prefill_gemm)
        return fail(h, L2_EINVAL, "batched kernel kinds need a handle with max_batch > 1");
    if (kind >= 14 && !h->fused)
        return fail(h, L2_EINVAL, "kinds 14 and 15 need a handle with two kernels per layer");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (kind >= 6 && kind <= 13) {
        const int M = prefill_gemm ? h->rows : h->cfg.max_batch, bk = kind - 6;
        L2_CUDA(h, clear_device_error(h, s));
        bset_kernel<<<(M + 127) / 128, 128, 0, s>>>(M, pos, h->b_pos, h->b_token, h->b_active,
                                                    h->b_keys, h->st);
        L2_CUDA(h, cudaGetLastError());
        L2_CUDA(h, launch_bkind(h, bk, 0, 0, M, 0, 0, false, s));
        L2_CUDA(h, cudaEventRecord(h->ev0, s));
        for (int i = 0; i < iters; ++i)
            L2_CUDA(h, launch_bkind(h, bk, i % h->cfg.n_layers, 0, M, 0, 0, false, s));
        L2_CUDA(h, cudaEventRecord(h->ev1, s));
        L2_CUDA(h, cudaEventSynchronize(h->ev1));
        float t = 0.0f;
        L2_CUDA(h, cudaEventElapsedTime(&t, h->ev0, h->ev1));
        *ms = t / iters;
        return check_device_error(h);
    }
    init_state_kernel<<<1, 1, 0, s>>>(h->st, pos, 1, nullptr, nullptr, h->cfg.vocab_size,
                                      h->cfg.seq_len, 0, 0, nullptr, nullptr, 1);
    L2_CUDA(h, cudaGetLastError());
    // warm-up launch, then the timed loop
    L2_CUDA(h, launch_kind(h, kind, 0, s));
    L2_CUDA(h, cudaEventRecord(h->ev0, s));
    for (int i = 0; i < iters; ++i) L2_CUDA(h, launch_kind(h, kind, i % h->cfg.n_layers, s));
    L2_CUDA(h, cudaEventRecord(h->ev1, s));
    // a forward starts from zeroed fixed-point residual buffers
    if (kind >= 14)
        L2_CUDA(h, cudaMemsetAsync(h->fx, 0, fx_words(h->cfg.dim) * sizeof(long long), s));
    L2_CUDA(h, cudaEventSynchronize(h->ev1));
    float t = 0.0f;
    L2_CUDA(h, cudaEventElapsedTime(&t, h->ev0, h->ev1));
    *ms = t / iters;
    L2_CUDA(h, cudaStreamSynchronize(s));
    return check_device_error(h);
}

int l2_status(l2_handle* h, void* stream) {
    if (!h) return fail(nullptr, L2_EINVAL, "handle is NULL");
    L2_CUDA(h, cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
    L2_CUDA(h, cudaStreamSynchronize(h->stream));
    int err = 0;
    L2_CUDA(h, cudaMemcpy(&err, &h->st->err, sizeof(int), cudaMemcpyDeviceToHost));
    L2_CUDA(h, cudaMemset(&h->st->err, 0, sizeof(int)));
    return status_of(h, err);
}

int l2_watchdog_check(l2_handle* h, int64_t spin_cycles) {
    if (!h) return fail(nullptr, L2_EINVAL, "handle is NULL");
    if (spin_cycles < 1 || spin_cycles > kSpinLimitCycles)
        return fail(h, L2_EINVAL, "spin_cycles outside [1, 2e9]");
    L2_CUDA(h, cudaStreamSynchronize(h->stream));
    L2_CUDA(h, cudaMemsetAsync(&h->st->err, 0, sizeof(int), h->stream));
    watchdog_kernel<<<1, 32, 0, h->stream>>>(h->st, static_cast<long long>(spin_cycles));
    L2_CUDA(h, cudaGetLastError());
    L2_CUDA(h, cudaStreamSynchronize(h->stream));
    int err = 0;
    L2_CUDA(h, cudaMemcpy(&err, &h->st->err, sizeof(int), cudaMemcpyDeviceToHost));
    L2_CUDA(h, cudaMemset(&h->st->err, 0, sizeof(int)));
    return status_of(h, err);
}

int32_t l2_layer_kernels(const l2_handle* h) { return h ? (h->fused ? 2 : 5) : 0; }

double l2_kernel_bytes(const l2_handle* h, int32_t kind, int32_t pos) {
    if (!h) return 0.0;
    const double d = h->cfg.dim, F = h->cfg.hidden_dim, V = h->cfg.vocab_size, kvd = h->kvd;
    switch (kind) {
        case 0: return 4.0 * ((d + 2 * kvd) * d + 2 * d + d + 2 * kvd);
        case 1: return 4.0 * (2.0 * (pos + 1) * kvd + 2 * d);
        case 2: return 4.0 * (d * d + d + 2 * d);
        case 3: return 4.0 * (2 * F * d + 2 * d + F);
        case 4: return 4.0 * (d * F + F + 2 * d);
        case 5: return 4.0 * (V * d + 2 * d + V);
        // the two-kernels-per-layer blocks: weights once, the KV rows once per
        // kv head, the residual in and out in 8-byte fixed point (the FFN
        // block's output row in kFfnCopies copies)
        case 14: return 4.0 * ((d + 2 * kvd) * d + d * d + 2.0 * (pos + 1) * kvd + 2 * kvd + d) +
                        8.0 * (2 * kFfnCopies + 1) * d;
        case 15: return 4.0 * (3 * F * d + d) + 8.0 * 3 * d;
        default: break;
    }
    // batched kinds: fp32 operands once (weights, input rows), outputs, KV rows
    const bool prefill_gemm = kind >= 8 && kind <= 10 && h->cfg.max_batch < 2 && h->rows > 1;
    const double M = prefill_gemm ? h->rows : h->cfg.max_batch;
    if (kind >= 6 && M < 2) return 0.0;
    switch (kind) {
        case 6: return 4.0 * ((d + 2 * kvd) * d + M * d + M * (d + 2 * kvd));
        case 7: return 4.0 * M * (2.0 * (pos + 1) * kvd + 2 * d);
        case 8: return 4.0 * (d * d + M * d + 2 * M * d);
        case 9: return 4.0 * (2 * F * d + M * d + M * F);
        case 10: return 4.0 * (d * F + M * F + 2 * M * d);
        case 11: return 4.0 * (V * d + M * d);
        case 12: return 4.0 * (4 * M * d + M);  // embedding rows in; x, its pair, sums out
        case 13: return 4.0 * 6 * M;
        default: return 0.0;
    }
}

}  // extern "C"
