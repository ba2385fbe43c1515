/*
 * l2decode.h -- C ABI of the B300 (sm_103a) fp32 Llama-2 decode library.
 *
 * What it computes. One decode step of the Llama 2 architecture in fp32, as
 * the llama2.c pages describe the single-file C engine: in
 * "llama2.c｜Baby LLaMA-openAI维基百科" (openai.wiki), introduction, a
 * Llama-2 model trained in PyTorch has its weights saved as a raw binary file
 * and run by a ~500-line C file in fp32 with the architecture hard-coded; the
 * 新智元 llama2.c article (m.greenbasetech.com) says the same in the paragraph
 * before "感受魔力" and runs it as `./run out/model.bin` under "使用指南".
 * Per token: embedding row, then per layer RMSNorm, Q/K/V projections, RoPE,
 * causal multi-head attention over a KV cache, output projection + residual,
 * RMSNorm, SwiGLU feed-forward (W1 gate, W3 up, W2 down) + residual; then a
 * final RMSNorm, the vocabulary classifier and the greedy argmax. The pages
 * name the architecture without writing its formulas; the readings taken are:
 *   RMSNorm  out_i = g_i * x_i / sqrt(mean(x^2) + eps)
 *   RoPE     adjacent pairs (2i, 2i+1) of each head turn by
 *            pos * theta^(-2i/head_dim) (angles evaluated in double)
 *   scores   (q . k) / sqrt(head_dim), softmax over positions 0..pos
 *   SwiGLU   silu(W1 x) * (W3 x), silu(z) = z / (1 + exp(-z))
 *   greedy   the lowest index wins a tie
 *
 * Threading and streams. A handle is not thread-safe. Every call is
 * synchronous unless it takes a stream (the *_device calls), in which case the
 * work is queued on that stream and the call returns without waiting.
 *
 * Errors. Every int-returning call returns L2_OK (0) or a negative code below;
 * l2_last_error() gives a one-line description of the last failure on that
 * handle. No call aborts the process, traps, or hangs: device-side waits are
 * bounded and report L2_ETIMEOUT.
 */
#ifndef L2DECODE_H
#define L2DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Symbols of the shared library are exported explicitly; everything else in it
 * is hidden. */
#if defined(__GNUC__)
#define L2_API __attribute__((visibility("default")))
#else
#define L2_API
#endif

#define L2_OK 0
#define L2_EINVAL (-1)   /* bad config or argument (range, size, batch)          */
#define L2_ENOMEM (-2)   /* device or pinned-host allocation failed              */
#define L2_ECUDA (-3)    /* a CUDA runtime call failed (no device, launch error) */
#define L2_ETIMEOUT (-4) /* a bounded device-side wait gave up                   */
#define L2_EBLOB (-5)    /* blob size does not match the config                  */

/* Model configuration. Shapes from the pages: dim 288 / 6 layers / 6 heads
 * (openai.wiki introduction) and dim 512 / 8 layers / 8 heads / context 1024
 * (openai.wiki "训练示例"); larger shapes follow the same architecture.
 * Requirements: all sizes > 0; dim % n_heads == 0; head_dim = dim / n_heads
 * even and <= 256; n_heads % n_kv_heads == 0; dim % 4 == 0;
 * hidden_dim % 4 == 0; 1 <= max_batch <= 1024; 0 <= max_prefill <= 1024.
 * max_batch sequences get a KV cache each; the tensor-core path (batched
 * decode, prefill) is set up when max_batch > 1 or max_prefill > 1, with
 * row buffers for max(max_batch, max_prefill) rows.
 * rolling_positions: 0 (or <= seq_len) keeps every position below seq_len.
 * N > seq_len lets a sequence decode positions 0 .. N-1 (batch 1 and
 * batched decode): position p writes cache slot p % seq_len and attends over
 * the last seq_len positions (a rolling cache; the openai.wiki page lists
 * decoding beyond max_seq_len as a to-do that has to handle the KV cache,
 * "未排序的待办事项"); RoPE keeps the absolute position. Prompts (and the
 * prefill pass) stay below seq_len.
 * layer_kernels: how a batch-1 forward is split into kernels (the same
 * arithmetic either way, up to summation order). 5: QKV + RoPE + KV append,
 * attention, Wo + residual, W1/W3 + SwiGLU, W2 + residual, each streaming its
 * weights over every SM (for models whose layers are large). 2: an attention
 * block (one cluster of 8 CTAs per query head: its Q/K/V rows, attention and
 * its share of Wo) and an FFN block (W1/W3, SwiGLU and W2 per hidden-unit
 * slice), with the residual kept in 64-bit fixed point so that the CTAs' sums
 * are exact and independent of their order (for models whose per-kernel work
 * is too small to hide a kernel boundary; needs head_dim a multiple of 4 and at
 * most 128, 3 * head_dim a multiple of 16, and each CTA's weight slice within
 * shared memory). 0: 2 for models under 2 GB of weights where it fits, else 5. */
typedef struct {
    int32_t dim;               /* d, width of the residual stream            */
    int32_t hidden_dim;        /* F, SwiGLU hidden width                     */
    int32_t n_layers;          /* L                                          */
    int32_t n_heads;           /* H query heads                              */
    int32_t n_kv_heads;        /* KVH key/value heads (H % KVH == 0)         */
    int32_t vocab_size;        /* V                                          */
    int32_t seq_len;           /* S, KV-cache length (positions 0..S-1)      */
    float rope_theta;          /* 10000 in the Llama 2 architecture          */
    float norm_eps;            /* 1e-5                                       */
    int32_t max_batch;         /* sequences one handle can decode at once    */
    int32_t shared_classifier; /* 1: classifier = embedding table (no Wcls)  */
    int32_t max_prefill;       /* prompt positions one prefill pass takes    */
    int32_t rolling_positions; /* > seq_len: decode up to this many positions */
    int32_t layer_kernels;     /* batch-1 kernels per layer: 0 = chosen at create,
                                  5 or 2 (see below)                           */
} l2_config;

typedef struct l2_handle l2_handle;

/* Floats in a weight blob for cfg; 0 for an invalid config.
 * Blob layout (the pages say only "raw binary file"; this is the documented
 * order), fp32 little-endian, contiguous, every matrix row-major [out][in]
 * acting as y = W x, kvd = n_kv_heads * head_dim:
 *   E[V][d], g_att[L][d], Wq[L][d][d], Wk[L][kvd][d], Wv[L][kvd][d],
 *   Wo[L][d][d], g_ffn[L][d], W1[L][F][d], W2[L][d][F], W3[L][F][d],
 *   g_final[d], Wcls[V][d] (absent when shared_classifier = 1). */
L2_API size_t l2_blob_floats(const l2_config* cfg);

/* Creates a handle on the current CUDA device: validates cfg, allocates the
 * weights, KV caches and run state, copies blob (host memory, blob_floats
 * floats, read only during the call; the caller keeps ownership) to the
 * device and re-tiles it into the streaming layout, and builds the per-step
 * CUDA graph. *out receives the handle (NULL on failure).
 * Errors: L2_EINVAL (cfg), L2_EBLOB (size), L2_ENOMEM, L2_ECUDA. */
L2_API int l2_create(const l2_config* cfg, const float* blob, size_t blob_floats, l2_handle** out);

/* As l2_create, with the blob in device memory (d_blob, blob_floats floats,
 * read only during the call; the caller keeps ownership and may free it when
 * the call returns). For callers that already hold the weights on the GPU, or
 * that stream a large blob to the device in pieces instead of holding it in
 * host memory. Same errors as l2_create. */
L2_API int l2_create_from_device(const l2_config* cfg, const float* d_blob, size_t blob_floats,
                                 l2_handle** out);

/* One decode step for B sequences; sequence b consumes token tokens[b] at
 * position pos[b], writes its KV-cache slot pos[b] and attends over slots
 * 0..pos[b] (slots below pos[b] must hold that sequence's earlier steps;
 * re-running a lower pos overwrites its slot). Sequence b uses cache b.
 * tokens, pos: host arrays [B]. logits_out: host [B][V] floats or NULL.
 * With a rolling cache (rolling_positions > S) positions run up to
 * rolling_positions - 1, position p using slot p % S and the last min(p+1, S)
 * positions being attended.
 * Errors: L2_EINVAL for B < 1, B > max_batch, a token outside [0, V) or a
 * position outside [0, S) (rolling: [0, rolling_positions)). Synchronous. */
L2_API int l2_forward(l2_handle* h, const int32_t* tokens, const int32_t* pos, int32_t B,
               float* logits_out);

/* Same as l2_forward with device buffers owned by the caller (for example
 * PyTorch tensors): d_tokens, d_pos int32 [B], d_logits fp32 [B][V] or NULL.
 * Queued on `stream` (a cudaStream_t, NULL = legacy default stream); returns
 * without waiting. Device values are checked on the device: a token outside
 * [0, V) or a position outside [0, S) (rolling: [0, rolling_positions)) is
 * clamped, so that every access stays in bounds, and reported as L2_EINVAL by
 * l2_status (see there). */
L2_API int l2_forward_device(l2_handle* h, const int32_t* d_tokens, const int32_t* d_pos, int32_t B,
                      float* d_logits, void* stream);

/* Greedy generation for one sequence (cache 0), the loop of the single-file
 * engine (新智元 article, "使用指南": `./run out/model.bin` streams token ids):
 * forwards at positions 0 .. n_prompt+steps-2; position p consumes prompt[p]
 * while p < n_prompt, afterwards the previous argmax; no stop token.
 * out_tokens[k] (host, [steps]) is the argmax at position n_prompt-1+k.
 * The token stays on the device between steps; one copy in, one copy out.
 * Errors: L2_EINVAL for n_prompt < 1, steps < 1, n_prompt+steps-1 > S
 * (rolling: > rolling_positions), or a prompt id outside [0, V). Synchronous. */
L2_API int l2_generate(l2_handle* h, const int32_t* prompt, int32_t n_prompt, int32_t steps,
                int32_t* out_tokens);

/* Parallel prompt prefill of sequence 0 (cache 0): the n tokens at positions
 * pos0 .. pos0+n-1 go through one causal pass in which every projection is a
 * tensor-core GEMM over the n positions (3xTF32, fp32 accuracy) and position p
 * attends over cache slots 0..p; it writes cache slots pos0 .. pos0+n-1 and
 * computes the logits of every position, exactly what n consecutive
 * l2_forward calls compute (up to summation order). Slots below pos0 must
 * hold the sequence's earlier positions. The pages' engine feeds a prompt one
 * token per forward (新智元 article, "使用指南"); this pass computes the same
 * positions at once, so the weights are read once for the whole prompt.
 * tokens: host [n]; logits_out: host [n][V] or NULL.
 * Errors: L2_EINVAL for n < 1, n > max(max_batch, max_prefill) (or a handle
 * without the tensor-core path), pos0 < 0, pos0 + n > S, or a token outside
 * [0, V). Synchronous. */
L2_API int l2_prefill(l2_handle* h, const int32_t* tokens, int32_t n, int32_t pos0,
                      float* logits_out);

/* l2_generate with the prompt taken by one prefill pass (l2_prefill) instead
 * of n_prompt decode forwards; then steps-1 decode forwards as l2_generate.
 * Same output contract as l2_generate: out_tokens[k] is the argmax at position
 * n_prompt-1+k. Extra error: L2_EINVAL when n_prompt exceeds the prefill
 * capacity. Synchronous. */
L2_API int l2_generate_prefill(l2_handle* h, const int32_t* prompt, int32_t n_prompt,
                               int32_t steps, int32_t* out_tokens);

/* l2_generate_prefill with device buffers (d_prompt int32 [n_prompt], d_out
 * int32 [steps]), queued on `stream`; returns without waiting. A device prompt
 * id outside [0, V) is clamped and reported by l2_status. */
L2_API int l2_generate_prefill_device(l2_handle* h, const int32_t* d_prompt, int32_t n_prompt,
                                      int32_t steps, int32_t* d_out, void* stream);

/* l2_generate with device buffers: d_prompt int32 [n_prompt], d_out int32
 * [steps]; queued on `stream`, returns without waiting. Host-side checks as
 * l2_generate; a device prompt id outside [0, V) is clamped and reported by
 * l2_status. */
L2_API int l2_generate_device(l2_handle* h, const int32_t* d_prompt, int32_t n_prompt, int32_t steps,
                       int32_t* d_out, void* stream);

/* l2_generate drawing every generated token from the softmax of the logits
 * instead of taking the greedy choice. The pages print sampled stories and
 * mention the engine's C sampling code without stating its rule; the rule
 * taken: temperature 0 is the greedy choice; otherwise
 * p_i = exp((l_i - max) / temperature); with topp < 1 only the smallest set of
 * highest p whose mass reaches topp * total is kept (widened to ties of the
 * last token taken); the token is the first kept token, in increasing index
 * order, whose running sum of p exceeds u * (kept mass).
 * uniforms: host [steps], the caller's uniform random numbers in [0, 1), one
 * per generated token (the draws are reproducible from them).
 * Errors: as l2_generate, plus L2_EINVAL for temperature < 0, topp outside
 * (0, 1] or a uniform number outside [0, 1). Synchronous. */
L2_API int l2_generate_sample(l2_handle* h, const int32_t* prompt, int32_t n_prompt, int32_t steps,
                              float temperature, float topp, const float* uniforms,
                              int32_t* out_tokens);

/* l2_generate_sample with device buffers: d_prompt int32 [n_prompt],
 * d_uniforms fp32 [steps], d_out int32 [steps]; queued on `stream`, returns
 * without waiting. A device prompt id outside [0, V) is clamped and reported
 * by l2_status; uniform numbers are not checked. */
L2_API int l2_generate_sample_device(l2_handle* h, const int32_t* d_prompt, int32_t n_prompt,
                                     int32_t steps, float temperature, float topp,
                                     const float* d_uniforms, int32_t* d_out, void* stream);

/* Greedy generation for B independent sequences in lockstep (batched
 * decode). prompts: host, the B prompts concatenated; lens: host [B], each
 * >= 1; out_tokens: host [B][steps]. Sequence b runs forwards at positions
 * 0 .. lens[b]+steps-2 of its own cache; a sequence that has produced its
 * `steps` tokens idles while the others finish.
 * With a rolling cache (rolling_positions > S) a sequence runs up to
 * rolling_positions positions.
 * Errors: L2_EINVAL for B < 1 or > max_batch, a length < 1 or > S,
 * lens[b]+steps-1 > S (rolling: > rolling_positions), or an id outside
 * [0, V). Synchronous. */
L2_API int l2_generate_batch(l2_handle* h, const int32_t* prompts, const int32_t* lens, int32_t B,
                      int32_t steps, int32_t* out_tokens);

/* l2_generate_batch with the prompts and the output in device memory:
 * d_prompts int32 [sum of lens], d_out int32 [B][steps]; `lens` stays a HOST
 * array [B] (the lockstep schedule is planned on the host). Queued on
 * `stream`, returns without waiting. Host-side checks as l2_generate_batch;
 * a device prompt id outside [0, V) is clamped and reported by l2_status. */
L2_API int l2_generate_batch_device(l2_handle* h, const int32_t* d_prompts, const int32_t* lens,
                                    int32_t B, int32_t steps, int32_t* d_out, void* stream);

/* l2_generate_batch with every prompt taken by prefill passes: the prompt
 * positions of all B sequences become rows of the tensor-core path (passes of
 * up to max(max_batch, max_prefill) rows, in order), each row writing its own
 * sequence's cache; the argmax of a sequence's last prompt position is its
 * first token, and the sequences then advance in lockstep for the remaining
 * steps - 1 tokens. Same arguments, output and errors as l2_generate_batch
 * (plus L2_EINVAL when max_batch == 1). Synchronous. */
L2_API int l2_generate_batch_prefill(l2_handle* h, const int32_t* prompts, const int32_t* lens,
                                     int32_t B, int32_t steps, int32_t* out_tokens);

/* l2_generate_batch_prefill with device prompts and output (as
 * l2_generate_batch_device; lens a HOST array [B]). Queued on `stream`,
 * returns without waiting. */
L2_API int l2_generate_batch_prefill_device(l2_handle* h, const int32_t* d_prompts,
                                            const int32_t* lens, int32_t B, int32_t steps,
                                            int32_t* d_out, void* stream);

/* l2_generate_batch with temperature / top-p sampling of the generated tokens
 * (the rule of l2_generate_sample, applied to each sequence's logits row).
 * uniforms: host fp32 [B][steps], each in [0, 1): uniforms[b * steps + k]
 * draws sequence b's k-th generated token; temperature <= 0 is the greedy
 * choice. Needs a handle with max_batch > 1.
 * Errors: as l2_generate_batch, plus L2_EINVAL for a NULL uniforms array,
 * temperature < 0, topp outside (0, 1], a uniform outside [0, 1), or
 * max_batch == 1. Synchronous. */
L2_API int l2_generate_batch_sample(l2_handle* h, const int32_t* prompts, const int32_t* lens,
                                    int32_t B, int32_t steps, float temperature, float topp,
                                    const float* uniforms, int32_t* out_tokens);

/* l2_generate_batch_sample with device buffers: d_prompts int32 [sum of
 * lens], d_uniforms fp32 [B][steps], d_out int32 [B][steps]; lens a HOST
 * array [B]. Queued on `stream`, returns without waiting; a device prompt id
 * outside [0, V) is clamped and reported by l2_status, uniform numbers are not
 * checked. */
L2_API int l2_generate_batch_sample_device(l2_handle* h, const int32_t* d_prompts,
                                           const int32_t* lens, int32_t B, int32_t steps,
                                           float temperature, float topp,
                                           const float* d_uniforms, int32_t* d_out,
                                           void* stream);

/* Status of the device-side work queued by the *_device calls, which return
 * before it runs: waits for `stream` (a cudaStream_t, NULL = legacy default
 * stream) and the handle's own stream, reads the handle's device error word,
 * clears it and returns what it holds: L2_OK; L2_EINVAL when a device token
 * id or position was out of range (the kernels clamped it, so the results are
 * not those of the input); L2_ETIMEOUT when a bounded device wait gave up.
 * The word accumulates over *_device calls until l2_status reads it; every
 * synchronous call clears it when it starts and reports its own work itself,
 * so call l2_status before the next synchronous call on the handle.
 * Errors: as listed, plus L2_ECUDA. */
L2_API int l2_status(l2_handle* h, void* stream);

/* Test hook of the failure-detection path. Every wait of a decode kernel on a
 * bulk-copy completion is bounded: when it gives up, the kernel sets the
 * handle's device error word, drains its own copies and returns, and the call
 * reports L2_ETIMEOUT. This hook runs that bounded wait, the same device
 * routine, on an mbarrier that nothing arrives at (no copy in flight), limited
 * to spin_cycles SM clock cycles, so that it gives up; the error word is then
 * read, cleared and reported as by a synchronous call. Returns L2_ETIMEOUT
 * when the wait gave up as designed; the handle stays usable.
 * Errors: L2_EINVAL for spin_cycles outside [1, 2e9], L2_ECUDA. Synchronous. */
L2_API int l2_watchdog_check(l2_handle* h, int64_t spin_cycles);

/* Clears KV cache `seq` (-1: all caches) to zero. Errors: L2_EINVAL. */
L2_API int l2_reset(l2_handle* h, int32_t seq);

/* Frees every device and host resource of h. NULL is accepted. */
L2_API void l2_destroy(l2_handle* h);

/* Text of the last error on h (or, when h is NULL, of the last failed
 * l2_create / l2_create_from_device on the calling thread). The pointer stays
 * valid until the next call on h (or the next failed create on that thread). */
L2_API const char* l2_last_error(const l2_handle* h);

/* Measurement hook: launches one kernel kind of the step `iters` times on
 * `stream`, cycling over layers, bracketed by CUDA events, and writes the mean
 * duration of one launch in milliseconds to *ms. Batch-1 kinds: 0 QKV+RoPE,
 * 1 attention, 2 Wo+residual, 3 W1/W3+SwiGLU, 4 W2+residual,
 * 5 classifier+argmax. Batched kinds (handles with max_batch > 1; all
 * max_batch rows at position pos): 6 QKV GEMM, 7 attention, 8 Wo GEMM,
 * 9 W1/W3 GEMM, 10 W2 GEMM, 11 classifier GEMM + argmax, 12 embedding gather
 * (residual rows, their tf32 pair and sums of squares; the RMSNorms are folded
 * into the GEMMs that consume them),
 * 13 advance; a handle with max_batch 1 and max_prefill > 1 times kinds
 * 8-10 (the GEMMs that touch no KV cache) on its max_prefill rows, the GEMMs of
 * a prefill pass. Kinds 14 and 15 (handles that run two kernels per layer, see
 * l2_layer_kernels): 14 the attention block (RMSNorm, Q/K/V, RoPE, KV append,
 * attention, Wo, residual), 15 the FFN block (RMSNorm, W1/W3, SwiGLU, W2,
 * residual), at batch 1. It reads and writes the handle's own run state (the KV cache
 * contents are left as they were, except slot `pos` of the caches used).
 * Errors: L2_EINVAL, L2_ECUDA. Synchronous. */
L2_API int l2_time_kernel(l2_handle* h, int32_t kind, int32_t pos, int32_t iters, void* stream,
                   float* ms);

/* Kernels per layer of the batch-1 forward this handle runs: 5 (Q/K/V, attention,
 * Wo, W1/W3, W2) or 2 (attention block, FFN block; l2_config.layer_kernels).
 * 0 for a NULL handle. */
L2_API int32_t l2_layer_kernels(const l2_handle* h);

/* Algorithmic bytes one launch of `kind` reads and writes at position pos
 * (fp32 weights once + activations + KV rows; batched kinds count max_batch
 * rows). 0 for an invalid kind. */
L2_API double l2_kernel_bytes(const l2_handle* h, int32_t kind, int32_t pos);

/* Test and measurement hook of the batched path's tensor-core GEMM:
 * C[M][N] = A[M][K] * W[N][K]^T, every matrix fp32 row-major in device memory
 * owned by the caller (16-byte aligned). The operands are split into tf32
 * (hi, lo) pairs and multiplied as A_hi W_hi + A_hi W_lo + A_lo W_hi on the
 * tcgen05 tensor cores with fp32 accumulation (the 3xTF32 scheme), the kernel
 * that carries every projection of batched decode. Allocates and frees its
 * split buffers; synchronous on `stream`. With iters > 0 it then times `iters`
 * launches of the GEMM kernel alone (CUDA events on `stream`) and writes the
 * mean milliseconds per launch to *ms.
 * Errors: L2_EINVAL (NULL or misaligned pointer, M or N < 1, K < 4 or not a
 * multiple of 4, iters < 0), L2_ENOMEM, L2_ECUDA, L2_ETIMEOUT. */
L2_API int l2_gemm_tf32x3(const float* d_A, const float* d_W, float* d_C, int32_t M, int32_t N,
                          int32_t K, int32_t iters, float* ms, void* stream);

/* Largest vocabulary l2_classify_greedy_noalloc accepts: its logits live in a
 * fixed device array of this many floats (1 MiB), after a 256-byte state block. */
#define L2_NOALLOC_MAX_VOCAB 262144

/* Final RMSNorm + vocabulary classifier + greedy argmax of one hidden state,
 * without allocating any memory. The pages have no counterpart: this is a
 * library convenience for callers that cannot call cudaMalloc, such as a host
 * program whose device memory belongs to another framework's arena, or a
 * serving loop that must not stall its other streams on cudaMalloc/cudaFree.
 * It computes logits = Wcls * rmsnorm(x, gain) and the lowest index of the
 * largest logit, with the same kernel as the classifier of l2_forward.
 *   d_x      device fp32 [dim], the hidden state after the last layer
 *   d_gain   device fp32 [dim], the final RMSNorm gain
 *   d_wcls   device fp32 [vocab][dim], row-major classifier
 *            (all three 16-byte aligned, read only, owned by the caller)
 *   d_token  device int32 [1], output: the greedy token, or -1 when a
 *            bounded device wait gave up
 *   d_logit  device fp32 [1], output, or NULL: the logit of that token
 * Queued on `stream` (a cudaStream_t, NULL = legacy default stream); returns
 * without waiting.
 * Scratch: a file-scope device array of 256 + 4 * L2_NOALLOC_MAX_VOCAB bytes,
 * which every GPU that loads the library holds until the process exits. All
 * calls on a device share it and it keeps the last call's contents; each call
 * clears what must start at zero itself. Calls that overlap on the GPU (on
 * unordered streams, or from several threads) race on it: order them.
 * The first call on a device, made with that device current, looks up the
 * array's device address and sets kernel attributes; make that first call
 * before any stream capture.
 * Errors (return code only; l2_last_error does not cover this call):
 * L2_EINVAL for a NULL input or token pointer, vocab outside
 * [1, L2_NOALLOC_MAX_VOCAB], dim not a multiple of 4 in [4, 16384], eps < 0 or
 * a pointer that is not 16-byte aligned; L2_ECUDA when a CUDA call fails. */
L2_API int l2_classify_greedy_noalloc(const float* d_x, const float* d_gain, const float* d_wcls,
                                      int32_t dim, int32_t vocab, float norm_eps,
                                      int32_t* d_token, float* d_logit, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* L2DECODE_H */
