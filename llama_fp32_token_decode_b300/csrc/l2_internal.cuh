// l2_internal.cuh -- device helpers and launch-parameter structs shared by the
// kernels of the decode library (sm_103a only).
#pragma once

#include <cuda.h>  // CUtensorMap and its enums (types only; the encoder is fetched at run time)
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/l2decode.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "this library targets sm_103a (Blackwell) only"
#endif

namespace l2 {

// Device error word bits (L2State::err).
enum : int {
    ERR_TIMEOUT_TMA = 1,   // a bulk-copy completion wait gave up
    ERR_BAD_PLAN = 2,      // a kernel received an impossible launch plan
    ERR_NAN = 4,           // the classifier met a NaN logit
    ERR_BAD_INPUT = 8,     // a device token id or position was out of range (clamped)
};

// Bound for every device-side spin: about one second at 2 GHz.
constexpr long long kSpinLimitCycles = 2000000000LL;

// Device-resident decode state of the batch-1 path. The classifier's last CTA
// advances it, so consecutive forwards need no host round trip.
struct L2State {
    int pos;            // position the next forward consumes
    int token;          // token the next forward consumes
    int n_prompt;       // generate: prompt length
    int mode;           // 0 = single forward, 1 = generate, 2 = generate with sampling
    int last_argmax;    // greedy choice of the last forward
    int err;            // ERR_* bits
    const int* prompt;  // generate: device prompt [n_prompt]
    int* out_tokens;    // generate: device output [steps]
    unsigned long long argmax_key;  // packed (orderable value, ~index) max
    unsigned int cls_done;          // classifier CTAs finished this forward
    unsigned int pad;
    // mode 2 (generate with sampling): the sampling kernel, not the classifier,
    // chooses the token and advances the position
    float temperature;
    float topp;
    const float* uniforms;  // one uniform number in [0, 1) per generated token
};

struct SampleArgs {
    L2State* st;
    const float* logits;    // [V] of the forward just computed
    int vocab;
};

enum Epilogue : int { EPI_QKV_ROPE = 0, EPI_RESIDUAL = 1, EPI_SWIGLU = 2, EPI_CLASSIFIER = 3 };

// Launch plan of one streaming matvec y = W xs (W row-major [R][K]).
struct MatvecPlan {
    int R, K;             // rows, columns
    int unit;             // rows kept together in one CTA (2 for pair epilogues)
    int rows_per_stage;   // TR: full rows per ring stage (1 when rows are chunked)
    int chunks_per_row;   // NCH: >1 splits a row over several stages
    int chunk_floats;     // floats per chunk (K when NCH == 1)
    int warps_per_row;    // WPR: consumer warps sharing one row of a slot
    int rows_per_warp;    // RPW: rows one warp handles per slot
    int stage_floats;     // ring slot size in floats (multiple of 32)
    int nstages;          // ring depth
    int grid;             // CTAs
    int max_rows_per_cta; // bound used to size the row-result buffer
    size_t smem_bytes;    // dynamic shared memory
};

struct MatvecArgs {
    const float* W;
    MatvecPlan plan;
    // prologue: xs = norm(src) * gain (gain != nullptr) or xs = src
    const float* src;      // input vector [K] (ignored when emb != nullptr)
    const float* gain;     // RMSNorm gain [K] or nullptr
    float eps;
    const float* emb;      // layer-0 QKV: src = emb[token] (token from state)
    float* x_init;         // layer-0 QKV: CTA 0 copies emb[token] here
    // epilogue
    float* out;            // RESIDUAL: x (+=); SWIGLU: hb; CLASSIFIER: logits
    // QKV + RoPE + KV append
    float* q_out;          // [d]
    float* k_cache;        // this layer's K cache, head-major [KVH][S][hd]
    float* v_cache;        // this layer's V cache
    const float2* rope;    // [S][hd/2] (cos, sin)
    int d, kvd, head_dim, seq_len, vocab;
    // state
    L2State* st;
    uint64_t l2_policy;    // createpolicy descriptor for the weight stream
    // two-kernels-per-layer path: the input vector in fixed point (instead of
    // src) and a fixed-point buffer CTA 0 zeroes (n entries)
    const long long* src_fixed;  // kFfnCopies copies of the row, summed
    long long* zero_fixed;
    int zero_n;
};

// Small-model batch-1 forward in two kernels per layer (fused_small.cu). The
// residual stream lives in 64-bit fixed point (value * 2^32) so that many CTAs
// can add into it with integer atomics, whose result does not depend on their
// order.
constexpr int kFusedCluster = 8;  // CTAs per query head in the attention block
// Copies of the FFN block's output row: its CTAs add into copy (CTA mod
// kFfnCopies), so each output address takes half of the CTAs' atomic adds
// (they serialise per address in L2); the next kernel sums the copies.
// Measured 15M / 44M / 110M: 2 copies +3.6 / +0.6 / -1.0 %, 4 copies +2.4 /
// +0.2 / -1.8 %, 8 copies +2.9 / -0.6 / -2.3 % against one.
constexpr int kFfnCopies = 2;

struct FAttnArgs {
    const float* wqkv;     // this layer's [d + 2 kvd][d]
    const float* wo_h;     // this layer's Wo re-tiled per head: [H][d][hd]
    const float* g_att;    // this layer's attention RMSNorm gain [d]
    const float* emb;      // layer 0: the input row is emb[token]
    const long long* x_in; // residual entering the layer (null at layer 0)
    long long* x_mid;      // += x_in + sum over heads of Wo_h att_h (zero on entry)
    long long* x_zero;     // zeroed here: the FFN block's output buffer
    float* k_cache;        // this layer's caches, head-major [KVH][S][hd]
    float* v_cache;
    const float2* rope;    // [positions][hd/2]
    L2State* st;
    int d, kvd, hd, H, KVH, S, vocab;
    float eps;
    uint64_t l2_policy;
    int smem_bytes;
};

struct FFfnArgs {
    const float* w13;      // this layer's interleaved W1/W3 rows [2F][d]
    const float* w2t;      // this layer's W2 transposed: [F][d]
    const float* g_ffn;    // this layer's FFN RMSNorm gain [d]
    const long long* x_mid;  // residual after attention
    long long* x_out;      // += x_mid + W2 (silu(W1 xn) * W3 xn) (zero on entry)
    long long* x_zero;     // zeroed here: the next layer's attention output buffer
    int* err;
    int d, F;
    float eps;
    uint64_t l2_policy;
    int smem_bytes;
};

struct AttnArgs {
    const float* q;        // [d] (RoPE applied)
    const float* k_cache;  // this layer: [KVH][S][hd]
    const float* v_cache;
    float* att;            // [d] output
    int n_heads, n_kv_heads, head_dim, seq_len;
    int nsplit;            // CTAs per head = cluster size (<= 16)
    L2State* st;
};

// Fused epilogues of the batched 3xTF32 GEMM (gemm_tf32x3.cu).
enum GemmEpilogue : int {
    GEPI_STORE = 0,     // out[r][c] = acc
    GEPI_RESIDUAL = 1,  // out[r][c] += acc
    GEPI_SWIGLU = 2,    // interleaved W1/W3 columns -> hb (tf32 hi/lo pair)
    GEPI_QKV_ROPE = 3,  // q rows rotated to q; k rotated and v appended to each row's cache
    GEPI_ARGMAX = 4,    // per-row packed (value, index) atomicMax; logits stored if out != null
};

// The four operand maps of one GEMM launch: X (hi, lo) [1][Mcap][K] and
// W (hi, lo) [L][N][K].
struct GemmMaps {
    CUtensorMap a_hi, a_lo, b_hi, b_lo;
    CUtensorMap b_raw;  // W in fp32, [L][N][K] (split in shared memory: GemmArgs::conv)
};

struct GemmArgs {
    int row0;             // first row (sequence) of this launch
    int M, N, K;          // rows (sequences) from row0, output columns, reduction length
    int layer;            // weight map z coordinate
    int ldc;              // row stride of out
    float* out;           // STORE / RESIDUAL / ARGMAX (logits, may be null)
    float* out_hi;        // SWIGLU: hb hi [M][N/2]
    float* out_lo;        // SWIGLU: hb lo
    // QKV + RoPE + KV append
    float* q;             // [M][d]
    float* k_cache;       // this layer's K cache of sequence 0; sequence r at + r*cache_seq
    float* v_cache;
    const float2* rope;   // [S][hd/2]
    const int* pos;       // [M] position of each row
    const int* active;    // [M] 0 = finished sequence (no KV write) or null
    const int* seq;       // [M] KV cache of each row, or null (row r uses cache r)
    int d, kvd, head_dim, seq_len;
    int rope_positions;   // positions of the RoPE table (> seq_len: the cache rolls)
    size_t cache_seq;     // floats of one sequence's cache (all layers)
    unsigned long long* argmax_keys;  // ARGMAX: [M]
    int* err;             // ERR_* bits
    int stages;           // ring depth (set by launch_gemm from the plan)
    int conv;             // drained launches read W once, in fp32 (GemmMaps::b_raw),
                          // and split it into the tf32 pair in shared memory
    int a_rows;           // rows of an A tile the maps load: 128, or 64 when at most
                          // 64 rows are ever multiplied (M = 64 MMAs then)
    // RMSNorm folded into the GEMM that consumes the normalised rows. The
    // weights carry the norm gain (W[n][k] * g[k]) and A holds the raw rows x
    // (tf32 pair), so the consumer scales row r of its result by
    // 1 / sqrt(ss_r / K + eps), ss_r = the sum of squares of x[r] as the sum of
    // ss_count partials at ss_in[r * ss_stride] (fixed order; ss_stride a
    // multiple of 4). Null: no norm.
    const float* ss_in;
    int ss_count, ss_stride;
    float eps;
    // RESIDUAL producer of such rows: also writes the new rows as a tf32 pair
    // (x_hi, x_lo) and its partial sums of squares (two slots per N tile, at
    // ss_out[r * ss_stride + 2 * tile], the second 0 unless warps split the
    // tile's columns). Null: not produced.
    float* x_hi;
    float* x_lo;
    float* ss_out;
};

// Batched decode (batched.cu). Row b of every [M][...] array is sequence b.
// Start of a batched step: the embedding rows of the tokens become the
// residual rows x, their tf32 pair (the first QKV GEMM's A operand, the norm
// being folded into that GEMM) and their sums of squares.
struct BNormArgs {
    int row0;              // rows row0 .. row0 + gridDim.x - 1
    float* x;              // [rows][d] residual rows, set to emb[token]
    const float* emb;      // embedding table [V][d]
    const int* token;      // [M]
    float* xn_hi;          // [M][d] x as a tf32 pair
    float* xn_lo;
    float* ss_out;         // [M][ss_stride]: slot 0 = sum of squares of x[r]
    int ss_stride;
    int d, vocab;
    const int* pos;        // [M] position of each row: checked against [0, pmax)
    int pmax;
    int* err;              // ERR_BAD_INPUT when a token or position is out of range
};

struct BAttnArgs {
    int row0;              // sequences row0 .. row0 + gridDim.y - 1
    const float* q;        // [rows][d], RoPE applied
    const float* k_cache;  // layer l of sequence 0; sequence b at + b * cache_seq
    const float* v_cache;
    float* att_hi;         // [M][d] output, tf32 pair
    float* att_lo;
    const int* pos;        // [M]
    const int* active;     // [M] or null
    const int* seq;        // [M] KV cache of each row, or null (row b uses cache b)
    int d, n_heads, n_kv_heads, head_dim, seq_len;
    size_t cache_seq;
};

// Sampling parameters of a batched generation, device-resident (written
// before the step graph replays, so the graph does not depend on them).
struct SampleParams {
    float temperature, topp;
    const float* uniforms;  // [B][steps]: sequence b's uniform for its k-th token
};

// The per-sequence advance of a batched generation with sampling (sample.cu).
struct BSampleArgs {
    int row0;
    int steps, vocab;
    const SampleParams* params;
    const float* logits;         // [M][V] of this step
    unsigned long long* keys;    // [M] packed argmax keys (reset to 0 here)
    int* last;
    int* pos;
    int* token;
    int* active;
    const int* len;
    const int* poff;
    const int* prompts;
    int* out;                    // [M][steps]
};

struct BAdvanceArgs {
    int row0;                    // rows row0 .. row0 + M - 1
    int M;
    int mode;                    // 0 = forward only, 1 = generate
    int steps;                   // generate: tokens per sequence (row stride of out)
    unsigned long long* keys;    // [M] packed argmax keys (reset to 0 here)
    int* last;                   // [M] greedy choice of this step
    int* pos;
    int* token;
    int* active;
    const int* len;              // [M] prompt lengths
    const int* poff;             // [M] offsets into prompts
    const int* prompts;          // concatenated prompts
    int* out;                    // [M][steps]
};

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Cluster barrier in two halves. A CTA may write another CTA's shared memory
// only once that CTA is running: every CTA arrives early (relaxed, no
// ordering) and waits just before its first remote write.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_all() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on a phase of an mbarrier; false once `limit` SM clock cycles
// have passed without the phase completing.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  long long limit = kSpinLimitCycles) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit) return false;
    }
    return true;
}

// The same wait with acquire at cluster scope, for phases completed by other
// CTAs' st.async writes into this CTA's shared memory.
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t* bar, uint32_t parity,
                                                          long long limit = kSpinLimitCycles) {
    const long long t0 = clock64();
    for (;;) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(smem_u32(bar)), "r"(parity)
            : "memory");
        if (ok) return true;
        if (clock64() - t0 > limit) return false;
    }
}

// Address of `p` (this CTA's shared memory) in the shared memory window of
// cluster rank `rank`.
__device__ __forceinline__ uint32_t cluster_smem(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

// Non-blocking stores into another CTA's shared memory that count their bytes
// on that CTA's mbarrier (at `bar`, in the same rank's window).
__device__ __forceinline__ void st_async_f2(uint32_t addr, float x, float y, uint32_t bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(
            addr),
        "f"(x), "f"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void st_async_f4(uint32_t addr, float4 v, uint32_t bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::
            "r"(addr),
        "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void st_async_f1(uint32_t addr, float x, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(
                     addr),
                 "r"(__float_as_uint(x)), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ uint64_t make_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t make_policy_evict_last(float frac) {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, %1;" : "=l"(p) : "f"(frac));
    return p;
}

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes % 16 == 0,
// both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Nearest tf32 value of v (10 explicit mantissa bits, ties away from zero);
// infinities and NaN pass through. v - tf32_round(v) is exact in fp32.
// v with its 13 low mantissa bits cleared: the part of v a tf32 operand keeps.
__device__ __forceinline__ float tf32_trunc(float v) {
    return __uint_as_float(__float_as_uint(v) & 0xffffe000u);
}

__device__ __forceinline__ float tf32_round(float v) {
    uint32_t u = __float_as_uint(v);
    if ((u & 0x7f800000u) != 0x7f800000u) u = (u + 0x1000u) & 0xffffe000u;
    return __uint_as_float(u);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
        v = w > v ? w : v;
    }
    return v;
}

// Key that orders (value, index) pairs by value, then by lower index; NaN maps
// below every number. -0 and +0 compare equal, as in a plain float comparison.
__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
    uint32_t u = __float_as_uint(v == 0.0f ? 0.0f : v);
    if (v != v) {
        u = 0u;
    } else {
        u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    }
    return (static_cast<unsigned long long>(u) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(idx));
}

__device__ __forceinline__ int argmax_key_index(unsigned long long k) {
    return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFull));
}

// ---------------------------------------------------------------- host launchers

// matvec.cu
MatvecPlan plan_matvec(int R, int K, int unit, int num_sms);
int matvec_threads();
cudaError_t launch_matvec(int epi, const MatvecArgs& a, cudaStream_t s, bool pdl);
cudaError_t set_matvec_smem_limits();

// attention.cu
int attn_nsplit(int n_heads, int seq_len, int num_sms);
cudaError_t prepare_attention();
int attn_cluster_ok(int head_dim, int nsplit, int n_heads);
cudaError_t launch_attention(const AttnArgs& a, cudaStream_t s, bool pdl);

// gemm_tf32x3.cu
cudaError_t make_gemm_map(CUtensorMap* map, const float* base, long long inner, long long rows,
                          long long layers, int box_rows);
struct GemmPlan {
    int bn;      // output tile width (64 or 128 columns)
    int ksplit;  // CTAs of a cluster that split K (1..8)
    int stages;  // shared-memory ring depth
};
// Clusters of each (tile width, split, ring depth) that the device runs at
// once, measured with cudaOccupancyMaxActiveClusters at set-up.
struct GemmOccupancy {
    int clusters[2][3][9][7];  // [A tile 128 / 64 rows][tile width 64 / 128 / 256][ksplit][stages]
    int num_sms;
};
cudaError_t prepare_gemm(GemmOccupancy* occ);
GemmPlan plan_gemm(const GemmOccupancy& occ, int M, int N, int K, int max_bn = 256,
                   int a_rows = 128);
GemmPlan plan_split(const GemmOccupancy& occ, int bn, int M, int N, int K, int a_rows = 128);
cudaError_t launch_gemm(int epi, const GemmPlan& p, const GemmMaps& m, const GemmArgs& g,
                        cudaStream_t s, bool pdl);
cudaError_t launch_split_tf32(const float* x, float* hi, float* lo, long long n, cudaStream_t s);
// The same split of gain-scaled weights: element k of every row of layer l
// is multiplied by gain[l * K + k] first ([layers][rows][K] weights).
cudaError_t launch_split_tf32_gain(const float* x, const float* gain, long long K, long long rows,
                                   long long layers, float* hi, float* lo, cudaStream_t s);
// The gain-scaled weights themselves in fp32 (what the GEMMs that split W in
// shared memory read).
cudaError_t launch_scale_gain(const float* x, const float* gain, long long K, long long rows,
                              long long layers, float* out, cudaStream_t s);
// Whether launches of this plan take the drained (and, on 64-row handles,
// split-in-shared-memory) build: more than 16 K-blocks per CTA.
bool gemm_drained(const GemmPlan& p, int K);

// batched.cu
cudaError_t launch_brmsnorm(const BNormArgs& a, int M, cudaStream_t s, bool pdl);
cudaError_t launch_battn(const BAttnArgs& a, int M, cudaStream_t s, bool pdl);
cudaError_t launch_badvance(const BAdvanceArgs& a, cudaStream_t s, bool pdl);

// sample.cu
cudaError_t launch_sample(const SampleArgs& a, cudaStream_t s, bool pdl);
cudaError_t launch_bsample(const BSampleArgs& a, int M, cudaStream_t s, bool pdl);

// fused_small.cu
// Whether the two-kernels-per-layer path fits this shape; fills the launch
// shared-memory sizes of the two kernels and the FFN block's grid.
bool plan_fused(FAttnArgs& a, FFfnArgs& f, int num_sms, size_t smem_optin, int* ffn_grid);
cudaError_t prepare_fused(const FAttnArgs& a, const FFfnArgs& f);
cudaError_t launch_fattn(const FAttnArgs& a, cudaStream_t s, bool pdl);
cudaError_t launch_fffn(const FFfnArgs& f, int grid, cudaStream_t s, bool pdl);

// layout.cu
cudaError_t launch_interleave_rows(float* dst, const float* a, const float* b, long long rows,
                                   int cols, cudaStream_t s);
// dst[l][h][r][e] = src[l][r][h*hd + e]: Wo [L][d][d] as per-head column blocks.
cudaError_t launch_retile_heads(float* dst, const float* src, int layers, int d, int hd,
                                cudaStream_t s);
// dst[l][c][r] = src[l][r][c]: per-layer transpose of [rows][cols].
cudaError_t launch_transpose_layers(float* dst, const float* src, int layers, int rows, int cols,
                                    cudaStream_t s);

}  // namespace l2
