// batched.cu -- the non-GEMM kernels of batched decode: B independent
// sequences advance one position per step in lockstep, each with its own
// position, token and KV cache (the decode step of the llama2.c pages' fp32
// engine, applied to B sequences at once). The projections of the step run in
// the 3xTF32 tensor-core GEMM (gemm_tf32x3.cu); this file holds
//   brmsnorm_kernel   embedding gather at the start of a step: the residual
//                     rows, their tf32 (hi, lo) pairs and sums of squares for
//                     the first QKV GEMM (every RMSNorm of the step is folded
//                     into the GEMM that consumes it: gains into the weights,
//                     the row scale into its epilogue)
//   battn_kernel      causal attention of every (row, head) over the row's KV
//                     cache (its own sequence's; in a prefill every row is a
//                     position of one sequence), ragged lengths pos + 1,
//                     output as a tf32 pair for the Wo GEMM
//   badvance_kernel   greedy choice per sequence and the move to the next
//                     position (prompt tokens are forced, then the argmax).
#include <math.h>

#include "l2_internal.cuh"

namespace l2 {

namespace {

constexpr int kNormThreads = 128;
constexpr int kBAttnThreads = 128;
constexpr int kBAttnWarps = kBAttnThreads / 32;

__global__ void __launch_bounds__(kNormThreads) brmsnorm_kernel(const BNormArgs a) {
    pdl_launch_dependents();
    pdl_wait();
    const int b = a.row0 + blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.d, d4 = d >> 2;
    float4* x4 = reinterpret_cast<float4*>(a.x + static_cast<size_t>(b) * d);
    // a token or position outside its range (device inputs are not checked
    // on the host) is reported; the token is clamped so that the read stays
    // inside the table, positions are clamped by their readers
    const int raw = __ldcg(a.token + b);
    const int tok = min(max(raw, 0), a.vocab - 1);
    if (tid == 0 && a.err != nullptr) {
        const int p = __ldcg(a.pos + b);
        if (raw != tok || p < 0 || p >= a.pmax) atomicOr(a.err, ERR_BAD_INPUT);
    }
    const float4* src4 = reinterpret_cast<const float4*>(a.emb + static_cast<size_t>(tok) * d);
    float4* hi4 = reinterpret_cast<float4*>(a.xn_hi + static_cast<size_t>(b) * d);
    float4* lo4 = reinterpret_cast<float4*>(a.xn_lo + static_cast<size_t>(b) * d);
    __shared__ float s_part[kNormThreads / 32];
    float ss = 0.0f;
    for (int i = tid; i < d4; i += kNormThreads) {
        const float4 v = __ldcg(src4 + i);
        x4[i] = v;
        const float4 h = make_float4(tf32_round(v.x), tf32_round(v.y), tf32_round(v.z), tf32_round(v.w));
        hi4[i] = h;
        lo4[i] = make_float4(tf32_round(v.x - h.x), tf32_round(v.y - h.y), tf32_round(v.z - h.z),
                             tf32_round(v.w - h.w));
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    ss = warp_sum(ss);
    if (lane == 0) s_part[warp] = ss;
    __syncthreads();
    if (tid == 0) {
        float tot = 0.0f;
#pragma unroll
        for (int w = 0; w < kNormThreads / 32; ++w) tot += s_part[w];
        a.ss_out[static_cast<size_t>(b) * a.ss_stride] = tot;
    }
}

// One CTA per (head, sequence). The four warps take groups of G positions
// round-robin; each group's key and value loads are all issued before its G
// dot products, then an online-softmax update. The warps' partial (max, sum,
// output) are merged with log-sum-exp rescaling in shared memory.
template <int EPL, int G>
__global__ void __launch_bounds__(kBAttnThreads) battn_kernel(const BAttnArgs a) {
    constexpr int HDMAX = 32 * EPL;
    pdl_launch_dependents();
    pdl_wait();
    const int h = blockIdx.x, b = a.row0 + blockIdx.y;
    if (a.active != nullptr && __ldcg(a.active + b) == 0) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hd = a.head_dim;
    const int kvh = h / (a.n_heads / a.n_kv_heads);
    const int n = min(max(__ldcg(a.pos + b), 0), a.seq_len - 1) + 1;
    const float* qrow = a.q + static_cast<size_t>(b) * a.d + static_cast<size_t>(h) * hd;
    const size_t head_off = static_cast<size_t>(a.seq ? __ldcg(a.seq + b) : b) * a.cache_seq +
                            static_cast<size_t>(kvh) * a.seq_len * hd;
    const float* Kh = a.k_cache + head_off;
    const float* Vh = a.v_cache + head_off;
    const float scale_div = sqrtf(static_cast<float>(hd));

    float qr[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
        const int e = lane + 32 * j;
        qr[j] = e < hd ? __ldcg(qrow + e) : 0.0f;
    }
    float m = -INFINITY, l = 0.0f, o[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) o[j] = 0.0f;

    for (int tb = warp * G; tb < n; tb += kBAttnWarps * G) {
        float kr[G][EPL], vr[G][EPL];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int t = tb + g;
#pragma unroll
            for (int j = 0; j < EPL; ++j) {
                const int e = lane + 32 * j;
                const bool ok = (t < n) && (e < hd);
                kr[g][j] = ok ? __ldcs(Kh + static_cast<size_t>(t) * hd + e) : 0.0f;
                vr[g][j] = ok ? __ldcs(Vh + static_cast<size_t>(t) * hd + e) : 0.0f;
            }
        }
        float sc[G];
        float gmax = -INFINITY;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float p = 0.0f;
#pragma unroll
            for (int j = 0; j < EPL; ++j) p = fmaf(qr[j], kr[g][j], p);
            p = warp_sum(p);
            sc[g] = (tb + g < n) ? p / scale_div : -INFINITY;
            gmax = fmaxf(gmax, sc[g]);
        }
        const float mnew = fmaxf(m, gmax);
        const float corr = (m == -INFINITY) ? 0.0f : expf(m - mnew);
        l *= corr;
#pragma unroll
        for (int j = 0; j < EPL; ++j) o[j] *= corr;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float p = (sc[g] == -INFINITY) ? 0.0f : expf(sc[g] - mnew);
            l += p;
#pragma unroll
            for (int j = 0; j < EPL; ++j) o[j] = fmaf(p, vr[g][j], o[j]);
        }
        m = mnew;
    }

    __shared__ float s_m[kBAttnWarps], s_l[kBAttnWarps];
    __shared__ float s_o[kBAttnWarps][HDMAX];
    if (lane == 0) {
        s_m[warp] = m;
        s_l[warp] = l;
    }
#pragma unroll
    for (int j = 0; j < EPL; ++j) s_o[warp][lane + 32 * j] = o[j];
    __syncthreads();
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kBAttnWarps; ++w) M = fmaxf(M, s_m[w]);
    float L = 0.0f;
#pragma unroll
    for (int w = 0; w < kBAttnWarps; ++w)
        if (s_m[w] != -INFINITY) L += s_l[w] * expf(s_m[w] - M);
    float* ohi = a.att_hi + static_cast<size_t>(b) * a.d + static_cast<size_t>(h) * hd;
    float* olo = a.att_lo + static_cast<size_t>(b) * a.d + static_cast<size_t>(h) * hd;
    for (int e = tid; e < hd; e += kBAttnThreads) {
        float acc = 0.0f;
#pragma unroll
        for (int w = 0; w < kBAttnWarps; ++w)
            if (s_m[w] != -INFINITY) acc += s_o[w][e] * expf(s_m[w] - M);
        const float v = acc / L;
        const float hi = tf32_round(v);
        ohi[e] = hi;
        olo[e] = tf32_round(v - hi);
    }
}

// Vectorised variant for head_dim % 4 == 0 and head_dim <= 4 * LPR: a row of
// the cache is read by LPR lanes with 16-byte loads (32 / LPR rows per warp
// load), G row slots per iteration, so a warp keeps 2 * G * 32/LPR rows of K
// and V in flight. Each lane group (one row slot) runs its own online softmax
// over its positions; groups merge by shuffles, warps through shared memory.
template <int LPR, int G, int MINB>
__global__ void __launch_bounds__(kBAttnThreads, MINB) battn4_kernel(const BAttnArgs a) {
    constexpr int RPW = 32 / LPR;  // rows per warp load
    constexpr int HD4MAX = LPR;    // float4 chunks of a row
    pdl_launch_dependents();
    pdl_wait();
    const int h = blockIdx.x, b = a.row0 + blockIdx.y;
    if (a.active != nullptr && __ldcg(a.active + b) == 0) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hd = a.head_dim, hd4 = hd >> 2;
    const int c4 = lane % LPR, slot = lane / LPR;
    const bool lane_on = c4 < hd4;
    const int kvh = h / (a.n_heads / a.n_kv_heads);
    const int n = min(max(__ldcg(a.pos + b), 0), a.seq_len - 1) + 1;
    const size_t head_off = static_cast<size_t>(a.seq ? __ldcg(a.seq + b) : b) * a.cache_seq +
                            static_cast<size_t>(kvh) * a.seq_len * hd;
    const float4* K4 = reinterpret_cast<const float4*>(a.k_cache + head_off);
    const float4* V4 = reinterpret_cast<const float4*>(a.v_cache + head_off);
    const float4 q = lane_on ? __ldcg(reinterpret_cast<const float4*>(
                                   a.q + static_cast<size_t>(b) * a.d + static_cast<size_t>(h) * hd) + c4)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
    const float scale_div = sqrtf(static_cast<float>(hd));

    float m = -INFINITY, l = 0.0f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    constexpr int PER_IT = G * RPW;  // positions per warp iteration
    for (int tb = warp * PER_IT; tb < n; tb += kBAttnWarps * PER_IT) {
        float4 kr[G], vr[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int t = tb + g * RPW + slot;
            const bool ok = lane_on && t < n;
            kr[g] = ok ? __ldcg(K4 + static_cast<size_t>(t) * hd4 + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
            vr[g] = ok ? __ldcg(V4 + static_cast<size_t>(t) * hd4 + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float sc[G];
        float gmax = -INFINITY;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float p = q.x * kr[g].x;
            p = fmaf(q.y, kr[g].y, p);
            p = fmaf(q.z, kr[g].z, p);
            p = fmaf(q.w, kr[g].w, p);
#pragma unroll
            for (int off = LPR / 2; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
            sc[g] = (tb + g * RPW + slot < n) ? p / scale_div : -INFINITY;
            gmax = fmaxf(gmax, sc[g]);
        }
        if (gmax == -INFINITY) continue;  // this slot has no positions left
        const float mnew = fmaxf(m, gmax);
        const float corr = (m == -INFINITY) ? 0.0f : expf(m - mnew);
        l *= corr;
        o.x *= corr;
        o.y *= corr;
        o.z *= corr;
        o.w *= corr;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float p = (sc[g] == -INFINITY) ? 0.0f : expf(sc[g] - mnew);
            l += p;
            o.x = fmaf(p, vr[g].x, o.x);
            o.y = fmaf(p, vr[g].y, o.y);
            o.z = fmaf(p, vr[g].z, o.z);
            o.w = fmaf(p, vr[g].w, o.w);
        }
        m = mnew;
    }
    // merge the row slots of this warp (lanes c4 + LPR * slot)
#pragma unroll
    for (int off = LPR; off < 32; off <<= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
        const float l2v = __shfl_xor_sync(0xffffffffu, l, off);
        float4 o2;
        o2.x = __shfl_xor_sync(0xffffffffu, o.x, off);
        o2.y = __shfl_xor_sync(0xffffffffu, o.y, off);
        o2.z = __shfl_xor_sync(0xffffffffu, o.z, off);
        o2.w = __shfl_xor_sync(0xffffffffu, o.w, off);
        const float M = fmaxf(m, m2);
        const float f1 = (m == -INFINITY) ? 0.0f : expf(m - M);
        const float f2 = (m2 == -INFINITY) ? 0.0f : expf(m2 - M);
        l = l * f1 + l2v * f2;
        o.x = o.x * f1 + o2.x * f2;
        o.y = o.y * f1 + o2.y * f2;
        o.z = o.z * f1 + o2.z * f2;
        o.w = o.w * f1 + o2.w * f2;
        m = M;
    }
    __shared__ float s_m[kBAttnWarps], s_l[kBAttnWarps];
    __shared__ float4 s_o[kBAttnWarps][HD4MAX];
    if (lane == 0) {
        s_m[warp] = m;
        s_l[warp] = l;
    }
    if (slot == 0) s_o[warp][c4] = o;
    __syncthreads();
    if (tid < hd4) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kBAttnWarps; ++w) M = fmaxf(M, s_m[w]);
        float L = 0.0f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kBAttnWarps; ++w) {
            if (s_m[w] == -INFINITY) continue;
            const float f = expf(s_m[w] - M);
            L += s_l[w] * f;
            const float4 v = s_o[w][tid];
            acc.x += v.x * f;
            acc.y += v.y * f;
            acc.z += v.z * f;
            acc.w += v.w * f;
        }
        const float4 r = make_float4(acc.x / L, acc.y / L, acc.z / L, acc.w / L);
        const float4 hi = make_float4(tf32_round(r.x), tf32_round(r.y), tf32_round(r.z), tf32_round(r.w));
        const size_t off = static_cast<size_t>(b) * a.d + static_cast<size_t>(h) * hd;
        reinterpret_cast<float4*>(a.att_hi + off)[tid] = hi;
        reinterpret_cast<float4*>(a.att_lo + off)[tid] =
            make_float4(tf32_round(r.x - hi.x), tf32_round(r.y - hi.y), tf32_round(r.z - hi.z),
                        tf32_round(r.w - hi.w));
    }
}

__global__ void badvance_kernel(const BAdvanceArgs a) {
    pdl_launch_dependents();
    pdl_wait();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= a.M) return;
    const int b = a.row0 + i;
    const unsigned long long k = a.keys[b];
    a.keys[b] = 0ull;
    const int idx = (k == 0ull) ? 0 : argmax_key_index(k);
    a.last[b] = idx;
    if (a.mode != 1 || a.active[b] == 0) return;
    const int p = a.pos[b], np = a.len[b];
    if (p >= np - 1) {
        const int k_out = p - (np - 1);
        a.out[static_cast<size_t>(b) * a.steps + k_out] = idx;
        if (k_out + 1 >= a.steps) {
            a.active[b] = 0;  // finished: its row is still computed, never used
            return;
        }
    }
    a.token[b] = (p + 1 < np) ? a.prompts[a.poff[b] + p + 1] : idx;
    a.pos[b] = p + 1;
}

template <typename Args, typename Kernel>
cudaError_t launch_pdl(Kernel k, dim3 grid, dim3 block, const Args& a, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k, a);
}

}  // namespace

cudaError_t launch_brmsnorm(const BNormArgs& a, int M, cudaStream_t s, bool pdl) {
    if (M < 1 || a.d % 4 != 0 || a.emb == nullptr || a.ss_out == nullptr || a.ss_stride < 1)
        return cudaErrorInvalidValue;
    return launch_pdl(brmsnorm_kernel, dim3(M), dim3(kNormThreads), a, s, pdl);
}

cudaError_t launch_battn(const BAttnArgs& a, int M, cudaStream_t s, bool pdl) {
    if (M < 1) return cudaErrorInvalidValue;
    const dim3 grid(a.n_heads, M), block(kBAttnThreads);
    if (a.head_dim % 4 == 0 && a.d % 4 == 0) {
        if (a.head_dim <= 64) return launch_pdl(battn4_kernel<16, 4, 8>, grid, block, a, s, pdl);
        if (a.head_dim <= 128) return launch_pdl(battn4_kernel<32, 4, 8>, grid, block, a, s, pdl);
    }
    if (a.head_dim <= 64) return launch_pdl(battn_kernel<2, 8>, grid, block, a, s, pdl);
    if (a.head_dim <= 128) return launch_pdl(battn_kernel<4, 8>, grid, block, a, s, pdl);
    if (a.head_dim <= 256) return launch_pdl(battn_kernel<8, 4>, grid, block, a, s, pdl);
    return cudaErrorInvalidValue;
}

cudaError_t launch_badvance(const BAdvanceArgs& a, cudaStream_t s, bool pdl) {
    if (a.M < 1) return cudaErrorInvalidValue;
    return launch_pdl(badvance_kernel, dim3((a.M + 127) / 128), dim3(128), a, s, pdl);
}

}  // namespace l2
