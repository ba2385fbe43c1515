// fused_small.cu -- the batch-1 forward of a small model in two kernels per
// layer instead of five.
//
// The step is the same fp32 Llama-2 decode step as matvec.cu + attention.cu
// compute (the llama2.c pages' single-file engine: per layer RMSNorm, Q/K/V,
// RoPE, KV append, causal attention, Wo + residual, RMSNorm, SwiGLU FFN +
// residual). For models whose layers are a few MB, each of those kernels is
// a few microseconds of dependency latency, not bandwidth, so this path cuts
// the number of kernel boundaries per layer from five to two:
//
//   attention block  grid (8, H), one thread-block cluster of 8 CTAs per query
//                    head h. CTA j computes rows [j*3hd/8, (j+1)*3hd/8) of the
//                    head's [q_h; k_kv; v_kv] projections (RoPE applied),
//                    hands them to every CTA of the cluster through
//                    distributed shared memory, then takes positions
//                    [n*j/8, n*(j+1)/8) of the cache in an online softmax;
//                    the 8 partials are exchanged the same way and merged in
//                    every CTA, which then multiplies rows [d*j/8, d*(j+1)/8)
//                    of Wo's head-h column block by att_h and adds the result
//                    into the residual. The first query head of each kv group
//                    also appends k and v to the cache.
//   FFN block        grid G, CTA c owns hidden units [F*c/G, F*(c+1)/G): it
//                    computes their SwiGLU values from its W1/W3 rows, then
//                    their contribution W2[:, units] * hb to all d outputs (W2
//                    stored transposed, so the columns are contiguous rows),
//                    and adds it into the residual.
//
// Both blocks add into a residual that many CTAs update, so the residual
// stream is kept in 64-bit fixed point (value * 2^32, rounded to nearest;
// magnitudes below 2^31): integer additions are exact and commutative, so
// the sum, and therefore every result, is the same whatever order the
// atomics land in. Each partial is rounded once to 2^-32 (about 2.3e-10),
// finer than fp32's own rounding for values above 2^-9. Buffers: P[2] (the
// residual between layers) and M[2] (after attention), each kernel zeroing
// the buffer the next one accumulates into (a buffer is zeroed only after
// its last reader has finished: kernel boundaries order them).
//
// Each CTA's weights (its Q/K/V rows and Wo block rows, or its W1/W3 rows
// and W2 columns) fit in shared memory and are requested with bulk copies at
// kernel start, before griddepcontrol.wait: weights never depend on the
// previous kernel, so they load while it finishes.
#include <cooperative_groups.h>
#include <math.h>

#include "l2_internal.cuh"

namespace cg = cooperative_groups;

namespace l2 {

namespace {

constexpr int kFAttnThreads = 512;  // attention block: 16 warps
constexpr int kFAttnWarps = kFAttnThreads / 32;
constexpr int kFFfnThreads = 512;   // FFN block
constexpr int kFFfnWarps = kFFfnThreads / 32;
constexpr int G8 = kFusedCluster;
static_assert(G8 <= kFAttnThreads, "one thread per partial forms its factor");

__device__ __forceinline__ long long to_fixed(float v) {
    return __float2ll_rn(v * 4294967296.0f);
}
__device__ __forceinline__ float from_fixed(long long x) {
    return __ll2float_rn(x) * (1.0f / 4294967296.0f);
}
// Adds without waiting for the old value (a reduction, not a returning
// atomic): a thread issues its adds back to back. Kernel completion makes them
// visible to the next kernel, which is the only reader.
__device__ __forceinline__ void add_fixed(long long* p, long long v) {
    asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Shared-memory carve-up of the attention block (floats; every piece 16-byte aligned).
struct FAttnLayout {
    int rows_qkv, rows_o;       // this CTA's Q/K/V rows and Wo block rows (maximum over ranks)
    int off_wq, off_wo, off_x, off_qkv, off_part, off_red, off_c, off_rs, total;
};
__host__ __device__ inline FAttnLayout fattn_layout(int d, int hd) {
    FAttnLayout L;
    L.rows_qkv = (3 * hd) / G8;
    L.rows_o = (d + G8 - 1) / G8;
    L.off_wq = 0;
    L.off_wo = L.off_wq + L.rows_qkv * d;
    L.off_x = L.off_wo + ((L.rows_o * hd + 3) & ~3);
    L.off_qkv = L.off_x + ((d + 3) & ~3);
    L.off_part = L.off_qkv + ((3 * hd + 3) & ~3);
    L.off_red = L.off_part + G8 * ((hd + 2 + 3) & ~3);
    L.off_c = L.off_red + kFAttnWarps * ((hd + 2 + 3) & ~3) + 64;  // carried rows, 8 bytes each
    L.off_rs = L.off_c + 2 * ((d / G8 + 1 + 3) & ~3);           // RoPE pairs of the rows
    L.total = L.off_rs + 2 * ((L.rows_qkv / 2 + 3) & ~3);
    return L;
}

// RMS norm of a row: loads x (float src, or fixed point srcf, the sum of
// `copies` copies d apart) and the gain g (the same round trip) into xs as
// g x, and returns inv = 1 / sqrt(mean(x^2) + eps): the normalised row is
// inv * xs, and the caller applies inv to the dot products it takes with xs. Each thread issues all its loads
// before using one (one L2 round trip for d <= 4 * threads). Rows c0..c1 of x
// are also added into `carry` and cleared in `zero` from the same loads, or,
// with `stash`, kept there in fixed point for the caller to add later.
constexpr int kRowRegs = 4;
template <int NT>
__device__ __forceinline__ float norm_load(float* xs, const float* src, const long long* srcf,
                                           int d, float eps, float* red, long long* carry,
                                           long long* zero, int c0, int c1,
                                           long long* stash = nullptr, int copies = 1,
                                           const float* gain = nullptr) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float ss = 0.0f;
    for (int base = 0; base < d; base += kRowRegs * NT) {
        long long fx[kRowRegs];
        float v[kRowRegs];
        float gk[kRowRegs];
#pragma unroll
        for (int k = 0; k < kRowRegs; ++k) {
            const int i = base + k * NT + tid;
            fx[k] = 0;
            v[k] = 0.0f;
            gk[k] = (gain != nullptr && i < d) ? __ldg(gain + i) : 1.0f;
            if (i < d) {
                if (srcf) {
                    fx[k] = __ldcg(srcf + i);
                    for (int c = 1; c < copies; ++c) fx[k] += __ldcg(srcf + static_cast<size_t>(c) * d + i);
                } else {
                    v[k] = __ldg(src + i);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < kRowRegs; ++k) {
            const int i = base + k * NT + tid;
            if (i < d) {
                if (srcf) v[k] = from_fixed(fx[k]);
                xs[i] = gk[k] * v[k];  // g x: the 1 / rms scale goes on the dot products
                ss += v[k] * v[k];
                if (i >= c0 && i < c1) {
                    const long long xf = srcf ? fx[k] : to_fixed(v[k]);
                    if (stash) {
                        stash[i - c0] = xf;
                    } else {
                        add_fixed(carry + i, xf);
                        zero[i] = 0;
                    }
                }
            }
        }
    }
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float t = lane < NT / 32 ? red[lane] : 0.0f;  // every warp forms the same total
    t = warp_sum(t);
    return 1.0f / sqrtf(t / static_cast<float>(d) + eps);
}

// Dot products of two shared-memory rows with xs by one warp (16-byte
// loads; the x loads are shared).
__device__ __forceinline__ float2 warp_dot2(const float* w0, const float* w1, const float* xs,
                                            int d, int lane) {
    const float4* a4 = reinterpret_cast<const float4*>(w0);
    const float4* b4 = reinterpret_cast<const float4*>(w1);
    const float4* x4 = reinterpret_cast<const float4*>(xs);
    float4 p = make_float4(0.f, 0.f, 0.f, 0.f), q = p;
    for (int c = lane; c < (d >> 2); c += 32) {
        const float4 x = x4[c], a = a4[c], b = b4[c];
        p.x = fmaf(a.x, x.x, p.x);
        p.y = fmaf(a.y, x.y, p.y);
        p.z = fmaf(a.z, x.z, p.z);
        p.w = fmaf(a.w, x.w, p.w);
        q.x = fmaf(b.x, x.x, q.x);
        q.y = fmaf(b.y, x.y, q.y);
        q.z = fmaf(b.z, x.z, q.z);
        q.w = fmaf(b.w, x.w, q.w);
    }
    float u = (p.x + p.y) + (p.z + p.w), v = (q.x + q.y) + (q.z + q.w);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        u += __shfl_xor_sync(0xffffffffu, u, off);
        v += __shfl_xor_sync(0xffffffffu, v, off);
    }
    return make_float2(u, v);
}

// LPR lanes read one 16-byte-vectorised cache row (head_dim <= 4 LPR).
template <int LPR>
// 80 registers: with the FFN block's 48 at the same thread count, an FFN CTA
// fits on an SM beside an attention CTA (where shared memory allows) and
// starts, copying its weights, while the attention block runs.
__global__ void __maxnreg__(80) fattn_kernel(const __grid_constant__ FAttnArgs a) {
    constexpr int RPW = 32 / LPR;  // rows per warp load
    constexpr int GR = 4;          // row slots per lane group and iteration
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float* sm = reinterpret_cast<float*>(smem_raw);
    cg::cluster_group cluster = cg::this_cluster();
    const int j = static_cast<int>(cluster.block_rank());
    const int h = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int d = a.d, hd = a.hd, kvd = a.kvd;
    const int grp = a.H / a.KVH, kvh = h / grp;
    const FAttnLayout L = fattn_layout(d, hd);
    float* wq = sm + L.off_wq;
    float* wo = sm + L.off_wo;
    float* xs = sm + L.off_x;
    float* qkv = sm + L.off_qkv;
    float* part = sm + L.off_part;
    float* red = sm + L.off_red;
    long long* cst = reinterpret_cast<long long*>(sm + L.off_c);
    float2* rs = reinterpret_cast<float2*>(sm + L.off_rs);
    const int pstride = (hd + 2 + 3) & ~3;
    __shared__ __align__(8) uint64_t wbar;
    __shared__ __align__(8) uint64_t qbar;  // q, k, v rows from the cluster's CTAs
    __shared__ __align__(8) uint64_t pbar;  // the 8 attention partials
    __shared__ float s_fac[kFAttnWarps + 1];    // the warps' softmax rescale factors, and M
    __shared__ float s_mfac[G8];            // the partials' rescale factors
    __shared__ int s_fail;

    // this CTA's slices
    const int t0 = (3 * hd) * j / G8, t1 = (3 * hd) * (j + 1) / G8;  // rows of [q; k; v]
    const int r0 = d * j / G8, r1 = d * (j + 1) / G8;                  // rows of the Wo block

    if (tid == 0) {
        s_fail = 0;
        mbar_init(&wbar, 1);
        mbar_init(&qbar, 1);
        mbar_init(&pbar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&qbar, static_cast<uint32_t>(3 * hd * 4));
        mbar_arrive_expect_tx(&pbar, static_cast<uint32_t>(G8 * (hd + 2) * 4));
    }
    __syncthreads();
    if (tid == 0) {
        const uint64_t pol = (a.l2_policy == 0) ? make_policy_evict_first()
                                                : make_policy_evict_last(__uint_as_float(
                                                      static_cast<uint32_t>(a.l2_policy)));
        const uint32_t bytes = static_cast<uint32_t>(((t1 - t0) * d + (r1 - r0) * hd) * 4);
        mbar_arrive_expect_tx(&wbar, bytes);
        // [q; k; v] rows t0..t1 as up to three runs of contiguous global rows
        int t = t0;
        while (t < t1) {
            const int part_end = t < hd ? hd : t < 2 * hd ? 2 * hd : 3 * hd;
            const int e = min(t1, part_end);
            const int g0 = t < hd ? h * hd + t : t < 2 * hd ? d + kvh * hd + (t - hd)
                                                               : d + kvd + kvh * hd + (t - 2 * hd);
            bulk_g2s(wq + static_cast<size_t>(t - t0) * d, a.wqkv + static_cast<size_t>(g0) * d,
                     static_cast<uint32_t>((e - t) * d * 4), &wbar, pol);
            t = e;
        }
        bulk_g2s(wo, a.wo_h + (static_cast<size_t>(h) * d + r0) * hd,
                 static_cast<uint32_t>((r1 - r0) * hd * 4), &wbar, pol);
    }
    pdl_launch_dependents();
    cluster_arrive_relaxed();  // this CTA runs (waited for before remote writes)

    // ---- everything below reads results of earlier kernels
    pdl_wait();
    L2State* st = a.st;
    const int pos = __ldcg(&st->pos);
    const int slot_cur = pos % a.S;
    const int n = min(pos + 1, a.S);
    const float* emb_row = nullptr;
    if (a.x_in == nullptr) {
        const int raw = __ldcg(&st->token);
        const int tok = min(max(raw, 0), a.vocab - 1);
        if (raw != tok && h == 0 && j == 0 && tid == 0) atomicOr(&st->err, ERR_BAD_INPUT);
        emb_row = a.emb + static_cast<size_t>(tok) * d;
    }
    // RoPE (cos, sin) of this CTA's q and k pairs, loaded beside x
    const int half = hd >> 1;
    const float2* rope = a.rope + static_cast<size_t>(pos) * half;
    for (int p = tid; 2 * p < t1 - t0; p += kFAttnThreads) {
        const int tg = t0 + 2 * p;
        if (tg < 2 * hd) rs[p] = __ldg(rope + ((tg < hd ? tg : tg - hd) >> 1));
    }
    // head 0's CTAs keep their rows of the residual, added into x_mid once the
    // cluster's exchanges are behind them
    const float inv = norm_load<kFAttnThreads>(xs, emb_row, a.x_in, d, a.eps, red, a.x_mid, a.x_zero,
                                h == 0 ? r0 : 0, h == 0 ? r1 : 0, cst, kFfnCopies, a.g_att);
    if (!mbar_wait_bounded(&wbar, 0u) && tid == 0) {
        atomicOr(&st->err, ERR_TIMEOUT_TMA);
        s_fail = 1;
        mbar_wait_bounded(&wbar, 0u);  // drain the copies still in flight (bounded)
    }
    __syncthreads();
    const bool ok = s_fail == 0;  // on a timeout the exchanges still run (every CTA
                                  // sends its rows and partials), with zeros

    // ---- Q/K/V rows of this CTA (pairs per warp: RoPE needs both)
    cluster_wait_all();  // every CTA of the cluster runs: remote writes allowed
    for (int p = warp; 2 * p < t1 - t0; p += kFAttnWarps) {
        const int tl = 2 * p, tg = t0 + tl;  // even: a pair never straddles q/k/v
        float v0 = 0.0f, v1 = 0.0f;
        if (ok) {
            const float2 r = warp_dot2(wq + static_cast<size_t>(tl) * d,
                                       wq + static_cast<size_t>(tl + 1) * d, xs, d, lane);
            v0 = r.x * inv;
            v1 = r.y * inv;
        }
        if (tg < 2 * hd) {  // q or k: rotate the pair
            const float2 cs = rs[p];
            const float y0 = v0 * cs.x - v1 * cs.y, y1 = v0 * cs.y + v1 * cs.x;
            v0 = y0;
            v1 = y1;
        }
        if (lane < G8)  // lane q sends the pair to rank q's copy
            st_async_f2(cluster_smem(qkv + tg, lane), v0, v1, cluster_smem(&qbar, lane));
    }
    // q, k, v of the head are in every CTA once 3 hd floats have landed here
    if (!mbar_wait_cluster_bounded(&qbar, 0u) && tid == 0) atomicOr(&st->err, ERR_TIMEOUT_TMA);

    // ---- attention over this CTA's share of the cache slots
    {
        const int hd4 = hd >> 2;
        const int c4 = lane % LPR, slot = lane / LPR;
        const bool lane_on = c4 < hd4;
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        const float4* K4 = reinterpret_cast<const float4*>(a.k_cache + static_cast<size_t>(kvh) * a.S * hd);
        const float4* V4 = reinterpret_cast<const float4*>(a.v_cache + static_cast<size_t>(kvh) * a.S * hd);
        const float4 q = lane_on ? reinterpret_cast<const float4*>(qkv)[c4] : z;
        const float4 kcur = lane_on ? reinterpret_cast<const float4*>(qkv + hd)[c4] : z;
        const float4 vcur = lane_on ? reinterpret_cast<const float4*>(qkv + 2 * hd)[c4] : z;
        const int s0 = static_cast<int>(static_cast<long long>(n) * j / G8);
        const int s1 = static_cast<int>(static_cast<long long>(n) * (j + 1) / G8);
        const float scale_div = sqrtf(static_cast<float>(hd));
        float m = -INFINITY, l = 0.0f;
        float4 o = z;
        constexpr int PER_IT = GR * RPW;
        for (int tb = s0 + warp * PER_IT; tb < s1; tb += kFAttnWarps * PER_IT) {
            float4 kr[GR], vr[GR];
#pragma unroll
            for (int g = 0; g < GR; ++g) {
                const int t = tb + g * RPW + slot;
                const bool in = lane_on && t < s1;
                if (in && t == slot_cur) {  // this position: from shared memory
                    kr[g] = kcur;
                    vr[g] = vcur;
                } else {
                    kr[g] = in ? __ldcg(K4 + static_cast<size_t>(t) * hd4 + c4) : z;
                    vr[g] = in ? __ldcg(V4 + static_cast<size_t>(t) * hd4 + c4) : z;
                }
            }
            float sc[GR];
            float gmax = -INFINITY;
#pragma unroll
            for (int g = 0; g < GR; ++g) {
                float pq = q.x * kr[g].x;
                pq = fmaf(q.y, kr[g].y, pq);
                pq = fmaf(q.z, kr[g].z, pq);
                pq = fmaf(q.w, kr[g].w, pq);
#pragma unroll
                for (int off = LPR / 2; off > 0; off >>= 1) pq += __shfl_xor_sync(0xffffffffu, pq, off);
                sc[g] = (tb + g * RPW + slot < s1) ? pq / scale_div : -INFINITY;
                gmax = fmaxf(gmax, sc[g]);
            }
            if (gmax == -INFINITY) continue;
            const float mnew = fmaxf(m, gmax);
            // __expf: the SFU exponential, within a few ulp for these
            // non-positive arguments, as close as the fp32 sums it weights
            const float corr = (m == -INFINITY) ? 0.0f : __expf(m - mnew);
            l *= corr;
            o.x *= corr;
            o.y *= corr;
            o.z *= corr;
            o.w *= corr;
#pragma unroll
            for (int g = 0; g < GR; ++g) {
                const float pe = (sc[g] == -INFINITY) ? 0.0f : __expf(sc[g] - mnew);
                l += pe;
                o.x = fmaf(pe, vr[g].x, o.x);
                o.y = fmaf(pe, vr[g].y, o.y);
                o.z = fmaf(pe, vr[g].z, o.z);
                o.w = fmaf(pe, vr[g].w, o.w);
            }
            m = mnew;
        }
#pragma unroll
        for (int off = LPR; off < 32; off <<= 1) {  // merge the row slots of the warp
            const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
            const float l2v = __shfl_xor_sync(0xffffffffu, l, off);
            float4 o2;
            o2.x = __shfl_xor_sync(0xffffffffu, o.x, off);
            o2.y = __shfl_xor_sync(0xffffffffu, o.y, off);
            o2.z = __shfl_xor_sync(0xffffffffu, o.z, off);
            o2.w = __shfl_xor_sync(0xffffffffu, o.w, off);
            const float M = fmaxf(m, m2);
            const float f1 = (m == -INFINITY) ? 0.0f : __expf(m - M);
            const float f2 = (m2 == -INFINITY) ? 0.0f : __expf(m2 - M);
            l = l * f1 + l2v * f2;
            o.x = o.x * f1 + o2.x * f2;
            o.y = o.y * f1 + o2.y * f2;
            o.z = o.z * f1 + o2.z * f2;
            o.w = o.w * f1 + o2.w * f2;
            m = M;
        }
        float* wp = red + warp * pstride;  // per-warp partial: o[hd], m, l
        if (slot == 0 && lane_on) reinterpret_cast<float4*>(wp)[c4] = o;
        if (lane == 0) {
            wp[hd] = m;
            wp[hd + 1] = l;
        }
        __syncthreads();
        // the CTA's partial, sent to every CTA of the cluster (slot j); the
        // warps' rescale factors exp(m_w - M) are formed once, by 8 threads
        if (tid < kFAttnWarps) {
            float M = -INFINITY;
            for (int w = 0; w < kFAttnWarps; ++w) M = fmaxf(M, red[w * pstride + hd]);
            const float mw = red[tid * pstride + hd];
            s_fac[tid] = (mw == -INFINITY) ? 0.0f : __expf(mw - M);
            if (tid == 0) s_fac[kFAttnWarps] = M;
        }
        __syncthreads();
        const float M = s_fac[kFAttnWarps];
        for (int e = tid; e < hd + 2; e += kFAttnThreads) {
            float acc = 0.0f;
            for (int w = 0; w < kFAttnWarps; ++w) {
                const float fw = s_fac[w];
                if (fw != 0.0f)
                    acc += (e < hd ? red[w * pstride + e] : red[w * pstride + hd + 1]) * fw;
            }
            const float val = (e == hd) ? M : acc;
            for (int q2 = 0; q2 < G8; ++q2)
                st_async_f1(cluster_smem(part + j * pstride + e, q2), val, cluster_smem(&pbar, q2));
        }
    }
    // every CTA holds the 8 partials once 8 (hd + 2) floats have landed here
    if (!mbar_wait_cluster_bounded(&pbar, 0u) && tid == 0) atomicOr(&st->err, ERR_TIMEOUT_TMA);
    cluster_arrive_relaxed();  // all remote writes into this CTA are done (waited
                               // for at the end: no CTA leaves before its peers)

    // ---- global writes that nothing in this kernel reads, issued after the
    // last exchange (a cluster barrier's release would have waited for them):
    // the carried residual rows, and this position's k and v, appended by the
    // first cluster of each kv head, 1/8 of the 2 hd values per CTA
    if (h == 0) {
        for (int r = r0 + tid; r < r1; r += kFAttnThreads) {
            add_fixed(a.x_mid + r, cst[r - r0]);
#pragma unroll
            for (int c = 0; c < kFfnCopies; ++c) a.x_zero[static_cast<size_t>(c) * d + r] = 0;
        }
    }
    if ((h % grp) == 0) {
        float* kc = a.k_cache + (static_cast<size_t>(kvh) * a.S + slot_cur) * hd;
        float* vc = a.v_cache + (static_cast<size_t>(kvh) * a.S + slot_cur) * hd;
        const int e0 = 2 * hd * j / G8, e1 = 2 * hd * (j + 1) / G8;
        for (int e = e0 + tid; e < e1; e += kFAttnThreads) {
            if (e < hd) kc[e] = qkv[hd + e];
            else vc[e - hd] = qkv[hd + e];
        }
    }

    // ---- merge the partials into att_h (in xs: x is no longer needed)
    float* att = xs;
    {
        // the partials' rescale factors exp(m_q - max m), formed once
        if (tid < G8) {
            float Mg = -INFINITY;
            for (int q2 = 0; q2 < G8; ++q2) Mg = fmaxf(Mg, part[q2 * pstride + hd]);
            const float mq = part[tid * pstride + hd];
            s_mfac[tid] = (mq == -INFINITY) ? 0.0f : expf(mq - Mg);
        }
        __syncthreads();
        float Lg = 0.0f;
        for (int q2 = 0; q2 < G8; ++q2)
            if (s_mfac[q2] != 0.0f) Lg += part[q2 * pstride + hd + 1] * s_mfac[q2];
        for (int e = tid; e < hd; e += kFAttnThreads) {
            float acc = 0.0f;
            for (int q2 = 0; q2 < G8; ++q2)
                if (s_mfac[q2] != 0.0f) acc += part[q2 * pstride + e] * s_mfac[q2];
            att[e] = acc / Lg;
        }
    }
    __syncthreads();

    // ---- rows r0..r1 of Wo's head-h block times att_h, into x_mid: 8 lanes
    // per row (16-byte steps), 4 rows per warp at once
    {
        const int sub = lane >> 3, l8 = lane & 7, hd4 = hd >> 2;
        const float4* a4 = reinterpret_cast<const float4*>(att);
        for (int rb = r0 + 4 * warp; rb < r1; rb += 4 * kFAttnWarps) {
            const int r = rb + sub;
            float acc = 0.0f;
            if (r < r1) {
                const float4* w4 = reinterpret_cast<const float4*>(wo + static_cast<size_t>(r - r0) * hd);
                float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int c = l8; c < hd4; c += 8) {
                    const float4 w = w4[c], x = a4[c];
                    t.x = fmaf(w.x, x.x, t.x);
                    t.y = fmaf(w.y, x.y, t.y);
                    t.z = fmaf(w.z, x.z, t.z);
                    t.w = fmaf(w.w, x.w, t.w);
                }
                acc = (t.x + t.y) + (t.z + t.w);
            }
            acc += __shfl_xor_sync(0xffffffffu, acc, 4);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            if (l8 == 0 && r < r1 && ok) add_fixed(a.x_mid + r, to_fixed(acc));
        }
    }
    cluster_wait_all();
}

// Shared-memory carve-up of the FFN block for at most `units` hidden units.
struct FFfnLayout {
    int off_w13, off_w2, off_x, off_hb, off_red, total;
};
__host__ __device__ inline FFfnLayout fffn_layout(int d, int units) {
    FFfnLayout L;
    L.off_w13 = 0;
    L.off_w2 = L.off_w13 + 2 * units * d;
    L.off_x = L.off_w2 + units * d;
    L.off_hb = L.off_x + ((d + 3) & ~3);
    L.off_red = L.off_hb + ((units + 3) & ~3);
    L.total = L.off_red + 64;
    return L;
}

__global__ void __launch_bounds__(kFFfnThreads) fffn_kernel(const __grid_constant__ FFfnArgs f) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float* sm = reinterpret_cast<float*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int d = f.d, G = gridDim.x, c = blockIdx.x;
    const int u0 = static_cast<int>(static_cast<long long>(f.F) * c / G);
    const int u1 = static_cast<int>(static_cast<long long>(f.F) * (c + 1) / G);
    const int nu = u1 - u0;
    const int umax = (f.F + G - 1) / G;
    const FFfnLayout L = fffn_layout(d, umax);
    float* w13 = sm + L.off_w13;
    float* w2t = sm + L.off_w2;
    float* xs = sm + L.off_x;
    float* hb = sm + L.off_hb;
    float* red = sm + L.off_red;
    __shared__ __align__(8) uint64_t wbar;
    __shared__ int s_fail;

    if (tid == 0) {
        s_fail = 0;
        mbar_init(&wbar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) mbar_arrive_expect_tx(&wbar, static_cast<uint32_t>(3 * nu * d * 4));
    if (tid == 0 && nu > 0) {
        const uint64_t pol = (f.l2_policy == 0) ? make_policy_evict_first()
                                                : make_policy_evict_last(__uint_as_float(
                                                      static_cast<uint32_t>(f.l2_policy)));
        bulk_g2s(w13, f.w13 + static_cast<size_t>(2 * u0) * d, static_cast<uint32_t>(2 * nu * d * 4),
                 &wbar, pol);
        bulk_g2s(w2t, f.w2t + static_cast<size_t>(u0) * d, static_cast<uint32_t>(nu * d * 4), &wbar,
                 pol);
    }
    pdl_launch_dependents();

    pdl_wait();
    // carry the residual into x_out and clear the next attention output,
    // rows split over the CTAs
    const int q0 = static_cast<int>(static_cast<long long>(d) * c / G);
    const int q1 = static_cast<int>(static_cast<long long>(d) * (c + 1) / G);
    long long* x_out = f.x_out + static_cast<size_t>(c % kFfnCopies) * d;  // this CTA's copy
    const float inv = norm_load<kFFfnThreads>(xs, nullptr, f.x_mid, d, f.eps, red, x_out, f.x_zero,
                                              q0, q1, nullptr, 1, f.g_ffn);
    if (!mbar_wait_bounded(&wbar, 0u) && tid == 0) {
        atomicOr(f.err, ERR_TIMEOUT_TMA);
        s_fail = 1;
        mbar_wait_bounded(&wbar, 0u);  // drain the copies still in flight (bounded)
    }
    __syncthreads();
    if (s_fail || nu == 0) return;

    // SwiGLU of the CTA's hidden units (interleaved rows: 2u gate, 2u + 1 up)
    for (int u = warp; u < nu; u += kFFfnWarps) {
        const float2 gu = warp_dot2(w13 + static_cast<size_t>(2 * u) * d,
                                    w13 + static_cast<size_t>(2 * u + 1) * d, xs, d, lane);
        const float gt = gu.x * inv, up = gu.y * inv;
        if (lane == 0) hb[u] = (gt / (1.0f + expf(-gt))) * up;
    }
    __syncthreads();
    // their contribution to every output: y[i] = sum_u W2[i][u0 + u] hb[u]
    for (int i = tid; i < d; i += kFFfnThreads) {
        float acc = 0.0f;
        for (int u = 0; u < nu; ++u) acc = fmaf(w2t[static_cast<size_t>(u) * d + i], hb[u], acc);
        add_fixed(x_out + i, to_fixed(acc));
    }
}

template <typename Kernel>
cudaError_t set_smem(Kernel k, int bytes) {
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

}  // namespace

bool plan_fused(FAttnArgs& a, FFfnArgs& f, int num_sms, size_t smem_optin, int* ffn_grid) {
    const int d = a.d, hd = a.hd;
    if (hd % 4 != 0 || hd > 128 || d % 4 != 0) return false;
    if ((3 * hd) % (2 * G8) != 0) return false;  // even row slices (RoPE pairs)
    const size_t budget = smem_optin - 1024;     // static shared memory
    const int attn_bytes = fattn_layout(d, hd).total * 4;
    if (static_cast<size_t>(attn_bytes) > budget) return false;
    const int G = num_sms < f.F ? num_sms : f.F;
    const int ffn_bytes = fffn_layout(d, (f.F + G - 1) / G).total * 4;
    if (static_cast<size_t>(ffn_bytes) > budget) return false;
    a.smem_bytes = attn_bytes;  // written only when the plan fits
    f.smem_bytes = ffn_bytes;
    *ffn_grid = G;
    return true;
}

cudaError_t prepare_fused(const FAttnArgs& a, const FFfnArgs& f) {
    cudaError_t e;
    if ((e = set_smem(fattn_kernel<16>, a.smem_bytes)) != cudaSuccess) return e;
    if ((e = set_smem(fattn_kernel<32>, a.smem_bytes)) != cudaSuccess) return e;
    return set_smem(fffn_kernel, f.smem_bytes);
}

cudaError_t launch_fattn(const FAttnArgs& a, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(G8, a.H);
    cfg.blockDim = dim3(kFAttnThreads);
    cfg.dynamicSmemBytes = a.smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = G8;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    if (a.hd <= 64) return cudaLaunchKernelEx(&cfg, fattn_kernel<16>, a);
    return cudaLaunchKernelEx(&cfg, fattn_kernel<32>, a);
}

cudaError_t launch_fffn(const FFfnArgs& f, int grid, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kFFfnThreads);
    cfg.dynamicSmemBytes = f.smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, fffn_kernel, f);
}

}  // namespace l2
