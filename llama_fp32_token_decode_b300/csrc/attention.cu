// attention.cu -- causal multi-head attention of one decode step over the KV
// cache, split over positions (flash-decoding) inside one thread-block cluster
// per head.
//
// For head h (kv head h / (n_heads / n_kv_heads)) the step computes
//   s_t = (q_h . k_t) / sqrt(head_dim),  t = 0..pos,
//   att_h = sum_t softmax(s)_t v_t.
// The llama2.c pages run this inside the single-file fp32 engine; the KV cache
// that bounds it is named in the to-do list of
// "llama2.c｜Baby LLaMA-openAI维基百科" ("未排序的待办事项"), and Flash Attention
// is suggested as a next step in the QbitAI article on Baby LLaMA 2.
//
// Grid (nsplit, n_heads), cluster (nsplit, 1, 1): the nsplit CTAs of a cluster
// share head h and take positions [r*n/nsplit, (r+1)*n/nsplit), n = pos + 1,
// so every position count keeps all CTAs busy. The cache is head-major
// [kv_head][S][head_dim]: a CTA's keys and values are contiguous rows. Each
// warp walks groups of 8 positions, issuing all key and value loads of a group
// before the 8 dot products (shuffle reductions) and an online-softmax update.
// The CTA merges its warps, then stores (max, sum, unnormalised output) into
// the shared memory of the cluster's rank-0 CTA (distributed shared memory);
// after one hardware cluster barrier rank 0 merges the nsplit partials with
// log-sum-exp rescaling and writes att_h (attn_kernel). attn4_kernel sends
// its partials with st.async instead, their bytes counted on an mbarrier in
// rank 0, whose bounded wait replaces the barrier: the other ranks leave as
// soon as they have sent. No global atomics or fences.
#include <cooperative_groups.h>
#include <math.h>

#include "l2_internal.cuh"

namespace cg = cooperative_groups;

namespace l2 {

namespace {

constexpr int kAttnThreads = 256;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kMaxCluster = 16;

// EPL: head elements per lane (head_dim <= 32 * EPL); G: positions per warp
// iteration (all their key/value loads are in flight together).
template <int EPL, int G>
__global__ void __launch_bounds__(kAttnThreads) attn_kernel(const AttnArgs a) {
    constexpr int kGroup = G;
    constexpr int HDMAX = 32 * EPL;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int nsplit = a.nsplit;
    const int h = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hd = a.head_dim;
    const int kvh = h / (a.n_heads / a.n_kv_heads);

    __shared__ float s_inbox[kMaxCluster][HDMAX + 2];  // rank 0: partials of the cluster
    __shared__ float s_m[kAttnWarps], s_l[kAttnWarps];
    __shared__ float s_o[kAttnWarps][HDMAX];

    pdl_launch_dependents();
    pdl_wait();
    cluster_arrive_relaxed();  // this CTA is running (waited for before the remote writes)

    float qr[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
        const int e = lane + 32 * j;
        qr[j] = e < hd ? __ldcg(a.q + static_cast<size_t>(h) * hd + e) : 0.0f;
    }
    // slots 0..pos, or every slot once the cache rolls (attention does not
    // depend on the order of the positions it sums over)
    const int n = min(__ldcg(&a.st->pos) + 1, a.seq_len);
    const int t0 = static_cast<int>(static_cast<long long>(n) * rank / nsplit);
    const int t1 = static_cast<int>(static_cast<long long>(n) * (rank + 1) / nsplit);
    const float* Kh = a.k_cache + static_cast<size_t>(kvh) * a.seq_len * hd;
    const float* Vh = a.v_cache + static_cast<size_t>(kvh) * a.seq_len * hd;
    const float scale_div = sqrtf(static_cast<float>(hd));

    float m = -INFINITY, l = 0.0f, o[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) o[j] = 0.0f;

    for (int tb = t0 + warp * kGroup; tb < t1; tb += kAttnWarps * kGroup) {
        float kr[kGroup][EPL], vr[kGroup][EPL];
#pragma unroll
        for (int g = 0; g < kGroup; ++g) {
            const int t = tb + g;
#pragma unroll
            for (int j = 0; j < EPL; ++j) {
                const int e = lane + 32 * j;
                const bool ok = (t < t1) && (e < hd);
                kr[g][j] = ok ? __ldcg(Kh + static_cast<size_t>(t) * hd + e) : 0.0f;
                vr[g][j] = ok ? __ldcg(Vh + static_cast<size_t>(t) * hd + e) : 0.0f;
            }
        }
        float sc[kGroup];
        float gmax = -INFINITY;
#pragma unroll
        for (int g = 0; g < kGroup; ++g) {
            float p = 0.0f;
#pragma unroll
            for (int j = 0; j < EPL; ++j) p = fmaf(qr[j], kr[g][j], p);
            p = warp_sum(p);
            sc[g] = (tb + g < t1) ? p / scale_div : -INFINITY;
            gmax = fmaxf(gmax, sc[g]);
        }
        const float mnew = fmaxf(m, gmax);
        const float corr = (m == -INFINITY) ? 0.0f : expf(m - mnew);
        l *= corr;
#pragma unroll
        for (int j = 0; j < EPL; ++j) o[j] *= corr;
#pragma unroll
        for (int g = 0; g < kGroup; ++g) {
            const float p = (sc[g] == -INFINITY) ? 0.0f : expf(sc[g] - mnew);
            l += p;
#pragma unroll
            for (int j = 0; j < EPL; ++j) o[j] = fmaf(p, vr[g][j], o[j]);
        }
        m = mnew;
    }

    // merge the warps of this CTA
    if (lane == 0) {
        s_m[warp] = m;
        s_l[warp] = l;
    }
#pragma unroll
    for (int j = 0; j < EPL; ++j) s_o[warp][lane + 32 * j] = o[j];
    __syncthreads();
    float M = -INFINITY;
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, s_m[w]);
    cluster_wait_all();  // every CTA of the cluster is running: rank 0's inbox exists
    float* inbox = cluster.map_shared_rank(&s_inbox[rank][0], 0);
    for (int e = tid; e < hd; e += kAttnThreads) {
        float acc = 0.0f;
        for (int w = 0; w < kAttnWarps; ++w)
            if (s_m[w] != -INFINITY) acc += s_o[w][e] * expf(s_m[w] - M);
        inbox[e] = acc;
    }
    if (tid == 0) {
        float L = 0.0f;
        for (int w = 0; w < kAttnWarps; ++w)
            if (s_m[w] != -INFINITY) L += s_l[w] * expf(s_m[w] - M);
        inbox[HDMAX] = M;
        inbox[HDMAX + 1] = L;
    }
    cluster.sync();  // partials of every rank are in rank 0's shared memory
    if (rank != 0) return;

    float Mg = -INFINITY;
    for (int r = 0; r < nsplit; ++r) Mg = fmaxf(Mg, s_inbox[r][HDMAX]);
    float Lg = 0.0f;
    for (int r = 0; r < nsplit; ++r)
        if (s_inbox[r][HDMAX] != -INFINITY) Lg += s_inbox[r][HDMAX + 1] * expf(s_inbox[r][HDMAX] - Mg);
    for (int e = tid; e < hd; e += kAttnThreads) {
        float acc = 0.0f;
        for (int r = 0; r < nsplit; ++r)
            if (s_inbox[r][HDMAX] != -INFINITY) acc += s_inbox[r][e] * expf(s_inbox[r][HDMAX] - Mg);
        a.att[static_cast<size_t>(h) * hd + e] = acc / Lg;
    }
}

// Vectorised variant (head_dim % 4 == 0, head_dim <= 4 * LPR): LPR lanes read
// one cache row with 16-byte loads (32 / LPR rows per warp load), G row slots
// per warp iteration, at most 64 registers, so one CTA fits on an SM beside a
// streaming-matvec CTA and programmatic dependent launch can overlap the two.
// The rows of earlier positions are final before this kernel's predecessor
// (the QKV matvec) ends, so the first iteration's loads are issued before
// griddepcontrol.wait; the position read at that point is only a hint: the
// split over the cluster is recomputed after the wait, and rows that the
// hint did not cover are loaded then. No early loads once the cache can roll
// (a slot may then be rewritten by the QKV matvec).
template <int LPR, int G>
__global__ void __launch_bounds__(kAttnThreads, 4) attn4_kernel(const AttnArgs a) {
    constexpr int RPW = 32 / LPR;
    constexpr int HD4MAX = LPR;
    constexpr int PER_IT = G * RPW;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int nsplit = a.nsplit;
    const int h = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hd = a.head_dim, hd4 = hd >> 2;
    const int c4 = lane % LPR, slot = lane / LPR;
    const bool lane_on = c4 < hd4;
    const int kvh = h / (a.n_heads / a.n_kv_heads);
    const float4* K4 = reinterpret_cast<const float4*>(a.k_cache + static_cast<size_t>(kvh) * a.seq_len * hd);
    const float4* V4 = reinterpret_cast<const float4*>(a.v_cache + static_cast<size_t>(kvh) * a.seq_len * hd);

    __shared__ float4 s_inbox[kMaxCluster][HD4MAX];    // rank 0: partial outputs of the cluster
    __shared__ __align__(8) float s_ml[kMaxCluster][2];  // rank 0: (max, sum) of the cluster
    __shared__ float s_m[kAttnWarps], s_l[kAttnWarps];
    __shared__ float4 s_o[kAttnWarps][HD4MAX];
    __shared__ __align__(8) uint64_t s_inbar;  // rank 0: the cluster's partials have landed

    // rank 0 counts the partials' bytes (st.async from every rank, itself
    // included) on an mbarrier instead of a cluster-wide barrier, so the other
    // ranks leave as soon as they have sent theirs
    if (rank == 0 && tid == 0) {
        mbar_init(&s_inbar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&s_inbar, static_cast<uint32_t>(nsplit * (hd4 * 16 + 8)));
    }
    pdl_launch_dependents();

    // ---- early loads: the first iteration's rows of earlier positions
    auto split_range = [&](int n, int& t0, int& t1) {
        t0 = static_cast<int>(static_cast<long long>(n) * rank / nsplit);
        t1 = static_cast<int>(static_cast<long long>(n) * (rank + 1) / nsplit);
    };
    const int pos_hint = __ldcg(&a.st->pos);
    const bool early = pos_hint >= 0 && pos_hint + 1 < a.seq_len;  // no slot reuse possible
    int h0 = 0, h1 = 0;
    if (early) split_range(pos_hint + 1, h0, h1);
    float4 kr[G], vr[G];
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const int t = h0 + warp * PER_IT + g * RPW + slot;
        const bool ok = early && lane_on && t < h1 && t < pos_hint;  // final rows only
        kr[g] = ok ? __ldcg(K4 + static_cast<size_t>(t) * hd4 + c4) : z;
        vr[g] = ok ? __ldcg(V4 + static_cast<size_t>(t) * hd4 + c4) : z;
    }

    pdl_wait();  // q and the current position's row come from the QKV matvec
    cluster_arrive_relaxed();  // this CTA is running (waited for before the remote writes)

    const int n = min(__ldcg(&a.st->pos) + 1, a.seq_len);
    int t0, t1;
    split_range(n, t0, t1);
    const bool reuse = early && t0 == h0;  // early rows sit where this split wants them
    const float4 q = lane_on ? __ldcg(reinterpret_cast<const float4*>(a.q + static_cast<size_t>(h) * hd) + c4) : z;
    const float scale_div = sqrtf(static_cast<float>(hd));

    float m = -INFINITY, l = 0.0f;
    float4 o = z;
    bool first = true;
    for (int tb = t0 + warp * PER_IT; tb < t1; tb += kAttnWarps * PER_IT) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int t = tb + g * RPW + slot;
            const bool have = first && reuse && t < h1 && t < pos_hint;
            if (!have) {
                const bool ok = lane_on && t < t1;
                kr[g] = ok ? __ldcg(K4 + static_cast<size_t>(t) * hd4 + c4) : z;
                vr[g] = ok ? __ldcg(V4 + static_cast<size_t>(t) * hd4 + c4) : z;
            }
        }
        first = false;
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
            sc[g] = (tb + g * RPW + slot < t1) ? p / scale_div : -INFINITY;
            gmax = fmaxf(gmax, sc[g]);
        }
        if (gmax == -INFINITY) continue;
        const float mnew = fmaxf(m, gmax);
        // __expf: the SFU exponential, within a few ulp for these non-positive
        // arguments, as close as the fp32 sums it weights
        const float corr = (m == -INFINITY) ? 0.0f : __expf(m - mnew);
        l *= corr;
        o.x *= corr;
        o.y *= corr;
        o.z *= corr;
        o.w *= corr;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float p = (sc[g] == -INFINITY) ? 0.0f : __expf(sc[g] - mnew);
            l += p;
            o.x = fmaf(p, vr[g].x, o.x);
            o.y = fmaf(p, vr[g].y, o.y);
            o.z = fmaf(p, vr[g].z, o.z);
            o.w = fmaf(p, vr[g].w, o.w);
        }
        m = mnew;
    }
    // merge the row slots of this warp
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
        const float f1 = (m == -INFINITY) ? 0.0f : __expf(m - M);
        const float f2 = (m2 == -INFINITY) ? 0.0f : __expf(m2 - M);
        l = l * f1 + l2v * f2;
        o.x = o.x * f1 + o2.x * f2;
        o.y = o.y * f1 + o2.y * f2;
        o.z = o.z * f1 + o2.z * f2;
        o.w = o.w * f1 + o2.w * f2;
        m = M;
    }
    if (lane == 0) {
        s_m[warp] = m;
        s_l[warp] = l;
    }
    if (slot == 0) s_o[warp][c4] = o;
    __syncthreads();
    // merge the warps of this CTA into rank 0's inbox (distributed shared memory)
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, s_m[w]);
    cluster_wait_all();  // every CTA of the cluster is running: rank 0's inbox exists
    const uint32_t inbar0 = cluster_smem(&s_inbar, 0);
    if (tid < hd4) {
        float4 acc = z;
#pragma unroll
        for (int w = 0; w < kAttnWarps; ++w) {
            if (s_m[w] == -INFINITY) continue;
            const float f = __expf(s_m[w] - M);
            const float4 v = s_o[w][tid];
            acc.x += v.x * f;
            acc.y += v.y * f;
            acc.z += v.z * f;
            acc.w += v.w * f;
        }
        st_async_f4(cluster_smem(&s_inbox[rank][tid], 0), acc, inbar0);
    }
    if (tid == 0) {
        float L = 0.0f;
        for (int w = 0; w < kAttnWarps; ++w)
            if (s_m[w] != -INFINITY) L += s_l[w] * __expf(s_m[w] - M);
        st_async_f2(cluster_smem(&s_ml[rank][0], 0), M, L, inbar0);
    }
    if (rank != 0) return;  // nothing of this CTA's shared memory is read remotely
    // partials of every rank are in rank 0's shared memory once their bytes land
    if (!mbar_wait_cluster_bounded(&s_inbar, 0u)) {
        if (tid == 0) atomicOr(&a.st->err, ERR_TIMEOUT_TMA);
        return;
    }
    float Mg = -INFINITY;
    for (int r = 0; r < nsplit; ++r) Mg = fmaxf(Mg, s_ml[r][0]);
    float Lg = 0.0f;
    for (int r = 0; r < nsplit; ++r)
        if (s_ml[r][0] != -INFINITY) Lg += s_ml[r][1] * __expf(s_ml[r][0] - Mg);
    if (tid < hd4) {
        float4 acc = z;
        for (int r = 0; r < nsplit; ++r) {
            if (s_ml[r][0] == -INFINITY) continue;
            const float f = __expf(s_ml[r][0] - Mg);
            const float4 v = s_inbox[r][tid];
            acc.x += v.x * f;
            acc.y += v.y * f;
            acc.z += v.z * f;
            acc.w += v.w * f;
        }
        reinterpret_cast<float4*>(a.att + static_cast<size_t>(h) * hd)[tid] =
            make_float4(acc.x / Lg, acc.y / Lg, acc.z / Lg, acc.w / Lg);
    }
}

template <typename Kernel>
cudaError_t launch_cluster(Kernel k, const AttnArgs& a, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(a.nsplit, a.n_heads);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = a.nsplit;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, k, a);
}

template <int EPL, int G>
cudaError_t launch_attn_t(const AttnArgs& a, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(a.nsplit, a.n_heads);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = a.nsplit;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, attn_kernel<EPL, G>, a);
}

template <int EPL, int G>
cudaError_t allow_large_clusters() {
    return cudaFuncSetAttribute(attn_kernel<EPL, G>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                                1);
}

template <int EPL, int G>
int max_active_clusters(int nsplit, int n_heads) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(nsplit, n_heads);
    cfg.blockDim = dim3(kAttnThreads);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = nsplit;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, attn_kernel<EPL, G>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace

int attn_nsplit(int n_heads, int seq_len, int num_sms) {
    // 16 CTAs per head (a non-portable cluster size) when 8 would leave SMs idle
    int ns = (n_heads * 8 < num_sms) ? 16 : 8;
    while (ns > 1 && ns > seq_len) ns >>= 1;
    return ns;
}

cudaError_t prepare_attention() {
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(attn4_kernel<16, 4>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                                  1)) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(attn4_kernel<32, 4>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                                  1)) != cudaSuccess)
        return e;
    if ((e = allow_large_clusters<2, 8>()) != cudaSuccess) return e;
    if ((e = allow_large_clusters<4, 8>()) != cudaSuccess) return e;
    return allow_large_clusters<8, 4>();
}

// Largest usable cluster size <= want for this head_dim (0 if none launches).
int attn_cluster_ok(int head_dim, int nsplit, int n_heads) {
    if (head_dim <= 64) return max_active_clusters<2, 8>(nsplit, n_heads);
    if (head_dim <= 128) return max_active_clusters<4, 8>(nsplit, n_heads);
    return max_active_clusters<8, 4>(nsplit, n_heads);
}

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t s, bool pdl) {
    if (a.nsplit < 1 || a.nsplit > kMaxCluster) return cudaErrorInvalidValue;
    if (a.head_dim % 4 == 0) {
        if (a.head_dim <= 64) return launch_cluster(attn4_kernel<16, 4>, a, s, pdl);
        if (a.head_dim <= 128) return launch_cluster(attn4_kernel<32, 4>, a, s, pdl);
    }
    if (a.head_dim <= 64) return launch_attn_t<2, 8>(a, s, pdl);
    if (a.head_dim <= 128) return launch_attn_t<4, 8>(a, s, pdl);
    if (a.head_dim <= 256) return launch_attn_t<8, 4>(a, s, pdl);
    return cudaErrorInvalidValue;
}

}  // namespace l2
