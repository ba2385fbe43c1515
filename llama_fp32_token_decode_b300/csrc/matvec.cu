// matvec.cu -- fused streaming matrix-vector kernels of the fp32 decode step.
//
// Each projection of the Llama-2 decode step (llama2.c pages: the fp32 engine
// of the 新智元 article and of "llama2.c｜Baby LLaMA-openAI维基百科") is
// y = W x with W row-major [R][K], one multiply-add per 4-byte weight: the
// step is bound by HBM bandwidth, not arithmetic. The kernel below is built
// for that:
//   * one CTA per SM (grid = SM count), rows split evenly over CTAs in
//     `unit`-row groups (2 when the epilogue needs row pairs);
//   * the CTA's rows are one contiguous byte range of W; thread 0 streams it
//     into a shared-memory ring with 1-D bulk async copies (cp.async.bulk,
//     completion on mbarriers), ~190 KB in flight per SM, with an L2 eviction
//     hint so the weight stream does not push the KV cache out of L2;
//   * the first ring slots are requested BEFORE griddepcontrol.wait: with
//     programmatic dependent launch the weight prefetch of kernel n+1 overlaps
//     the tail of kernel n (weights never depend on the previous kernel);
//   * the prologue builds the (optionally RMS-normalised) input vector in
//     shared memory; warps read 16-byte weight and input vectors from shared
//     memory, reduce with shuffles, and keep every row result of the CTA in
//     shared memory for the epilogue:
//       EPI_QKV_ROPE    q/k rows rotated by RoPE, k and v appended to the cache
//       EPI_RESIDUAL    x += y                (Wo and W2)
//       EPI_SWIGLU      hb = silu(W1 x) * (W3 x) from interleaved W1/W3 rows
//       EPI_CLASSIFIER  logits, packed (value, index) atomicMax, and the last
//                       CTA advances the device-resident decode state.
#include <algorithm>

#include "l2_internal.cuh"

namespace l2 {

namespace {

constexpr int kConsumerWarps = 16;
constexpr int kWarps = kConsumerWarps + 1;    // + one producer warp
constexpr int kThreads = kWarps * 32;         // 544
constexpr int kStageMaxFloats = 12288;        // 48 KB ring slot
constexpr size_t kSmemBudget = 200 * 1024;    // one CTA per SM
constexpr int kMaxStages = 8;
constexpr int kVec = 6;                       // 16-byte input vectors held per lane

inline int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }
inline int round_up(int a, int b) { return (a + b - 1) / b * b; }

}  // namespace

MatvecPlan plan_matvec(int R, int K, int unit, int num_sms) {
    MatvecPlan p{};
    p.R = R;
    p.K = K;
    p.unit = unit;
    if (K <= kStageMaxFloats) {
        int tr = kStageMaxFloats / K;
        if (tr >= kConsumerWarps)
            tr = tr / kConsumerWarps * kConsumerWarps;
        else
            tr = tr >= 8 ? 8 : tr >= 4 ? 4 : tr >= 2 ? 2 : 1;
        p.rows_per_stage = tr;
        p.chunks_per_row = 1;
        p.chunk_floats = K;
        p.stage_floats = round_up(tr * K, 32);
    } else {
        const int nch = ceil_div(K, kStageMaxFloats);
        const int ch = round_up(ceil_div(K, nch), 4);
        p.rows_per_stage = 1;
        p.chunks_per_row = nch;
        p.chunk_floats = ch;
        p.stage_floats = round_up(ch, 32);
    }
    p.warps_per_row = kConsumerWarps / std::min(p.rows_per_stage, kConsumerWarps);
    p.rows_per_warp = std::max(1, p.rows_per_stage / kConsumerWarps);
    const int units = R / unit;
    p.grid = std::max(1, std::min(num_sms, units));
    p.max_rows_per_cta = ceil_div(units, p.grid) * unit;
    const size_t xs_bytes = static_cast<size_t>(round_up(K, 32)) * 4;
    const size_t misc =
        static_cast<size_t>(round_up(p.max_rows_per_cta * p.warps_per_row, 32)) * 4  // partials
        + 64 * 4                                                                     // scratch
        + 2 * kMaxStages * 8;                                                        // mbarriers
    const size_t stage_bytes = static_cast<size_t>(p.stage_floats) * 4;
    long long n = (static_cast<long long>(kSmemBudget) - static_cast<long long>(xs_bytes + misc)) /
                  static_cast<long long>(stage_bytes);
    n = std::max(2LL, std::min<long long>(kMaxStages, n));
    p.nstages = static_cast<int>(n);
    p.smem_bytes = p.nstages * stage_bytes + xs_bytes + misc;
    return p;
}

int matvec_threads() { return kThreads; }

namespace {

// One CTA: 16 consumer warps and 1 producer warp. Consumer warp w owns the
// columns  (w % WPR) * 32 + lane + 32 * WPR * j  (j < 4) of every row it
// touches, so its slice of the input vector lives in registers; rows of a
// ring slot are spread over the 16 / WPR warp groups. Each warp leaves one
// partial sum per (row, column part) in shared memory; the epilogue adds the
// WPR partials of a row in a fixed order.
// 88 registers: 544 threads x 88 leave a 256-thread, 64-register attention
// CTA room on the same SM (programmatic dependent launch overlaps the two).
template <int EPI>
__global__ void __maxnreg__(88) matvec_kernel(const MatvecArgs a) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const MatvecPlan& P = a.plan;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int K = P.K, K4 = K >> 2;
    const int NS = P.nstages, TR = P.rows_per_stage, NCH = P.chunks_per_row;
    const int WPR = P.warps_per_row, RPW = P.rows_per_warp;

    float* ring = reinterpret_cast<float*>(smem_raw);
    float* xs = ring + static_cast<size_t>(NS) * P.stage_floats;
    float* part = xs + ((K + 31) & ~31);
    float* scratch = part + ((P.max_rows_per_cta * WPR + 31) & ~31);  // [64]
    uint64_t* full = reinterpret_cast<uint64_t*>(scratch + 64);
    uint64_t* empty = full + kMaxStages;
    __shared__ int s_flag;

    // rows of this CTA
    const long long units = P.R / P.unit;
    const int u0 = static_cast<int>(units * blockIdx.x / gridDim.x);
    const int u1 = static_cast<int>(units * (blockIdx.x + 1) / gridDim.x);
    const int r0 = u0 * P.unit;
    const int nrows = (u1 - u0) * P.unit;
    const int total = NCH > 1 ? nrows * NCH : (nrows + TR - 1) / TR;
    const bool producer = (warp == kConsumerWarps);

    if (tid == 0) {
        for (int b = 0; b < NS; ++b) {
            mbar_init(&full[b], 1);
            mbar_init(&empty[b], kConsumerWarps);
        }
        fence_mbar_init();
        s_flag = 0;
    }
    __syncthreads();
    pdl_launch_dependents();

    uint64_t policy = 0;
    auto issue = [&](int s) {
        const int b = s % NS;
        const float* src;
        uint32_t bytes;
        if (NCH > 1) {
            const int row = s / NCH, c = s % NCH;
            const int c0 = c * P.chunk_floats;
            const int len = min(P.chunk_floats, K - c0);
            src = a.W + static_cast<size_t>(r0 + row) * K + c0;
            bytes = static_cast<uint32_t>(len) * 4u;
        } else {
            const int lr0 = s * TR;
            const int nr = min(TR, nrows - lr0);
            src = a.W + static_cast<size_t>(r0 + lr0) * K;
            bytes = static_cast<uint32_t>(nr) * static_cast<uint32_t>(K) * 4u;
        }
        mbar_arrive_expect_tx(&full[b], bytes);
        bulk_g2s(ring + static_cast<size_t>(b) * P.stage_floats, src, bytes, &full[b], policy);
    };

    // weights never depend on earlier kernels: request the first slots now
    int issued = 0;
    if (producer && lane == 0) {
        policy = (a.l2_policy == 0) ? make_policy_evict_first()
                                    : make_policy_evict_last(__uint_as_float(
                                          static_cast<uint32_t>(a.l2_policy)));
        issued = min(NS, total);
        for (int s = 0; s < issued; ++s) issue(s);
    }

    // ---- everything below reads results of earlier kernels
    pdl_wait();
    L2State* st = a.st;
    // QKV: the epilogue's position and this thread's first RoPE pair, requested
    // now so that their two dependent round trips hide under the input load
    // (kept in shared memory through the stream: no registers held there)
    __shared__ int s_pos;
    __shared__ float2 s_cs[EPI == EPI_QKV_ROPE ? kThreads : 1];
    int e_pos = 0;
    float2 e_cs = make_float2(1.0f, 0.0f);
    if constexpr (EPI == EPI_QKV_ROPE) {
        e_pos = __ldcg(&st->pos);
        const int gr = r0 + 2 * tid;
        if (tid < nrows / 2 && gr < a.d + a.kvd) {
            const int e = (gr < a.d ? gr : gr - a.d) % a.head_dim;
            e_cs = a.rope[static_cast<size_t>(e_pos) * (a.head_dim >> 1) + (e >> 1)];
        }
    }

    const float* src = a.src;
    if (a.emb != nullptr) {
        // every consumed token passes here (from the caller, a prompt or the
        // previous argmax): an id outside [0, V) is reported, and clamped so
        // that the read stays inside the table
        const int raw = __ldcg(&st->token);
        const int tok = min(max(raw, 0), a.vocab - 1);
        if (raw != tok && blockIdx.x == 0 && tid == 0) atomicOr(&st->err, ERR_BAD_INPUT);
        src = a.emb + static_cast<size_t>(tok) * K;
    }
    const float4* src4 = reinterpret_cast<const float4*>(src);
    float4* xs4 = reinterpret_cast<float4*>(xs);
    if (a.zero_fixed != nullptr && blockIdx.x == 0)
        for (int i = tid; i < a.zero_n; i += kThreads) a.zero_fixed[i] = 0;
    if (a.src_fixed != nullptr) {
        // the residual in fixed point (value * 2^32): converted once into xs
        float ss = 0.0f;
        for (int i = tid; i < K; i += kThreads) {
            long long f = 0;
#pragma unroll
            for (int c = 0; c < kFfnCopies; ++c) f += __ldcg(a.src_fixed + static_cast<size_t>(c) * K + i);
            const float v = __ll2float_rn(f) * (1.0f / 4294967296.0f);
            xs[i] = v;
            ss += v * v;
        }
        ss = warp_sum(ss);
        if (lane == 0) scratch[warp] = ss;
        __syncthreads();
        if (warp == 0) {
            float t = lane < kWarps ? scratch[lane] : 0.0f;
            t = warp_sum(t);
            if (lane == 0) scratch[32] = 1.0f / sqrtf(t / static_cast<float>(K) + a.eps);
        }
        __syncthreads();
        if (a.gain != nullptr) {
            const float inv = scratch[32];
            for (int i = tid; i < K; i += kThreads) xs[i] = __ldg(a.gain + i) * (inv * xs[i]);
        }
    } else if (a.gain != nullptr) {
        float ss = 0.0f;
        for (int i = tid; i < K4; i += kThreads) {
            const float4 v = __ldcg(src4 + i);
            ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
        ss = warp_sum(ss);
        if (lane == 0) scratch[warp] = ss;
        __syncthreads();
        if (warp == 0) {
            float t = lane < kWarps ? scratch[lane] : 0.0f;
            t = warp_sum(t);
            if (lane == 0) scratch[32] = 1.0f / sqrtf(t / static_cast<float>(K) + a.eps);
        }
        __syncthreads();
        const float inv = scratch[32];
        const float4* g4 = reinterpret_cast<const float4*>(a.gain);
        for (int i = tid; i < K4; i += kThreads) {
            const float4 v = __ldcg(src4 + i);
            const float4 g = __ldg(g4 + i);
            xs4[i] = make_float4(g.x * (inv * v.x), g.y * (inv * v.y), g.z * (inv * v.z),
                                 g.w * (inv * v.w));
            if (a.x_init != nullptr && blockIdx.x == 0) reinterpret_cast<float4*>(a.x_init)[i] = v;
        }
    } else {
        for (int i = tid; i < K4; i += kThreads) xs4[i] = __ldcg(src4 + i);
    }
    if constexpr (EPI == EPI_QKV_ROPE) {
        if (tid == 0) s_pos = e_pos;
        s_cs[tid] = e_cs;
    }
    __syncthreads();

    if (producer) {
        if (lane == 0) {
            for (int s = issued; s < total; ++s) {
                const int b = s % NS;
                if (!mbar_wait_bounded(&empty[b], static_cast<uint32_t>(s / NS - 1) & 1u)) {
                    atomicOr(&st->err, ERR_TIMEOUT_TMA);
                    s_flag = 1;
                    break;
                }
                issue(s);
                issued = s + 1;
            }
            if (s_flag) {
                // drain the copies still in flight (bounded) before leaving
                for (int q = max(0, issued - NS); q < issued; ++q)
                    mbar_wait_bounded(&full[q % NS], static_cast<uint32_t>(q / NS) & 1u);
            }
        }
    } else {
        const int pc = warp % WPR;           // column part of this warp
        const int rw = warp / WPR;           // first row slot of this warp
        const int rstep = kConsumerWarps / WPR;
        const int cstride = 32 * WPR;
        float4 xr[kVec];
        if (NCH == 1) {
#pragma unroll
            for (int j = 0; j < kVec; ++j) {
                const int c = pc * 32 + lane + cstride * j;
                xr[j] = c < K4 ? xs4[c] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        float run = 0.0f;
        for (int s = 0; s < total; ++s) {
            const int b = s % NS;
            if (!mbar_wait_bounded(&full[b], static_cast<uint32_t>(s / NS) & 1u)) {
                if (lane == 0) {
                    atomicOr(&st->err, ERR_TIMEOUT_TMA);
                    s_flag = 1;
                }
                break;
            }
            const float4* stage4 =
                reinterpret_cast<const float4*>(ring + static_cast<size_t>(b) * P.stage_floats);
            if (NCH > 1) {
                const int c0 = (s % NCH) * P.chunk_floats;
                const int len4 = min(P.chunk_floats, K - c0) >> 2;
                const float4* x4 = xs4 + (c0 >> 2);
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int j = 0; j < kVec; ++j) {
                    const int c = pc * 32 + lane + cstride * j;
                    if (c < len4) {
                        const float4 w = stage4[c], x = x4[c];
                        acc.x = fmaf(w.x, x.x, acc.x);
                        acc.y = fmaf(w.y, x.y, acc.y);
                        acc.z = fmaf(w.z, x.z, acc.z);
                        acc.w = fmaf(w.w, x.w, acc.w);
                    }
                }
                run += warp_sum((acc.x + acc.y) + (acc.z + acc.w));
                if (s % NCH == NCH - 1) {
                    if (lane == 0) part[(s / NCH) * WPR + pc] = run;
                    run = 0.0f;
                }
            } else {
                const int lr0 = s * TR;
                const int nr = min(TR, nrows - lr0);
                for (int rr = 0; rr < RPW; ++rr) {
                    const int r = rw + rr * rstep;
                    if (r >= nr) break;
                    const float4* w4 = stage4 + static_cast<size_t>(r) * K4;
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int j = 0; j < kVec; ++j) {
                        const int c = pc * 32 + lane + cstride * j;
                        if (c < K4) {
                            const float4 w = w4[c];
                            acc.x = fmaf(w.x, xr[j].x, acc.x);
                            acc.y = fmaf(w.y, xr[j].y, acc.y);
                            acc.z = fmaf(w.z, xr[j].z, acc.z);
                            acc.w = fmaf(w.w, xr[j].w, acc.w);
                        }
                    }
                    const float sum = warp_sum((acc.x + acc.y) + (acc.z + acc.w));
                    if (lane == 0) part[(lr0 + r) * WPR + pc] = sum;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[b]);
        }
    }
    __syncthreads();
    if (s_flag) return;

    auto rowval = [&](int i) {
        float v = 0.0f;
        for (int q = 0; q < WPR; ++q) v += part[i * WPR + q];
        return v;
    };

    // ---- epilogue
    if constexpr (EPI == EPI_RESIDUAL) {
        for (int i = tid; i < nrows; i += kThreads) {
            float* o = a.out + r0 + i;
            *o = __ldcg(o) + rowval(i);
        }
    } else if constexpr (EPI == EPI_SWIGLU) {
        for (int i = tid; i < nrows / 2; i += kThreads) {
            const float g = rowval(2 * i), u = rowval(2 * i + 1);
            a.out[r0 / 2 + i] = (g / (1.0f + expf(-g))) * u;
        }
    } else if constexpr (EPI == EPI_QKV_ROPE) {
        const int pos = s_pos;
        const int slot = pos % a.seq_len;  // == pos unless the cache rolls
        const int hd = a.head_dim, half = hd >> 1;
        const float2* rope = a.rope + static_cast<size_t>(pos) * half;  // absolute position
        for (int i = tid; i < nrows / 2; i += kThreads) {
            const int gr = r0 + 2 * i;
            const float x0 = rowval(2 * i), x1 = rowval(2 * i + 1);
            if (gr < a.d) {
                const float2 cs = i == tid ? s_cs[tid] : rope[(gr % hd) >> 1];
                a.q_out[gr] = x0 * cs.x - x1 * cs.y;
                a.q_out[gr + 1] = x0 * cs.y + x1 * cs.x;
            } else if (gr < a.d + a.kvd) {
                const int j = gr - a.d, kvh = j / hd, e = j % hd;
                const float2 cs = i == tid ? s_cs[tid] : rope[e >> 1];
                float* dst = a.k_cache + (static_cast<size_t>(kvh) * a.seq_len + slot) * hd + e;
                dst[0] = x0 * cs.x - x1 * cs.y;
                dst[1] = x0 * cs.y + x1 * cs.x;
            } else {
                const int j = gr - a.d - a.kvd, kvh = j / hd, e = j % hd;
                float* dst = a.v_cache + (static_cast<size_t>(kvh) * a.seq_len + slot) * hd + e;
                dst[0] = x0;
                dst[1] = x1;
            }
        }
    } else if constexpr (EPI == EPI_CLASSIFIER) {
        unsigned long long best = 0ull;
        bool nan = false;
        for (int i = tid; i < nrows; i += kThreads) {
            const float v = rowval(i);
            a.out[r0 + i] = v;
            nan |= (v != v);
            const unsigned long long k = argmax_key(v, r0 + i);
            best = k > best ? k : best;
        }
        best = warp_max_u64(best);
        __shared__ unsigned long long s_best[kWarps];
        if (lane == 0) s_best[warp] = best;
        if (__syncthreads_or(nan) && tid == 0) atomicOr(&st->err, ERR_NAN);
        if (tid == 0) {
            for (int w = 0; w < kWarps; ++w) best = s_best[w] > best ? s_best[w] : best;
            atomicMax(&st->argmax_key, best);
            __threadfence();
            const unsigned int prev = atomicAdd(&st->cls_done, 1u);
            if (prev == gridDim.x - 1) {
                // last CTA: every CTA's atomicMax is visible
                __threadfence();
                const unsigned long long k = atomicExch(&st->argmax_key, 0ull);
                st->cls_done = 0u;
                const int idx = (k == 0ull) ? 0 : argmax_key_index(k);
                st->last_argmax = idx;
                const int pos = st->pos;
                if (st->mode == 1) {
                    const int np = st->n_prompt;
                    if (pos >= np - 1) st->out_tokens[pos - (np - 1)] = idx;
                    st->token = (pos + 1 < np) ? st->prompt[pos + 1] : idx;
                }
                if (st->mode != 2) st->pos = pos + 1;  // mode 2: the sampler advances
                __threadfence();
            }
        }
    }
}

template <int EPI>
cudaError_t launch_one(const MatvecArgs& a, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(a.plan.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = a.plan.smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, matvec_kernel<EPI>, a);
}

}  // namespace

namespace {

template <int EPI>
cudaError_t raise_smem_limit(int optin) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, matvec_kernel<EPI>);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(matvec_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                optin - static_cast<int>(fa.sharedSizeBytes));
}

}  // namespace

// Sets every instantiation's dynamic shared-memory limit to the most the current
// device allows. The attribute is process-wide, so it is never set to one
// handle's smaller need: that would break launches of a larger live handle.
cudaError_t set_matvec_smem_limits() {
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    if ((e = raise_smem_limit<EPI_QKV_ROPE>(optin)) != cudaSuccess) return e;
    if ((e = raise_smem_limit<EPI_RESIDUAL>(optin)) != cudaSuccess) return e;
    if ((e = raise_smem_limit<EPI_SWIGLU>(optin)) != cudaSuccess) return e;
    return raise_smem_limit<EPI_CLASSIFIER>(optin);
}

cudaError_t launch_matvec(int epi, const MatvecArgs& a, cudaStream_t s, bool pdl) {
    switch (epi) {
        case EPI_QKV_ROPE: return launch_one<EPI_QKV_ROPE>(a, s, pdl);
        case EPI_RESIDUAL: return launch_one<EPI_RESIDUAL>(a, s, pdl);
        case EPI_SWIGLU: return launch_one<EPI_SWIGLU>(a, s, pdl);
        case EPI_CLASSIFIER: return launch_one<EPI_CLASSIFIER>(a, s, pdl);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace l2
