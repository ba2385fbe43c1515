// sample.cu -- temperature / top-p sampling of the next token on the device,
// in place of the greedy choice, for generation on the batch-1 path.
//
// The pages print stories sampled by the single-file engine (新智元 article,
// "使用指南"; openai.wiki "模型推理") and mention its C sampling code
// (openai.wiki "未排序的待办事项") without stating the rule. Reading taken:
//   temperature <= 0: the greedy choice;
//   p_i = expf((l_i - max_j l_j) / temperature), total = sum of p;
//   0 < topp < 1: the nucleus is the smallest set of highest p whose mass
//   reaches topp * total, widened to every token whose p equals the last one
//   taken (otherwise the nucleus is every token); with r = u * (mass of the
//   nucleus), the token is the first nucleus member, in increasing index
//   order, whose running sum exceeds r (the last member if none does).
// u is the caller's uniform number of this draw (one per generated token).
//
// Batch-1 generation draws after every forward (sample_kernel); batched
// generation draws every sequence's token of a lockstep step, one CTA per
// sequence (bsample_kernel). One CTA of 1024 threads per draw; thread t owns
// the contiguous indices
// [t * per, (t + 1) * per). Every sum is a fixed-order block reduction, so the
// result does not depend on timing. The nucleus threshold is found without a
// sort: the mass of {p >= v} only falls as v grows, so a binary search over
// the bit patterns of positive floats (31 steps) finds the largest v whose
// mass still reaches topp * total; that v is the p of the last token a
// sorted walk would take.
#include <math.h>

#include "l2_internal.cuh"

namespace l2 {

namespace {

constexpr int kSampleThreads = 1024;
constexpr int kSampleWarps = kSampleThreads / 32;

// Sum of v over the block in a fixed order, returned to every thread.
__device__ __forceinline__ float block_sum(float v, float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_sum(v);
    __syncthreads();  // red is free again
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = lane < kSampleWarps ? red[lane] : 0.0f;
    t = warp_sum(t);  // every warp reduces the same 32 values in the same order
    return t;
}

// Exclusive prefix sum of v in thread order, fixed order.
__device__ __forceinline__ float block_exclusive_scan(float v, float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float n = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += n;
    }
    __syncthreads();
    if (lane == 31) red[warp] = inc;
    __syncthreads();
    float off = 0.0f;
    for (int w = 0; w < warp; ++w) off += red[w];
    float ex = __shfl_up_sync(0xffffffffu, inc, 1);
    if (lane == 0) ex = 0.0f;
    return off + ex;
}

// The draw of one token from logits lg[0..V) (every thread of the CTA calls
// it; the token is returned to all). amax: index of the largest logit (its
// value is subtracted before exp). T <= 0: amax itself.
__device__ int sample_from_logits(const float* lg, int V, float T, float topp, float u, int amax,
                                  float* red, int* s_pick, int* s_owner) {
    if (!(T > 0.0f)) return amax;
    const float mx = __ldcg(lg + amax);
    const int per = (V + kSampleThreads - 1) / kSampleThreads;
    const int i0 = min(V, static_cast<int>(threadIdx.x) * per), i1 = min(V, i0 + per);
    auto prob = [&](int i) { return expf((__ldcg(lg + i) - mx) / T); };
    float part = 0.0f;
    for (int i = i0; i < i1; ++i) part += prob(i);
    const float total = block_sum(part, red);
    float v = 0.0f;  // nucleus: p >= v
    if (topp > 0.0f && topp < 1.0f) {
        const float target = topp * total;
        uint32_t lo = 0u, hi = 0x3f800001u;  // mass(p >= 0) = total; nothing is > 1
        while (hi - lo > 1u) {
            const uint32_t mid = lo + (hi - lo) / 2u;
            const float vm = __uint_as_float(mid);
            float m = 0.0f;
            for (int i = i0; i < i1; ++i) {
                const float p = prob(i);
                if (p >= vm) m += p;
            }
            if (block_sum(m, red) >= target)
                lo = mid;
            else
                hi = mid;
        }
        v = __uint_as_float(lo);
    }
    float mine = 0.0f;
    int last_here = -1;
    for (int i = i0; i < i1; ++i) {
        const float p = prob(i);
        if (p >= v) {
            mine += p;
            last_here = i;
        }
    }
    const float mass = block_sum(mine, red);
    const float r = u * mass;
    const float before = block_exclusive_scan(mine, red);
    if (threadIdx.x == 0) {
        *s_pick = -1;
        *s_owner = kSampleThreads;
    }
    __syncthreads();
    // the draw falls in the first range whose running end passes r
    if (mine > 0.0f && before + mine > r) atomicMin(s_owner, static_cast<int>(threadIdx.x));
    if (last_here >= 0) atomicMax(s_pick, last_here);  // last nucleus member
    __syncthreads();
    if (static_cast<int>(threadIdx.x) == *s_owner) {
        float cum = before;
        int found = last_here;  // rounding: r past this range's own sum
        for (int i = i0; i < i1; ++i) {
            const float p = prob(i);
            if (p < v) continue;
            cum += p;
            if (cum > r) {
                found = i;
                break;
            }
        }
        *s_pick = found;
    }
    __syncthreads();
    const int pick = *s_pick;
    __syncthreads();  // s_pick / s_owner are free for the next call
    return pick;
}

__global__ void __launch_bounds__(kSampleThreads) sample_kernel(const SampleArgs a) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ float red[kSampleWarps];
    __shared__ int s_pick, s_owner;
    L2State* st = a.st;
    const int pos = st->pos, np = st->n_prompt;
    if (pos < np - 1) {  // a prompt position: the next token is forced
        if (threadIdx.x == 0) {
            st->token = st->prompt[pos + 1];
            st->pos = pos + 1;
        }
        return;
    }
    const int k = pos - (np - 1);
    const int pick = sample_from_logits(a.logits, a.vocab, st->temperature, st->topp,
                                        st->uniforms[k], st->last_argmax, red, &s_pick, &s_owner);
    if (threadIdx.x == 0) {
        st->out_tokens[k] = pick;
        st->token = pick;
        st->last_argmax = pick;
        st->pos = pos + 1;
    }
}

// Batched generation with sampling: the per-sequence advance of a lockstep
// step (as the greedy advance: prompt tokens forced, finished sequences
// inactive), the token of a generated position drawn from the row's logits
// with that sequence's uniform number for this token.
__global__ void __launch_bounds__(kSampleThreads) bsample_kernel(const BSampleArgs a) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ float red[kSampleWarps];
    __shared__ int s_pick, s_owner;
    const int b = a.row0 + blockIdx.x;
    const unsigned long long key = a.keys[b];
    const int amax = (key == 0ull) ? 0 : argmax_key_index(key);
    __syncthreads();  // every thread read the key before it is cleared
    if (threadIdx.x == 0) a.keys[b] = 0ull;
    if (a.active[b] == 0) return;
    const int p = a.pos[b], np = a.len[b];
    int idx = amax;
    if (p >= np - 1) {
        const int k_out = p - (np - 1);
        const SampleParams sp = *a.params;
        idx = sample_from_logits(a.logits + static_cast<size_t>(b) * a.vocab, a.vocab,
                                 sp.temperature, sp.topp,
                                 sp.uniforms[static_cast<size_t>(b) * a.steps + k_out], amax, red,
                                 &s_pick, &s_owner);
        if (threadIdx.x == 0) {
            a.last[b] = idx;
            a.out[static_cast<size_t>(b) * a.steps + k_out] = idx;
            if (k_out + 1 >= a.steps) {
                a.active[b] = 0;  // finished: its row is still computed, never used
                return;
            }
        }
        if (k_out + 1 >= a.steps) return;
    } else if (threadIdx.x == 0) {
        a.last[b] = amax;
    }
    if (threadIdx.x == 0) {
        a.token[b] = (p + 1 < np) ? a.prompts[a.poff[b] + p + 1] : idx;
        a.pos[b] = p + 1;
    }
}

}  // namespace

cudaError_t launch_bsample(const BSampleArgs& a, int M, cudaStream_t s, bool pdl) {
    if (M < 1 || a.params == nullptr || a.logits == nullptr) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(M);
    cfg.blockDim = dim3(kSampleThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, bsample_kernel, a);
}

cudaError_t launch_sample(const SampleArgs& a, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kSampleThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, sample_kernel, a);
}

}  // namespace l2
