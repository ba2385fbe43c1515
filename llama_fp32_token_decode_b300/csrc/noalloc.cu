// noalloc.cu -- greedy classifier entry point that allocates no memory.
//
// The classifier + argmax kernel needs scratch beyond its inputs and outputs:
// the vocabulary's logits and the cross-CTA argmax state (a packed
// (value, index) key and an arrival counter). The handle-based calls keep that
// scratch in memory l2_create allocated. l2_classify_greedy_noalloc serves
// callers that cannot allocate device memory themselves (a host whose device
// memory is owned by another framework's arena, or a serving loop that must
// not stall other streams on cudaMalloc/cudaFree): its scratch is the
// file-scope device array below, which every GPU that loads the library holds
// until the process exits.
//
// Host code must not pass the array's name to a kernel: on the host it is a
// stand-in symbol, not a device address. The device address is looked up once
// per device with cudaGetSymbolAddress (on the first call made with that
// device current) and passed to the kernels.
#include <mutex>

#include "l2_internal.cuh"

namespace l2 {
namespace {

// State block first (256 bytes), then logits[L2_NOALLOC_MAX_VOCAB].
constexpr size_t kStateBytes = 256;
static_assert(sizeof(L2State) <= kStateBytes, "state block too small");
constexpr size_t kScratchBytes = kStateBytes + sizeof(float) * L2_NOALLOC_MAX_VOCAB;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

struct DeviceSetup {
    bool done = false;
    unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch
    int num_sms = 0;
    int smem_optin = 0;  // shared memory a CTA may opt in to
};
DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mu;

// The entry point reports through its return code only (it has no handle to
// hold an error text).
int fail(int code, const char*) { return code; }

int cuda_fail(cudaError_t e, const char*) {
    return e == cudaErrorMemoryAllocation ? L2_ENOMEM : L2_ECUDA;
}

// Clears the state block: no argmax yet, no arrivals, no error, token -1.
__global__ void noalloc_init_kernel(L2State* st) {
    st->pos = 0;
    st->token = 0;
    st->n_prompt = 0;
    st->mode = 0;
    st->last_argmax = -1;
    st->err = 0;
    st->prompt = nullptr;
    st->out_tokens = nullptr;
    st->argmax_key = 0ull;
    st->cls_done = 0u;
}

// Copies the result out of the scratch: the token (-1 when a bounded wait gave
// up) and, when requested, its logit.
__global__ void noalloc_finish_kernel(const L2State* st, const float* logits, int32_t* token,
                                      float* logit) {
    const int idx = (st->err & (ERR_TIMEOUT_TMA | ERR_BAD_PLAN)) ? -1 : st->last_argmax;
    *token = idx;
    if (logit) *logit = idx >= 0 ? logits[idx] : __int_as_float(0x7fc00000);
}

int setup_device(int dev, DeviceSetup** out) {
    if (dev < 0 || dev >= kMaxDevices) return fail(L2_ECUDA, "device index out of range");
    std::lock_guard<std::mutex> lock(g_setup_mu);
    DeviceSetup& s = g_setup[dev];
    if (!s.done) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
        int sms = 0, optin = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        e = set_matvec_smem_limits();
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
        s.scratch = static_cast<unsigned char*>(p);
        s.num_sms = sms;
        s.smem_optin = optin;
        s.done = true;
    }
    *out = &s;
    return L2_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace l2

using namespace l2;

extern "C" {

int l2_classify_greedy_noalloc(const float* d_x, const float* d_gain, const float* d_wcls,
                               int32_t dim, int32_t vocab, float norm_eps, int32_t* d_token,
                               float* d_logit, void* stream) {
    if (!d_x || !d_gain || !d_wcls || !d_token)
        return fail(L2_EINVAL, "NULL input or token buffer");
    if (vocab < 1 || vocab > L2_NOALLOC_MAX_VOCAB)
        return fail(L2_EINVAL, "vocab must be in [1, L2_NOALLOC_MAX_VOCAB] (scratch holds that many logits)");
    if (dim < 4 || dim > 16384 || dim % 4 != 0)
        return fail(L2_EINVAL, "dim must be a multiple of 4 in [4, 16384]");
    if (!(norm_eps >= 0.0f)) return fail(L2_EINVAL, "norm_eps must be >= 0");
    if (!aligned16(d_x) || !aligned16(d_gain) || !aligned16(d_wcls))
        return fail(L2_EINVAL, "d_x, d_gain and d_wcls must be 16-byte aligned");

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    DeviceSetup* s = nullptr;
    int rc = setup_device(dev, &s);
    if (rc != L2_OK) return rc;

    L2State* st = reinterpret_cast<L2State*>(s->scratch);
    float* logits = reinterpret_cast<float*>(s->scratch + kStateBytes);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);

    MatvecArgs a{};
    a.W = d_wcls;
    a.plan = plan_matvec(vocab, dim, 1, s->num_sms);
    // the opt-in limit covers static + dynamic shared memory; keep 1 KB for the static part
    if (a.plan.smem_bytes + 1024 > static_cast<size_t>(s->smem_optin))
        return fail(L2_EINVAL, "dim needs more shared memory than a CTA has");
    a.src = d_x;
    a.gain = d_gain;
    a.eps = norm_eps;
    a.out = logits;
    a.vocab = vocab;
    a.d = dim;
    a.st = st;
    // the classifier belongs to the caller: stream it with the evict_first hint
    // (policy 0), so that the call leaves none of it marked to stay in L2 at
    // the expense of the caller's own working set
    a.l2_policy = 0;

    noalloc_init_kernel<<<1, 1, 0, cs>>>(st);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "init launch");
    if ((e = launch_matvec(EPI_CLASSIFIER, a, cs, false)) != cudaSuccess)
        return cuda_fail(e, "classifier launch");
    noalloc_finish_kernel<<<1, 1, 0, cs>>>(st, logits, d_token, d_logit);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "finish launch");
    return L2_OK;
}

}  // extern "C"
