// layout.cu -- one-time re-tiling of the documented row-major blob into the
// streaming layout the decode kernels read.
//
// The blob (a raw fp32 file in the llama2.c pages) stores W1 and W3 as two
// separate [F][d] matrices per layer. The SwiGLU epilogue needs the gate row
// and the up row of the same hidden unit in the same CTA, so the layout pass
// interleaves them: row 2j = W1 row j, row 2j+1 = W3 row j. Q, K and V are
// concatenated per layer ([Wq; Wk; Wv]) by the uploader with plain copies, so
// one launch streams all three and RoPE pairs (2i, 2i+1) stay adjacent.
// Rows stay row-major: a warp reading 32 consecutive 16-byte vectors of a row
// is already a fully coalesced 512-byte access.
#include "l2_internal.cuh"

namespace l2 {

namespace {

__global__ void interleave_rows_kernel(float4* __restrict__ dst, const float4* __restrict__ a,
                                       const float4* __restrict__ b, long long rows, int cols4) {
    const long long total = rows * cols4;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long r = i / cols4;
        const int c = static_cast<int>(i - r * cols4);
        dst[(2 * r) * cols4 + c] = a[i];
        dst[(2 * r + 1) * cols4 + c] = b[i];
    }
}

// Wo as per-head column blocks, so that the CTAs of head h read rows of a
// contiguous [d][hd] block.
__global__ void retile_heads_kernel(float* __restrict__ dst, const float* __restrict__ src,
                                    long long total, int d, int hd) {
    const int H = d / hd;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int e = static_cast<int>(i % hd);
        long long t = i / hd;
        const int r = static_cast<int>(t % d);
        t /= d;
        const int h = static_cast<int>(t % H);
        const long long l = t / H;
        dst[i] = src[(l * d + r) * d + static_cast<long long>(h) * hd + e];
    }
}

// W2 transposed per layer, so that the CTA owning hidden units u0..u1 reads
// their columns as contiguous rows.
__global__ void transpose_layers_kernel(float* __restrict__ dst, const float* __restrict__ src,
                                        long long total, int rows, int cols) {
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int r = static_cast<int>(i % rows);
        long long t = i / rows;
        const int c = static_cast<int>(t % cols);
        const long long l = t / cols;
        dst[i] = src[(l * rows + r) * cols + c];
    }
}

}  // namespace

cudaError_t launch_retile_heads(float* dst, const float* src, int layers, int d, int hd,
                                cudaStream_t s) {
    if (hd < 1 || d % hd != 0) return cudaErrorInvalidValue;
    retile_heads_kernel<<<4096, 256, 0, s>>>(dst, src, static_cast<long long>(layers) * d * d, d, hd);
    return cudaGetLastError();
}

cudaError_t launch_transpose_layers(float* dst, const float* src, int layers, int rows, int cols,
                                    cudaStream_t s) {
    transpose_layers_kernel<<<4096, 256, 0, s>>>(
        dst, src, static_cast<long long>(layers) * rows * cols, rows, cols);
    return cudaGetLastError();
}

cudaError_t launch_interleave_rows(float* dst, const float* a, const float* b, long long rows,
                                   int cols, cudaStream_t s) {
    if (cols % 4 != 0) return cudaErrorInvalidValue;
    const int cols4 = cols / 4;
    interleave_rows_kernel<<<4096, 256, 0, s>>>(reinterpret_cast<float4*>(dst),
                                                reinterpret_cast<const float4*>(a),
                                                reinterpret_cast<const float4*>(b), rows, cols4);
    return cudaGetLastError();
}

}  // namespace l2
