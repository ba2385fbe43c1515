// gemm_tf32x3.cu -- fp32-accurate tensor-core GEMM of the batched decode step.
//
// With B sequences decoded in lockstep, every projection of the Llama-2
// decode step (the fp32 engine of the llama2.c pages) becomes a dense
// contraction  C[B][N] = X[B][K] * W[N][K]^T.  fp32 accuracy on the tensor
// cores comes from the 3xTF32 split: every operand is stored as a pair
// hi = round_tf32(v), lo = v - hi (exact in fp32), and
//     C = Xhi*Whi + Xhi*Wlo + Xlo*Whi
// drops only the Xlo*Wlo term (relative size 2^-22), with fp32 accumulation.
//
// Kernel (sm_103a, one 128 x BN output tile per CTA, 256 threads; BN 64,
// 128 or 256; details at the kernel):
//   * warp 0 lane 0 streams K-blocks of 32 floats (128 bytes, one 128-byte
//     swizzle row) of Xhi, Xlo, Whi, Wlo into a ring of shared-memory stages
//     with 3-D TMA tile loads (completion on mbarriers); weight tiles of the
//     first stages are requested before griddepcontrol.wait, since weights
//     never depend on the previous kernel;
//   * warp 1 lane 0 issues tcgen05.mma kind::tf32 (M 128, or 64 for launches of
//     at most 64 rows; N BN, K 8) from the
//     stages into a TMEM accumulator (128 lanes x BN fp32 columns) and frees
//     each stage with tcgen05.commit; idle warps meanwhile stage per-row data
//     the epilogue needs (row positions, RMSNorm row scales);
//   * every warp then reads the accumulator with tcgen05.ld (warp w: TMEM
//     lanes 32 (w mod 4) .. + 31 = output rows) and applies the fused
//     epilogue; a K split over a thread-block cluster first adds the CTAs'
//     partial tiles through distributed shared memory.
// Every wait is bounded; on a timeout the kernel records ERR_TIMEOUT_TMA,
// drains its own copies, frees its TMEM and returns.
#include <math.h>
#include <stdio.h>

#include <mutex>

#include "l2_internal.cuh"

namespace l2 {

namespace {

// ------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::tf32, cta_group::1.
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives on `bar` once every tcgen05.mma this thread issued before has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart (stride
// byte offset), leading byte offset unused for this layout (encoded 1),
// descriptor version 1 (bits 46-48), swizzle mode 2 = 128-byte (bits 61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor, kind::tf32: D fp32 (bits 4-5 = 1), A and B tf32
// (bits 7-9 and 10-12 = 2), both K-major (bits 15, 16 = 0), N >> 3 at bits
// 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// Dynamic shared memory one CTA may use (227 KB opt-in, minus static use:
// the row-state and row-scale arrays and the error flag).
constexpr size_t kMaxDynSmem = 227 * 1024 - 3072;

template <int BN>
struct Cfg {
    static constexpr int BM = 128, BK = 32;
    static constexpr int A_BYTES = BM * BK * 4;  // 16 KB
    static constexpr int B_BYTES = BN * BK * 4;
    static constexpr int STAGE = 2 * A_BYTES + 2 * B_BYTES;
    static constexpr int STAGES = (BN >= 256) ? 2 : (BN == 128) ? 3 : 4;  // deepest ring that fits
    static constexpr int MAX_STAGES = 6;  // with 64-row A tiles
    // bytes of one ring slot when the A tiles hold a_rows rows (Ahi, Alo, Bhi, Blo)
    __host__ __device__ static constexpr int stage_bytes(int a_rows) {
        return 2 * a_rows * BK * 4 + 2 * B_BYTES;
    }
    // TMEM columns: one accumulator, or two when chunks are drained
    __host__ __device__ static constexpr uint32_t tmem_cols(bool drain) {
        return drain ? 2 * BN : BN;
    }
    static constexpr int PS = BN + 4;  // row stride (floats) of a staged partial tile
    // split-K receive buffer: one slot per peer, ceil(a_rows / S) rows of PS
    // floats (each CTA of the cluster owns that share of the tile's rows)
    __host__ __device__ static constexpr size_t recv_bytes(int ksplit, int a_rows = 128) {
        return ksplit > 1
                   ? static_cast<size_t>(ksplit - 1) * ((a_rows + ksplit - 1) / ksplit) * PS * 4
                   : 0;
    }
    // dynamic shared memory of a launch: alignment slack, a ring of `stages`
    // slots (>= 2: the staged partial tile reuses the first two), the receive
    // buffer of a split launch, barriers
    __host__ __device__ static constexpr size_t smem_for(int stages, int ksplit, int a_rows = 128) {
        return 1024 + static_cast<size_t>(stages) * stage_bytes(a_rows) + recv_bytes(ksplit, a_rows) + 256;
    }
    static_assert(128 * PS * 4 <= 2 * STAGE, "partial tile must fit in two slots");
    static_assert(128 * PS * 4 <= 2 * (2 * 64 * BK * 4 + 2 * B_BYTES),
                  "partial tile must fit in two slots of 64-row A tiles");
    static_assert((64 * BK * 4) % 1024 == 0, "64-row A tiles keep 1024-byte alignment");
    static_assert(STAGE % 1024 == 0, "stages must keep 1024-byte alignment");
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "N tile");
};

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// ---- cluster helpers (split-K reduction through distributed shared memory)

__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_peer(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
// Generic-proxy shared-memory writes become visible to bulk copies.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Bulk copy of `bytes` from this CTA's shared memory into a peer's (dst and
// bar are shared::cluster addresses from mapa), completion counted on bar.
__device__ __forceinline__ void bulk_s2peer(uint32_t dst, uint32_t src, uint32_t bytes,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes"
        " [%0], [%1], %2, [%3];" ::"r"(dst),
        "r"(src), "r"(bytes), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void bulk_commit_and_wait_read() {
    asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Per-row state the QKV epilogue needs: position, whether the row is active,
// and the KV cache it appends to.
struct RowState {
    int pos, active, cache;
};

// Global operands of one output group's epilogue, loaded ahead of the
// partial sums so that their latency overlaps the reduction: the residual's
// four values (RESIDUAL), the RoPE (cos, sin) pairs of the group's two
// column pairs (QKV).
struct EpiPre {
    float4 x;
    float2 cs[2];
};

template <int EPI>
__device__ __forceinline__ EpiPre epi_pre(const GemmArgs& g, int r, int gc, const RowState& rs) {
    EpiPre p;
    p.x = make_float4(0.f, 0.f, 0.f, 0.f);
    p.cs[0] = p.cs[1] = make_float2(1.f, 0.f);
    if constexpr (EPI == GEPI_RESIDUAL) {
        if (gc + 4 <= g.N && (g.ldc & 3) == 0)
            p.x = __ldcg(reinterpret_cast<const float4*>(g.out + static_cast<size_t>(r) * g.ldc + gc));
    } else if constexpr (EPI == GEPI_QKV_ROPE) {
        if (rs.active) {
            const int hd = g.head_dim;
            const float2* rope = g.rope + static_cast<size_t>(rs.pos) * (hd >> 1);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int c = gc + 2 * j;
                if (c + 1 < g.N && c < g.d + g.kvd)
                    p.cs[j] = rope[((c < g.d ? c : c - g.d) % hd) >> 1];
            }
        }
    }
    return p;
}

// Fused epilogue of four consecutive output columns gc..gc+3 (gc % 4 == 0) of
// row r. rs: the row's state (QKV only); pre: from epi_pre for the same group.
// ARGMAX folds the columns into `best`; the caller publishes it. Returns the
// sum of squares of the residual values written (RESIDUAL with x_hi set),
// else 0.
template <int EPI>
__device__ __forceinline__ float epi4(const GemmArgs& g, int r, int gc, const float (&a)[4],
                                      const RowState& rs, const EpiPre& pre,
                                      unsigned long long& best) {
    if constexpr (EPI == GEPI_STORE || EPI == GEPI_RESIDUAL) {
        float* o = g.out + static_cast<size_t>(r) * g.ldc + gc;
        float w4[4] = {a[0], a[1], a[2], a[3]};
        int nw = 4;
        if (gc + 4 <= g.N && (g.ldc & 3) == 0) {
            if constexpr (EPI == GEPI_RESIDUAL) {
                w4[0] += pre.x.x;
                w4[1] += pre.x.y;
                w4[2] += pre.x.z;
                w4[3] += pre.x.w;
            }
            *reinterpret_cast<float4*>(o) = make_float4(w4[0], w4[1], w4[2], w4[3]);
        } else {
            nw = 0;
            for (int j = 0; j < 4 && gc + j < g.N; ++j, ++nw) {
                w4[j] = (EPI == GEPI_RESIDUAL) ? __ldcg(o + j) + a[j] : a[j];
                o[j] = w4[j];
            }
        }
        if constexpr (EPI == GEPI_RESIDUAL) {
            if (g.x_hi != nullptr) {  // the rows the next (norm-folded) GEMM reads
                float ss = 0.0f;
                float* xh = g.x_hi + static_cast<size_t>(r) * g.ldc + gc;
                float* xl = g.x_lo + static_cast<size_t>(r) * g.ldc + gc;
                if (nw == 4 && (g.ldc & 3) == 0) {
                    const float4 h = make_float4(tf32_round(w4[0]), tf32_round(w4[1]),
                                                 tf32_round(w4[2]), tf32_round(w4[3]));
                    *reinterpret_cast<float4*>(xh) = h;
                    *reinterpret_cast<float4*>(xl) =
                        make_float4(tf32_round(w4[0] - h.x), tf32_round(w4[1] - h.y),
                                    tf32_round(w4[2] - h.z), tf32_round(w4[3] - h.w));
                } else {
                    for (int j = 0; j < nw; ++j) {
                        const float h = tf32_round(w4[j]);
                        xh[j] = h;
                        xl[j] = tf32_round(w4[j] - h);
                    }
                }
                for (int j = 0; j < nw; ++j) ss = fmaf(w4[j], w4[j], ss);
                return ss;
            }
        }
    } else if constexpr (EPI == GEPI_SWIGLU) {
        // interleaved rows: column 2j is the gate, 2j+1 the up projection
        const size_t F = static_cast<size_t>(g.N) >> 1;
        const size_t idx = static_cast<size_t>(r) * F + (gc >> 1);
        if (gc + 4 <= g.N && (F & 1) == 0) {  // both outputs of the group, 8-byte aligned
            const float h0 = silu(a[0]) * a[1], h1 = silu(a[2]) * a[3];
            const float2 hi = make_float2(tf32_round(h0), tf32_round(h1));
            *reinterpret_cast<float2*>(g.out_hi + idx) = hi;
            *reinterpret_cast<float2*>(g.out_lo + idx) =
                make_float2(tf32_round(h0 - hi.x), tf32_round(h1 - hi.y));
        } else {
#pragma unroll
            for (int j = 0; j < 4; j += 2) {
                if (gc + j + 1 < g.N) {
                    const float h = silu(a[j]) * a[j + 1];
                    const float hi = tf32_round(h);
                    g.out_hi[idx + (j >> 1)] = hi;
                    g.out_lo[idx + (j >> 1)] = tf32_round(h - hi);
                }
            }
        }
    } else if constexpr (EPI == GEPI_QKV_ROPE) {
        if (!rs.active) return 0.0f;
        const int hd = g.head_dim, pos = rs.pos;
#pragma unroll
        for (int j = 0; j < 4; j += 2) {
            const int c = gc + j;
            if (c + 1 >= g.N) break;
            const float x0 = a[j], x1 = a[j + 1];
            const float2 cs = pre.cs[j >> 1];
            if (c < g.d) {
                float* q = g.q + static_cast<size_t>(r) * g.d + c;
                q[0] = x0 * cs.x - x1 * cs.y;
                q[1] = x0 * cs.y + x1 * cs.x;
            } else if (c < g.d + g.kvd) {
                const int jj = c - g.d, kvh = jj / hd, e = jj % hd;
                float* dst = g.k_cache + static_cast<size_t>(rs.cache) * g.cache_seq +
                             (static_cast<size_t>(kvh) * g.seq_len + pos % g.seq_len) * hd + e;
                dst[0] = x0 * cs.x - x1 * cs.y;
                dst[1] = x0 * cs.y + x1 * cs.x;
            } else {
                const int jj = c - g.d - g.kvd, kvh = jj / hd, e = jj % hd;
                float* dst = g.v_cache + static_cast<size_t>(rs.cache) * g.cache_seq +
                             (static_cast<size_t>(kvh) * g.seq_len + pos % g.seq_len) * hd + e;
                dst[0] = x0;
                dst[1] = x1;
            }
        }
    } else if constexpr (EPI == GEPI_ARGMAX) {
        float* o = g.out ? g.out + static_cast<size_t>(r) * g.ldc + gc : nullptr;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (gc + j < g.N) {
                if (o) o[j] = a[j];
                const unsigned long long k = argmax_key(a[j], gc + j);
                best = k > best ? k : best;
            }
        }
    }
    return 0.0f;
}

// Scale of row r of a norm-folded GEMM: 1 / sqrt(mean of x[r]^2 + eps), the
// sum of squares being the producer's partials added in slot order.
__device__ __forceinline__ float row_scale(const GemmArgs& g, int r) {
    // ss_stride is a multiple of 4: the slots are read as independent 16-byte loads
    const float4* p = reinterpret_cast<const float4*>(g.ss_in + static_cast<size_t>(r) * g.ss_stride);
    const int n = g.ss_count, n4 = (n + 3) >> 2;
    float ss = 0.0f;
#pragma unroll 4
    for (int j = 0; j < n4; ++j) {
        const float4 v = __ldcg(p + j);
        const int k = 4 * j;
        ss += v.x;
        ss += k + 1 < n ? v.y : 0.0f;
        ss += k + 2 < n ? v.z : 0.0f;
        ss += k + 3 < n ? v.w : 0.0f;
    }
    return 1.0f / sqrtf(ss / static_cast<float>(g.K) + g.eps);
}

// Row r's state, read from the arrays the previous kernels wrote.
__device__ __forceinline__ RowState load_row_state(const GemmArgs& g, int r) {
    RowState rs;
    // positions run past seq_len when the cache rolls: RoPE at the absolute
    // position (the table covers rope_positions), the KV slot pos % seq_len
    rs.pos = min(max(__ldcg(g.pos + r), 0),
                 (g.rope_positions > g.seq_len ? g.rope_positions : g.seq_len) - 1);
    rs.active = g.active ? __ldcg(g.active + r) : 1;
    rs.cache = g.seq ? __ldcg(g.seq + r) : r;
    return rs;
}

// Grid (S, tiles): blockIdx.x is the K split (the CTA's rank in a cluster of S
// CTAs that share one 128 x BN output tile), blockIdx.y the tile (M tiles of
// one N tile adjacent). Warp w reads TMEM lane quarter w % 4 (tile rows
// 32(w % 4) .. + 31). Without the chunk drain (eight warps) warp 0 lane 0
// issues TMA and warp 1 lane 0 the MMAs; afterwards warps w and w + 4 share
// the accumulator's 32-column chunks, and all eight run the epilogue (the
// epilogue is a chain of dependent loads and stores per output group, so it
// wants many warps in flight). With the drain (six warps) warps 0-3 drain
// chunks during the mainloop, so TMA and MMA issue move to warps 4 and 5.
//
// Accumulation precision: the tensor core adds into its fp32 accumulator
// without round-to-nearest. Measured against float64 (M 64, N 512): letting
// one accumulator absorb all of K gives a relative L2 error that grows with K
// and is biased toward zero (7.7e-5 at K = 11008, 2.3e-4 at 32768; a
// sequential fp32 loop gives 1.9e-6 and 3.3e-6), while the error of a chunk
// of c K-blocks is about 2.3e-7 * c whatever K is. So the MMAs of every
// kChunk K-blocks go into one of two TMEM accumulators in turn, and warps 0-3
// drain each finished chunk into registers with ordinary fp32 additions while
// the next chunk accumulates in the other buffer (accfull / accfree
// barriers): about 1e-6 at any K with 4-block chunks (2-block chunks halve
// that and cost the MMA thread twice the commits and waits: the 7B-shape
// prefill GEMMs 2-3 % slower).
//
// S == 1: the epilogue runs on the register sums (thread = row). S > 1: every
// CTA stages its partial tile in its own shared memory and pushes each peer's
// row slice into that peer's receive buffer (bulk copy, completion on the
// peer's mbarrier); CTA s adds rows [TR s / S, TR (s+1) / S) of the S
// partials (TR = 128, or 64 with 64-row A tiles) in rank order (a fixed
// order: the result does not depend on timing) and applies the epilogue to
// them.
// CONV (drained launches of 64-row handles): the weight tiles arrive as fp32
// (one copy, W * g where the RMSNorm gain is folded in, half the bytes of the
// tf32 pair) and kConvWarps extra warps split each landed tile in shared
// memory: the tensor core reads an fp32 operand as tf32 by dropping its 13
// low mantissa bits, so hi = w stays in place and lo = w - trunc(w), exact in
// fp32, goes to the lo tile (the tensor core truncates lo in turn: a relative
// error below 2^-20 of w, against 2^-23 for the rounded pair of the copies);
// the MMA warp waits for the split tile.
// SWAP (CONV with 128-wide tiles): the operands trade places, D^T = W x^T,
// the 128 weight rows being the M = 128 operand and the tile's 64 rows the
// N = 64 one. A tf32 MMA (K = 8) takes max(51, N / 2) cycles whether M is 64
// or 128 (measured on B300), so the same products cost 51 cycles each
// instead of 64; TMEM lane i then holds weight row n0 + i and column t tile
// row t, the drain leaves each thread one weight row's 64 sums, and the
// epilogue always stages the partial tile (row-major, as the unswapped path
// does) before it reads it back by rows, split or not.
constexpr int kConvWarps = 2;  // 8 warps in all: a ninth would cap a thread at 168 registers
constexpr int gemm_threads(bool drain, bool conv = false) {
    return drain ? (conv ? 192 + 32 * kConvWarps : 192) : 256;
}
constexpr int kChunk = 4;         // K-blocks per TMEM accumulation chunk (DRAIN)
constexpr int kDrainAbove = 16;   // a CTA with more K-blocks than this drains chunks

// DRAIN == false (a CTA's K range is at most kDrainAbove K-blocks, error below
// about 4e-6): one accumulator takes the whole range and the epilogue reads it
// from TMEM 32 columns at a time, without a register copy of the tile row.
template <int BN, int EPI, bool DRAIN, bool CONV>
__global__ void __launch_bounds__(gemm_threads(DRAIN, CONV), 1)
    gemm_tf32x3_kernel(const __grid_constant__ CUtensorMap mA_hi,
                       const __grid_constant__ CUtensorMap mA_lo,
                       const __grid_constant__ CUtensorMap mB_hi,
                       const __grid_constant__ CUtensorMap mB_lo, const GemmArgs g) {
    using C = Cfg<BN>;
    const int S = g.stages;       // ring depth of this launch
    constexpr int PS = C::PS;     // row stride of the staged partial (floats)
    // A tiles of g.a_rows rows (128, or 64 with M = 64 MMAs: launches of at
    // most 64 rows)
    // (CONV launches always hold 64-row tiles: compile-time sizes there)
    const int a_bytes = CONV ? 64 * C::BK * 4 : (g.a_rows == 64 ? 64 : 128) * C::BK * 4;
    const int stage_b = 2 * a_bytes + 2 * C::B_BYTES;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char* gbase = smem_raw + (base - raw);
    const int nsplit = gridDim.x, split = blockIdx.x;
    const uint32_t recv_base = base + static_cast<uint32_t>(S * stage_b);
    uint64_t* full = reinterpret_cast<uint64_t*>(gbase + static_cast<size_t>(S) * stage_b +
                                                 C::recv_bytes(nsplit, g.a_rows == 64 ? 64 : 128));
    uint64_t* empty = full + S;
    uint64_t* accfull = empty + S;   // [2] chunk accumulated in TMEM buffer b
    uint64_t* accfree = accfull + 2; // [2] TMEM buffer b drained
    uint64_t* recvb = accfree + 2;   // split-K: the peers' slices of this CTA's rows
    uint64_t* convb = recvb + 1;     // CONV: [S] the slot's weight tile is split
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(convb + (CONV ? S : 0));
    static_assert(!CONV || DRAIN, "the split warps come with the drained layout");
    // SWAP (CONV with 128-wide tiles, whose launches hold at most 64 rows): the
    // weight tile is the M = 128 operand and the 64 rows the N = 64 one
    constexpr bool SWAP = CONV && BN == 128;
    constexpr int RN = SWAP ? 64 : BN;  // TMEM columns of one accumulator
    __shared__ int s_err;
    // QKV epilogue: state of the tile's rows, loaded once during the mainloop
    __shared__ RowState s_rows[EPI == GEPI_QKV_ROPE ? 128 : 1];
    // norm-folded consumers (g.ss_in set): the tile's row scales, likewise
    __shared__ float s_scale[EPI == GEPI_RESIDUAL || EPI == GEPI_STORE ? 1 : 128];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mt = (g.M + 127) / 128;
    const int m0 = g.row0 + (blockIdx.y % mt) * 128;  // first row of this tile
    const int n0 = (blockIdx.y / mt) * BN;
    const int m_end = g.row0 + g.M;                   // rows of this launch end here
    const int KB = (g.K + 31) / 32;
    const int kb0 = KB * split / nsplit, kb1 = KB * (split + 1) / nsplit;
    const int NK = kb1 - kb0;
    constexpr int CH = DRAIN ? kChunk : (1 << 30);   // K-blocks per accumulation chunk
    const int NCH = DRAIN ? (NK + CH - 1) / CH : 1;  // chunks (the last drains in the epilogue)

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accfull[b], 1);
            mbar_init(&accfree[b], 4);
        }
        mbar_init(recvb, 1);
        if constexpr (CONV)
            for (int s = 0; s < S; ++s) mbar_init(&convb[s], kConvWarps);
        fence_mbar_init();
        s_err = 0;
        prefetch_map(&mA_hi);
        prefetch_map(&mA_lo);
        prefetch_map(&mB_hi);
        prefetch_map(&mB_lo);
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, C::tmem_cols(DRAIN));
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_launch_dependents();
    // split-K: announce this CTA's initialised barriers to the cluster now and
    // collect the peers' announcements only before pushing to them
    if (nsplit > 1) cluster_arrive_release();

    auto a_hi = [&](int s) { return base + static_cast<uint32_t>(s * stage_b); };
    auto a_lo = [&](int s) { return a_hi(s) + static_cast<uint32_t>(a_bytes); };
    auto b_hi = [&](int s) { return a_hi(s) + static_cast<uint32_t>(2 * a_bytes); };
    auto b_lo = [&](int s) { return b_hi(s) + C::B_BYTES; };

    // DRAIN, warps 0-3: this thread's row of the tile (SWAP: its weight row's
    // column of 64 tile rows), summed over chunks
    float R[DRAIN ? RN : 1];
#pragma unroll
    for (int j = 0; j < (DRAIN ? RN : 1); ++j) R[j] = 0.0f;

    constexpr int kProdWarp = DRAIN ? 4 : 0, kMmaWarp = DRAIN ? 5 : 1;
    // bytes a slot's copies bring: with CONV one fp32 weight tile, not the pair
    const uint32_t slot_tx = static_cast<uint32_t>(CONV ? 2 * a_bytes + C::B_BYTES : stage_b);
    if (warp == kProdWarp && (DRAIN || lane == 0)) {
        if (lane == 0) {
            // ---- producer: local K-block i is global K-block kb0 + i
            const int pre = NK < S ? NK : S;
            for (int i = 0; i < pre; ++i) {
                const int kc = (kb0 + i) * 32;
                mbar_arrive_expect_tx(&full[i], slot_tx);
                tma_load_3d(b_hi(i), &mB_hi, kc, n0, g.layer, &full[i]);
                if (!CONV) tma_load_3d(b_lo(i), &mB_lo, kc, n0, g.layer, &full[i]);
            }
            pdl_wait();  // activations come from the previous kernel
            for (int i = 0; i < pre; ++i) {
                const int kc = (kb0 + i) * 32;
                tma_load_3d(a_hi(i), &mA_hi, kc, m0, 0, &full[i]);
                tma_load_3d(a_lo(i), &mA_lo, kc, m0, 0, &full[i]);
            }
            int issued = pre;
            int s = 0;        // slot of K-block i (i % S), counted
            uint32_t ph = 0;  // parity of the empty phase it waits for ((i / S - 1) & 1)
            for (int i = pre; i < NK; ++i) {
                const int kc = (kb0 + i) * 32;
                if (!mbar_wait_bounded(&empty[s], ph)) {
                    s_err = 1;
                    break;
                }
                mbar_arrive_expect_tx(&full[s], slot_tx);
                tma_load_3d(b_hi(s), &mB_hi, kc, n0, g.layer, &full[s]);
                if (!CONV) tma_load_3d(b_lo(s), &mB_lo, kc, n0, g.layer, &full[s]);
                tma_load_3d(a_hi(s), &mA_hi, kc, m0, 0, &full[s]);
                tma_load_3d(a_lo(s), &mA_lo, kc, m0, 0, &full[s]);
                issued = i + 1;
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (s_err) {  // let the copies in flight land before the CTA leaves
                for (int q = issued - S < 0 ? 0 : issued - S; q < issued; ++q)
                    mbar_wait_bounded(&full[q % S], static_cast<uint32_t>(q / S) & 1u);
            }
        }
    } else if (warp == kMmaWarp && (DRAIN || lane == 0)) {
        if (lane == 0) {
            // ---- MMA issuer: chunk c accumulates in TMEM buffer c & 1; 64-row
            // A tiles take M = 64 MMAs (half the A reads), or with SWAP the
            // weight tile is M and the rows N = 64. The one issuing thread
            // sets the pace (each MMA waits for its own issue), so the loop
            // keeps its per-MMA work to additions: the slot's descriptors come
            // from the first slot's by constant offsets, and slot and phase
            // advance by counting.
            const uint32_t idesc = SWAP             ? idesc_tf32(128, 64)
                                   : g.a_rows == 64 ? idesc_tf32(64, BN)
                                                    : idesc_tf32(128, BN);
            const uint64_t d_base = sw128_desc(base);  // Ahi of slot 0
            const uint64_t d_slot = static_cast<uint64_t>(stage_b >> 4);
            const uint64_t o_al = static_cast<uint64_t>(a_bytes >> 4);
            const uint64_t o_bh = static_cast<uint64_t>((2 * a_bytes) >> 4);
            const uint64_t o_bl = o_bh + static_cast<uint64_t>(C::B_BYTES >> 4);
            int s = 0;
            uint32_t ph = 0;  // phase parity of slot s's barriers
            for (int i = 0; i < NK; ++i) {
                const int c = i / CH, w = i % CH, buf = c & 1;
                if (w == 0 && c >= 2 &&
                    !mbar_wait_bounded(&accfree[buf], static_cast<uint32_t>(c / 2 - 1) & 1u)) {
                    s_err = 1;
                    break;
                }
                uint64_t* ready = CONV ? &convb[s] : &full[s];
                if (!mbar_wait_bounded(ready, ph)) {
                    s_err = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t acc = tmem + static_cast<uint32_t>(buf * RN);
                // descriptor start addresses are in 16-byte units: + 2 per
                // 32-byte K step (the slots lie within shared memory, so the
                // 14-bit field does not carry)
                const uint64_t d_ah = d_base + static_cast<uint64_t>(s) * d_slot;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint64_t ah = d_ah + 2 * k;
                    const uint64_t al = ah + o_al;
                    const uint64_t bh = ah + o_bh;
                    const uint64_t bl = ah + o_bl;
                    if constexpr (SWAP) {  // D^T = W x^T: the same three products
                        mma_tf32(acc, bh, al, idesc, (w | k) != 0);
                        mma_tf32(acc, bl, ah, idesc, 1u);
                        mma_tf32(acc, bh, ah, idesc, 1u);
                    } else {
                        mma_tf32(acc, al, bh, idesc, (w | k) != 0);
                        mma_tf32(acc, ah, bl, idesc, 1u);
                        mma_tf32(acc, ah, bh, idesc, 1u);
                    }
                }
                mma_commit(&empty[s]);
                if (w == CH - 1 || i == NK - 1) mma_commit(&accfull[buf]);
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
    } else if (CONV && warp >= 6) {
        // ---- split warps (see CONV): lo of each landed fp32 weight tile (an
        // elementwise map, so the tiles' 128-byte swizzle needs no decoding)
        const int ct = threadIdx.x - 192;
        constexpr int NCV = 32 * kConvWarps;
        constexpr int PER = BN * 8 / NCV;  // float4 per thread and tile
        static_assert(BN * 8 % NCV == 0, "whole float4 passes over a tile");
        int s = 0;
        uint32_t ph = 0;  // slot i % S and parity (i / S) & 1, counted
        for (int i = 0; i < NK; ++i) {
            if (!mbar_wait_bounded(&full[s], ph)) {
                s_err = 1;
                break;
            }
            const float4* bh = reinterpret_cast<const float4*>(gbase + (b_hi(s) - base));
            float4* bl = reinterpret_cast<float4*>(gbase + (b_lo(s) - base));
            float4 v[PER];
#pragma unroll
            for (int j = 0; j < PER; ++j) v[j] = bh[ct + NCV * j];
#pragma unroll
            for (int j = 0; j < PER; ++j)
                bl[ct + NCV * j] = make_float4(v[j].x - tf32_trunc(v[j].x), v[j].y - tf32_trunc(v[j].y),
                                               v[j].z - tf32_trunc(v[j].z), v[j].w - tf32_trunc(v[j].w));
            fence_proxy_async_smem();  // the tensor core reads what was just written
            __syncwarp();
            if (lane == 0) mbar_arrive(&convb[s]);
            if (++s == S) {
                s = 0;
                ph ^= 1u;
            }
        }
    } else if constexpr (!DRAIN) {
        // the other warps wait below for the single accumulator; warp 2 first
        // fetches the QKV rows' state (written by earlier kernels)
        if (EPI == GEPI_QKV_ROPE && warp == 2) {
            pdl_wait();
            for (int i = lane; i < 128; i += 32)
                if (m0 + i < m_end) s_rows[i] = load_row_state(g, m0 + i);
        }
        if constexpr (EPI != GEPI_RESIDUAL && EPI != GEPI_STORE) {
            static_assert(gemm_threads(false) == 256, "warps 4-7 load the 128 row scales");
            if (warp >= 4 && g.ss_in != nullptr) {  // ... and warps 4-7 the row scales
                pdl_wait();
                const int i = threadIdx.x - 128;
                if (m0 + i < m_end) s_scale[i] = row_scale(g, m0 + i);
            }
        }
    } else {
        // ---- warps 0-3: drain every chunk into registers (fp32 round-to-nearest adds)
        if (EPI == GEPI_QKV_ROPE && m0 + threadIdx.x < m_end) {
            pdl_wait();
            s_rows[threadIdx.x] = load_row_state(g, m0 + threadIdx.x);
        }
        if constexpr (EPI != GEPI_RESIDUAL && EPI != GEPI_STORE) {
            if (g.ss_in != nullptr && m0 + threadIdx.x < m_end) {
                pdl_wait();
                s_scale[threadIdx.x] = row_scale(g, m0 + threadIdx.x);
            }
        }
        const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
        for (int c = 0; c < NCH; ++c) {
            const int buf = c & 1;
            if (!mbar_wait_bounded(&accfull[buf], static_cast<uint32_t>(c / 2) & 1u)) {
                s_err = 1;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int j = 0; j < RN / 32; ++j) {
                float v[32];
                __syncwarp();  // tcgen05.ld is warp-collective
                tmem_ld32(tmem + lane_base + static_cast<uint32_t>(buf * RN + 32 * j), v);
#pragma unroll
                for (int t = 0; t < 32; ++t) R[32 * j + t] += v[t];
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&accfree[buf]);
        }
    }
    __syncwarp();
    if constexpr (!DRAIN) {
        // ---- all warps: wait for the single accumulator (read in the epilogue)
        if (NK > 0 && !mbar_wait_bounded(&accfull[0], 0u)) s_err = 1;
        tc_fence_after();
    }
    __syncthreads();  // mainloop and drain done; s_err settled; s_rows loaded
    constexpr int NT = gemm_threads(DRAIN, CONV);
    // TMEM readers: warps 0-3 with the drain (all columns, from R); without
    // it every warp, warp w taking chunks w / 4, w / 4 + NT / 128, ...
    constexpr int kHalves = DRAIN ? 1 : NT / 128;
    const int half = DRAIN ? 0 : (warp >> 2);
    const bool reader = DRAIN ? (warp < 4) : true;
    // this reader's tile row: an M = 128 accumulator keeps row i in TMEM lane
    // i; an M = 64 one keeps rows 16 q .. 16 q + 15 in the first 16 lanes of
    // lane quarter q (-1: a lane that holds no row)
    const int TR = g.a_rows == 64 ? 64 : 128;  // rows of the tile
    const int row = TR == 128 ? 32 * (warp & 3) + lane : (lane < 16 ? 16 * (warp & 3) + lane : -1);
    const uint32_t lane_addr = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    auto rstate = [&](int lr) {
        if constexpr (EPI == GEPI_QKV_ROPE) return s_rows[lr];
        return RowState{0, 1, 0};
    };
    auto rscale = [&](int lr) {
        if constexpr (EPI == GEPI_RESIDUAL || EPI == GEPI_STORE) return 1.0f;
        return g.ss_in != nullptr ? s_scale[lr] : 1.0f;
    };
    const int ss_slot = 2 * (n0 / BN);  // this tile's sum-of-squares slots

    if (nsplit == 1 && !SWAP) {
        if (s_err) {
            if (threadIdx.x == 0) atomicOr(g.err, ERR_TIMEOUT_TMA);
        } else if (reader) {
            const int r = m0 + row;
            const bool row_ok = row >= 0 && r < m_end;
            const RowState rs = row_ok ? rstate(row) : RowState{0, 0, 0};
            const float sc = row_ok ? rscale(row) : 1.0f;
            unsigned long long best = 0ull;
            float ssq = 0.0f;  // RESIDUAL producer: sum of squares of this thread's values
            if constexpr (DRAIN) {
                if (row_ok) {
#pragma unroll
                    for (int j = 0; j < RN; j += 4) {  // RN == BN on this path
                        const int gc = n0 + j;
                        if (gc < g.N) {
                            const float a4[4] = {R[j] * sc, R[j + 1] * sc, R[j + 2] * sc,
                                                 R[j + 3] * sc};
                            ssq += epi4<EPI>(g, r, gc, a4, rs, epi_pre<EPI>(g, r, gc, rs), best);
                        }
                    }
                }
            } else {
#pragma unroll 1
                for (int c = half; c < BN / 32; c += kHalves) {
                    float v[32];
                    __syncwarp();  // tcgen05.ld is warp-collective
                    tmem_ld32(tmem + lane_addr + 32 * c, v);
                    const int gc0 = n0 + 32 * c;
                    if (!row_ok || gc0 >= g.N) continue;
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        const float a4[4] = {v[j] * sc, v[j + 1] * sc, v[j + 2] * sc,
                                             v[j + 3] * sc};
                        if (gc0 + j < g.N)
                            ssq += epi4<EPI>(g, r, gc0 + j, a4, rs,
                                             epi_pre<EPI>(g, r, gc0 + j, rs), best);
                    }
                }
            }
            if constexpr (EPI == GEPI_ARGMAX) {
                if (row_ok && best != 0ull) atomicMax(g.argmax_keys + r, best);
            }
            if constexpr (EPI == GEPI_RESIDUAL) {
                if (g.ss_out != nullptr && row_ok) {
                    float* so = g.ss_out + static_cast<size_t>(r) * g.ss_stride + ss_slot;
                    if constexpr (DRAIN) {
                        so[0] = ssq;
                        so[1] = 0.0f;
                    } else {
                        so[half] = ssq;  // kHalves == 2: both slots written
                    }
                }
            }
        }
    } else {
        // stage this CTA's partial tile (row-major, stride PS) in the ring
        float* P = reinterpret_cast<float*>(gbase);
        if (reader) {
            if constexpr (SWAP) {
                // this thread's weight row is column n of the row-major tile
                const int n = 32 * (warp & 3) + lane;
#pragma unroll
                for (int t = 0; t < 64; ++t) P[t * PS + n] = R[t];
            } else if constexpr (DRAIN) {
                if (row >= 0) {
#pragma unroll
                    for (int j = 0; j < BN; j += 4)
                        *reinterpret_cast<float4*>(P + row * PS + j) =
                            make_float4(R[j], R[j + 1], R[j + 2], R[j + 3]);
                }
            } else {
#pragma unroll 1
                for (int c = half; c < BN / 32; c += kHalves) {
                    float v[32];
                    __syncwarp();
                    tmem_ld32(tmem + lane_addr + 32 * c, v);
                    if (NK == 0) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = 0.0f;
                    }
                    if (row < 0) continue;
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4*>(P + row * PS + 32 * c + j) =
                            make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                }
            }
            fence_proxy_async_smem();
        }
        __syncthreads();
        if (nsplit > 1) cluster_wait_acquire();  // every peer's barriers are initialised
        const int R_ = (TR + nsplit - 1) / nsplit;  // rows of a receive slot
        const int r0 = TR * split / nsplit, r1 = TR * (split + 1) / nsplit;
        const uint32_t pbase = smem_u32(P);
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(recvb, static_cast<uint32_t>((nsplit - 1) * (r1 - r0) * PS * 4));
            // push rows [TR q/S, TR (q+1)/S) of this partial to their owner q
            for (int q = 0; q < nsplit; ++q) {
                if (q == split) continue;
                const int q0 = TR * q / nsplit, q1 = TR * (q + 1) / nsplit;
                const int slot = split < q ? split : split - 1;  // slot of this sender at q
                bulk_s2peer(map_peer(recv_base + static_cast<uint32_t>(slot * R_ * PS * 4), q),
                            pbase + static_cast<uint32_t>(q0 * PS * 4),
                            static_cast<uint32_t>((q1 - q0) * PS * 4), map_peer(smem_u32(recvb), q));
            }
        }
        {
            const int gpr = BN / 4;  // float4 groups per row
            const int ngroups = (r1 - r0) * gpr;
            const float* recv =
                reinterpret_cast<const float*>(gbase + static_cast<size_t>(S) * stage_b);
            // Each thread takes its groups kU at a time: group t is row r0 + t / gpr,
            // columns 4 (t % gpr) .. + 3 of the tile. The global operands of a batch
            // are requested first (for the first batch, while the slices travel),
            // then all its partial-sum loads, then the epilogue math and stores, so
            // a batch has kU * S loads in flight rather than one chain per group.
            constexpr int kU = 4;
            int t0 = threadIdx.x;
            bool ok[kU];
            int lrs[kU];
            EpiPre pre[kU];
            auto fetch = [&](int tb) {
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int t = tb + NT * u;
                    lrs[u] = r0 + t / gpr;
                    const int r = m0 + lrs[u], gc = n0 + 4 * (t % gpr);
                    ok[u] = t < ngroups && r < m_end && gc < g.N;
                    pre[u] = ok[u] ? epi_pre<EPI>(g, r, gc, rstate(lrs[u])) : EpiPre{};
                }
            };
            fetch(t0);
            const bool got = mbar_wait_bounded(recvb, 0u);
            if (!got) s_err = 1;
            if (!s_err) {
                // warp-uniform trip count (the sum-of-squares reduction shuffles)
                for (; t0 - lane < ngroups; t0 += kU * NT) {
                    float4 acc[kU];
#pragma unroll
                    for (int u = 0; u < kU; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                    // the S partials in rank order (a fixed order, whoever arrived first)
                    for (int q = 0; q < nsplit; ++q) {
#pragma unroll
                        for (int u = 0; u < kU; ++u) {
                            if (!ok[u]) continue;
                            const int c4 = (t0 + NT * u) % gpr;
                            const float* src =
                                (q == split)
                                    ? P + lrs[u] * PS
                                    : recv + static_cast<size_t>((q < split ? q : q - 1) * R_ +
                                                                 (lrs[u] - r0)) * PS;
                            const float4 v = *reinterpret_cast<const float4*>(src + 4 * c4);
                            acc[u].x += v.x;
                            acc[u].y += v.y;
                            acc[u].z += v.z;
                            acc[u].w += v.w;
                        }
                    }
#pragma unroll
                    for (int u = 0; u < kU; ++u) {
                        const int t = t0 + NT * u;
                        const int r = m0 + lrs[u], gc = n0 + 4 * (t % gpr);
                        float sq = 0.0f;
                        if (ok[u]) {
                            unsigned long long best = 0ull;
                            const float sc = rscale(lrs[u]);
                            const float a4[4] = {acc[u].x * sc, acc[u].y * sc, acc[u].z * sc,
                                                 acc[u].w * sc};
                            sq = epi4<EPI>(g, r, gc, a4, rstate(lrs[u]), pre[u], best);
                            if constexpr (EPI == GEPI_ARGMAX) {
                                if (best != 0ull) atomicMax(g.argmax_keys + r, best);
                            }
                        }
                        if constexpr (EPI == GEPI_RESIDUAL) {
                            if (g.ss_out != nullptr) {
                                // the gpr lanes of a row (gpr divides 32) add their
                                // squares in a fixed shuffle tree
                                for (int o = gpr / 2; o > 0; o >>= 1)
                                    sq += __shfl_xor_sync(0xffffffffu, sq, o);
                                if (ok[u] && t % gpr == 0) {
                                    float* so = g.ss_out + static_cast<size_t>(r) * g.ss_stride +
                                                ss_slot;
                                    so[0] = sq;
                                    so[1] = 0.0f;
                                }
                            }
                        }
                    }
                    if (t0 + kU * NT < ngroups) fetch(t0 + kU * NT);
                }
            } else if (threadIdx.x == 0) {
                atomicOr(g.err, ERR_TIMEOUT_TMA);
            }
            if (threadIdx.x == 0) bulk_commit_and_wait_read();  // this CTA's pushes have read P
        }
    }

    // ---- teardown: every tcgen05 access of this CTA is complete
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, C::tmem_cols(DRAIN));
}

__global__ void split_tf32_kernel(const float4* __restrict__ x, float4* __restrict__ hi,
                                  float4* __restrict__ lo, long long n4) {
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n4;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const float4 v = x[i];
        float4 h;
        h.x = tf32_round(v.x);
        h.y = tf32_round(v.y);
        h.z = tf32_round(v.z);
        h.w = tf32_round(v.w);
        hi[i] = h;
        // lo rounded to tf32 as well: the tensor core would otherwise truncate it
        lo[i] = make_float4(tf32_round(v.x - h.x), tf32_round(v.y - h.y), tf32_round(v.z - h.z),
                            tf32_round(v.w - h.w));
    }
}

__global__ void split_tf32_gain_kernel(const float* __restrict__ x, const float* __restrict__ gain,
                                       long long K, long long rows, long long n,
                                       float* __restrict__ hi, float* __restrict__ lo) {
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long k = i % K, layer = i / (K * rows);
        const float v = x[i] * gain[layer * K + k];
        const float h = tf32_round(v);
        hi[i] = h;
        lo[i] = tf32_round(v - h);
    }
}

// ------------------------------------------------------------- host side

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

template <int BN, int EPI, bool DRAIN, bool CONV = false>
cudaError_t launch_t(const GemmMaps& m, const GemmArgs& g, int ksplit, cudaStream_t s, bool pdl) {
    using C = Cfg<BN>;
    cudaLaunchConfig_t cfg{};
    const int mt = (g.M + 127) / 128, nt = (g.N + BN - 1) / BN;
    cfg.gridDim = dim3(ksplit, mt * nt);
    cfg.blockDim = dim3(gemm_threads(DRAIN, CONV));
    cfg.dynamicSmemBytes = C::smem_for(g.stages, ksplit, g.a_rows == 64 ? 64 : 128);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ksplit;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    // CONV: the weight map is the fp32 array's (the lo map is not read)
    return cudaLaunchKernelEx(&cfg, gemm_tf32x3_kernel<BN, EPI, DRAIN, CONV>, m.a_hi, m.a_lo,
                              CONV ? m.b_raw : m.b_hi, m.b_lo, g);
}

// Tiles wider than 128 columns have no drained variant (its register copy of
// the tile row would not fit): they serve only K ranges of at most
// kDrainAbove K-blocks per CTA.
template <int BN>
constexpr bool has_drain() { return BN <= 128; }

template <int BN, int EPI>
cudaError_t set_smem() {
    cudaError_t e = cudaFuncSetAttribute(gemm_tf32x3_kernel<BN, EPI, false, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kMaxDynSmem));
    if (e != cudaSuccess) return e;
    if constexpr (has_drain<BN>()) {
        e = cudaFuncSetAttribute(gemm_tf32x3_kernel<BN, EPI, true, false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kMaxDynSmem));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(gemm_tf32x3_kernel<BN, EPI, true, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kMaxDynSmem));
    }
    return e;
}

template <int BN>
cudaError_t set_smem_bn() {
    cudaError_t e;
    if ((e = set_smem<BN, GEPI_STORE>()) != cudaSuccess) return e;
    if ((e = set_smem<BN, GEPI_RESIDUAL>()) != cudaSuccess) return e;
    if ((e = set_smem<BN, GEPI_SWIGLU>()) != cudaSuccess) return e;
    if ((e = set_smem<BN, GEPI_QKV_ROPE>()) != cudaSuccess) return e;
    return set_smem<BN, GEPI_ARGMAX>();
}

template <int BN, bool DRAIN, bool CONV = false>
cudaError_t launch_bd(int epi, const GemmMaps& m, const GemmArgs& g, int ks, cudaStream_t s,
                      bool pdl) {
    switch (epi) {
        case GEPI_STORE: return launch_t<BN, GEPI_STORE, DRAIN, CONV>(m, g, ks, s, pdl);
        case GEPI_RESIDUAL: return launch_t<BN, GEPI_RESIDUAL, DRAIN, CONV>(m, g, ks, s, pdl);
        case GEPI_SWIGLU: return launch_t<BN, GEPI_SWIGLU, DRAIN, CONV>(m, g, ks, s, pdl);
        case GEPI_QKV_ROPE: return launch_t<BN, GEPI_QKV_ROPE, DRAIN, CONV>(m, g, ks, s, pdl);
        case GEPI_ARGMAX: return launch_t<BN, GEPI_ARGMAX, DRAIN, CONV>(m, g, ks, s, pdl);
        default: return cudaErrorInvalidValue;
    }
}

// The drained variant when some CTA's share of K exceeds kDrainAbove K-blocks.
template <int BN>
cudaError_t launch_bn(int epi, const GemmMaps& m, const GemmArgs& g, int ks, cudaStream_t s,
                      bool pdl) {
    const int KB = (g.K + 31) / 32;
    const int per_cta = (KB + ks - 1) / ks;
    if (per_cta > kDrainAbove) {
        if constexpr (has_drain<BN>()) {
            if (g.conv && g.a_rows != 64) return cudaErrorInvalidValue;  // tiles of <= 64 rows
            if (g.conv) return launch_bd<BN, true, true>(epi, m, g, ks, s, pdl);
            return launch_bd<BN, true>(epi, m, g, ks, s, pdl);
        }
        return cudaErrorInvalidValue;
    }
    // a handle that kept no tf32 pair for this GEMM plans only drained launches
    if (g.conv) return cudaErrorInvalidValue;
    return launch_bd<BN, false>(epi, m, g, ks, s, pdl);
}

}  // namespace

// Tensor map of a fp32 array [layers][rows][inner] (inner contiguous) read in
// boxes of 32 x box_rows x 1 with the 128-byte swizzle; out-of-range
// elements read as zero.
cudaError_t make_gemm_map(CUtensorMap* map, const float* base, long long inner, long long rows,
                          long long layers, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0 || inner % 4 != 0 || box_rows < 1 ||
        box_rows > 256)
        return cudaErrorInvalidValue;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(layers)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner) * 4,
                                   static_cast<cuuint64_t>(inner) * rows * 4};
    const cuuint32_t box[3] = {32, static_cast<cuuint32_t>(box_rows), 1};
    const cuuint32_t es[3] = {1, 1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims,
                          strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Deepest ring of a tile width: 2-4 slots with 128-row A tiles; with 64-row A
// tiles the smaller slots allow up to Cfg::MAX_STAGES.
template <int BN>
int ring_limit(int a_rows) { return a_rows == 64 ? Cfg<BN>::MAX_STAGES : Cfg<BN>::STAGES; }

// Whether a ring of `stages` slots (and the receive buffer of a split launch)
// fits in one CTA's shared memory.
template <int BN>
bool fits(int stages, int ksplit, int a_rows) {
    return stages <= ring_limit<BN>(a_rows) &&
           Cfg<BN>::smem_for(stages, ksplit, a_rows) <= kMaxDynSmem;
}

template <int BN>
int active_clusters(int ksplit, int stages, int a_rows) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(ksplit, 1024);
    cfg.blockDim = dim3(gemm_threads(has_drain<BN>()));
    cfg.dynamicSmemBytes = Cfg<BN>::smem_for(stages, ksplit, a_rows);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ksplit;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(
            &n, gemm_tf32x3_kernel<BN, GEPI_QKV_ROPE, has_drain<BN>(), false>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

// Raises the dynamic shared-memory limit of every GEMM instantiation on the
// current device and measures how many clusters of each launch shape run at
// once (call before the first launch and outside stream capture).
cudaError_t prepare_gemm(GemmOccupancy* occ) {
    cudaError_t e = set_smem_bn<64>();
    if (e == cudaSuccess) e = set_smem_bn<128>();
    if (e == cudaSuccess) e = set_smem_bn<256>();
    if (e != cudaSuccess || occ == nullptr) return e;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&occ->num_sms, cudaDevAttrMultiProcessorCount, dev)) !=
        cudaSuccess)
        return e;
    for (int ar = 0; ar < 2; ++ar) {
        const int a_rows = ar == 0 ? 128 : 64;
        for (int sp = 1; sp <= 8; ++sp)
            for (int st = 2; st <= 6; ++st) {
                occ->clusters[ar][0][sp][st] = fits<64>(st, sp, a_rows) ? active_clusters<64>(sp, st, a_rows) : 0;
                occ->clusters[ar][1][sp][st] = fits<128>(st, sp, a_rows) ? active_clusters<128>(sp, st, a_rows) : 0;
                occ->clusters[ar][2][sp][st] = fits<256>(st, sp, a_rows) ? active_clusters<256>(sp, st, a_rows) : 0;
            }
    }
    return cudaSuccess;
}

// The ring depth, whether a ring fits, and the occupancy table row of a tile width.
int max_stages(int bn, int a_rows) {
    return bn == 256 ? ring_limit<256>(a_rows) : bn == 128 ? ring_limit<128>(a_rows)
                                                           : ring_limit<64>(a_rows);
}
bool fits_bn(int bn, int stages, int ksplit, int a_rows) {
    return bn == 256 ? fits<256>(stages, ksplit, a_rows)
           : bn == 128 ? fits<128>(stages, ksplit, a_rows)
                       : fits<64>(stages, ksplit, a_rows);
}
int bn_row(int bn) { return bn == 256 ? 2 : bn == 128 ? 1 : 0; }
int stage_bytes_bn(int bn, int a_rows) { return 2 * a_rows * 32 * 4 + 2 * bn * 32 * 4; }

// Estimated time of a plan, in bytes one CTA streams: every wave of
// co-resident clusters takes the per-CTA K range times a slot's bytes, plus
// the split-K exchange (about three slots' worth); waves are counted whole.
// Used for GEMMs of at most 64 rows, whose long K ranges make the kernel a
// weight stream: a plan that leaves SMs idle in a partial last wave, or one
// wave on two thirds of the SMs, loses to a deeper split in balanced waves.
long long plan_cost(const GemmOccupancy& occ, int bn, int sp, int st, int tiles, int KB,
                    int a_rows) {
    const int cl = occ.clusters[a_rows == 64 ? 1 : 0][bn_row(bn)][sp][st];
    if (cl < 1) return -1;
    const long long waves = (tiles + cl - 1) / cl;
    const long long kb = (KB + sp - 1) / sp;
    const long long slot = stage_bytes_bn(bn, a_rows);
    return waves * (kb * slot + (sp > 1 ? 3 * slot : 0));
}

// ksplit == 0 in the result: no plan with this tile width (a 256-wide tile
// needs a split that leaves each CTA at most kDrainAbove K-blocks and fits).
//
// 128-row A tiles (decode rows): the largest split S <= 8 that keeps at
// least two K-blocks per CTA and runs every cluster in one wave; the ring
// holds one CTA's K-blocks, at least 2 and at most what fits. (Measured on
// the batched decode GEMMs: two co-resident CTAs per SM with 2-slot rings are
// no faster than one CTA per SM with a deeper ring.)
// 64-row A tiles (prefill passes of at most 64 rows): the split of least
// plan_cost, the ring as deep as fits.
GemmPlan plan_split(const GemmOccupancy& occ, int bn, int M, int N, int K, int a_rows) {
    const int KB = (K + 31) / 32, mt = (M + 127) / 128;
    const int tiles = mt * ((N + bn - 1) / bn);
    const int max_st = max_stages(bn, a_rows);
    const bool drainable = bn <= 128;
    auto depth = [&](int sp) {
        const int per = (KB + sp - 1) / sp;
        int st = per < 2 ? 2 : per > max_st ? max_st : per;
        while (st > 2 && !fits_bn(bn, st, sp, a_rows)) --st;
        return st;
    };
    auto ok = [&](int sp) { return drainable || (KB + sp - 1) / sp <= kDrainAbove; };
    if (a_rows == 64) {
        GemmPlan best{bn, 0, 2};
        long long best_cost = -1;
        for (int sp = 1; sp <= 8; ++sp) {
            if ((sp > 1 && KB / sp < 2) || !ok(sp)) continue;
            const int st = depth(sp);
            if (!fits_bn(bn, st, sp, a_rows)) continue;
            const long long c = plan_cost(occ, bn, sp, st, tiles, KB, a_rows);
            if (c >= 0 && (best_cost < 0 || c < best_cost)) {
                best_cost = c;
                best = GemmPlan{bn, sp, st};
            }
        }
        return best;
    }
    for (int sp = 8; sp > 1; --sp) {
        if (KB / sp < 2 || !ok(sp)) continue;
        const int st = depth(sp);
        if (fits_bn(bn, st, sp, a_rows) && tiles <= occ.clusters[0][bn_row(bn)][sp][st])
            return GemmPlan{bn, sp, st};
    }
    if (!ok(1) || !fits_bn(bn, depth(1), 1, a_rows)) return GemmPlan{bn, 0, 2};
    return GemmPlan{bn, 1, depth(1)};
}

// Tile width and split of an M x N x K GEMM. 128-row A tiles: the plan that
// keeps more SMs busy in its first wave wins, ties going to the wider tile
// (fewer activation re-reads, and fewer waves when the tiles outnumber the
// SMs: the 256 x 32000 classifier runs 250 tiles of 256 columns in two rounds
// instead of 500 of 128 in four). 64-row A tiles: the plan of least
// plan_cost. max_bn caps the width (a GEMM whose epilogue produces per-row
// sums of squares needs a tile row within one warp: 128).
GemmPlan plan_gemm(const GemmOccupancy& occ, int M, int N, int K, int max_bn, int a_rows) {
    GemmPlan best{64, 1, Cfg<64>::STAGES};
    long long best_score = -1;
    const int mt = (M + 127) / 128, KB = (K + 31) / 32;
    for (int bn : {256, 128, 64}) {
        if (bn > max_bn || (bn > 64 && bn > N)) continue;  // a tile wider than N is waste
        const GemmPlan p = plan_split(occ, bn, M, N, K, a_rows);
        if (p.ksplit < 1) continue;
        const int tiles = mt * ((N + bn - 1) / bn);
        if (a_rows == 64) {
            const long long c = plan_cost(occ, bn, p.ksplit, p.stages, tiles, KB, a_rows);
            if (c >= 0 && (best_score < 0 || c < best_score)) {
                best_score = c;
                best = p;
            }
            continue;
        }
        long long ctas = static_cast<long long>(tiles) * p.ksplit;
        if (ctas > occ.num_sms) ctas = occ.num_sms;
        if (ctas > best_score) {
            best_score = ctas;
            best = p;
        }
    }
    return best;
}

cudaError_t launch_gemm(int epi, const GemmPlan& p, const GemmMaps& m, const GemmArgs& g0,
                        cudaStream_t s, bool pdl) {
    const int a_rows = g0.a_rows == 64 ? 64 : 128;
    if (a_rows == 64 && g0.M > 64) return cudaErrorInvalidValue;  // one 64-row A tile per launch
    const int max_st = max_stages(p.bn, a_rows);
    if (g0.M < 1 || g0.N < 1 || g0.K < 4 || g0.K % 4 != 0 || p.ksplit < 1 || p.ksplit > 8 ||
        p.stages < 2 || p.stages > max_st)
        return cudaErrorInvalidValue;
    // a sum-of-squares producer needs a tile row within one warp (gpr <= 32)
    // and room for two slots per N tile
    if (g0.ss_out != nullptr &&
        (p.bn > 128 || 2 * ((g0.N + p.bn - 1) / p.bn) > g0.ss_stride || epi != GEPI_RESIDUAL))
        return cudaErrorInvalidValue;
    GemmArgs g = g0;
    g.stages = p.stages;
    g.a_rows = a_rows;
    if (p.bn == 256) return launch_bn<256>(epi, m, g, p.ksplit, s, pdl);
    if (p.bn == 128) return launch_bn<128>(epi, m, g, p.ksplit, s, pdl);
    if (p.bn == 64) return launch_bn<64>(epi, m, g, p.ksplit, s, pdl);
    return cudaErrorInvalidValue;
}

cudaError_t launch_split_tf32_gain(const float* x, const float* gain, long long K, long long rows,
                                   long long layers, float* hi, float* lo, cudaStream_t s) {
    if (K < 1 || rows < 1 || layers < 1) return cudaErrorInvalidValue;
    const long long n = K * rows * layers;
    const int blocks = static_cast<int>(n / 256 + 1 < 8192 ? n / 256 + 1 : 8192);
    split_tf32_gain_kernel<<<blocks, 256, 0, s>>>(x, gain, K, rows, n, hi, lo);
    return cudaGetLastError();
}

__global__ void scale_gain_kernel(const float* __restrict__ x, const float* __restrict__ gain,
                                  long long K, long long rows, long long n, float* __restrict__ out) {
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long k = i % K, layer = i / (K * rows);
        out[i] = x[i] * gain[layer * K + k];  // the product the pair split starts from
    }
}

cudaError_t launch_scale_gain(const float* x, const float* gain, long long K, long long rows,
                              long long layers, float* out, cudaStream_t s) {
    if (K < 1 || rows < 1 || layers < 1) return cudaErrorInvalidValue;
    const long long n = K * rows * layers;
    const int blocks = static_cast<int>(n / 256 + 1 < 8192 ? n / 256 + 1 : 8192);
    scale_gain_kernel<<<blocks, 256, 0, s>>>(x, gain, K, rows, n, out);
    return cudaGetLastError();
}

bool gemm_drained(const GemmPlan& p, int K) {
    const int KB = (K + 31) / 32;
    return p.ksplit >= 1 && p.bn <= 128 && (KB + p.ksplit - 1) / p.ksplit > kDrainAbove;
}

cudaError_t launch_split_tf32(const float* x, float* hi, float* lo, long long n, cudaStream_t s) {
    if (n % 4 != 0) return cudaErrorInvalidValue;
    const long long n4 = n / 4;
    const int blocks = static_cast<int>(n4 / 256 + 1 < 8192 ? n4 / 256 + 1 : 8192);
    split_tf32_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<const float4*>(x),
                                             reinterpret_cast<float4*>(hi),
                                             reinterpret_cast<float4*>(lo), n4);
    return cudaGetLastError();
}

}  // namespace l2

// ------------------------------------------------------------- test / measurement hook

extern "C" int l2_gemm_tf32x3(const float* d_A, const float* d_W, float* d_C, int32_t M,
                              int32_t N, int32_t K, int32_t iters, float* ms, void* stream) {
    using namespace l2;
    if (!d_A || !d_W || !d_C || M < 1 || N < 1 || K < 4 || K % 4 != 0 || iters < 0 ||
        (iters > 0 && !ms))
        return L2_EINVAL;
    if ((reinterpret_cast<uintptr_t>(d_A) | reinterpret_cast<uintptr_t>(d_W) |
         reinterpret_cast<uintptr_t>(d_C)) & 15u)
        return L2_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t na = static_cast<size_t>(M) * K, nw = static_cast<size_t>(N) * K;
    const size_t na_pad = (na + 63) & ~static_cast<size_t>(63);
    const size_t nw_pad = (nw + 63) & ~static_cast<size_t>(63);
    float* buf = nullptr;
    cudaError_t e = cudaMalloc(&buf, (2 * na_pad + 2 * nw_pad) * sizeof(float) + 256);
    if (e != cudaSuccess) return e == cudaErrorMemoryAllocation ? L2_ENOMEM : L2_ECUDA;
    float *a_hi = buf, *a_lo = buf + na_pad, *w_hi = a_lo + na_pad, *w_lo = w_hi + nw_pad;
    int* d_err = reinterpret_cast<int*>(w_lo + nw_pad);
    int rc = L2_OK;
    GemmOccupancy occ{};
    if (prepare_gemm(&occ) != cudaSuccess) return L2_ECUDA;
    const GemmPlan plan = plan_gemm(occ, M, N, K);
    const int bn = plan.bn;
    GemmMaps maps;
    GemmArgs g{};
    g.M = M;
    g.N = N;
    g.K = K;
    g.ldc = N;
    g.out = d_C;
    g.err = d_err;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    do {
        if ((e = cudaMemsetAsync(d_err, 0, sizeof(int), s)) != cudaSuccess) break;
        if ((e = launch_split_tf32(d_A, a_hi, a_lo, static_cast<long long>(na), s)) != cudaSuccess)
            break;
        if ((e = launch_split_tf32(d_W, w_hi, w_lo, static_cast<long long>(nw), s)) != cudaSuccess)
            break;
        if ((e = make_gemm_map(&maps.a_hi, a_hi, K, M, 1, 128)) != cudaSuccess) break;
        if ((e = make_gemm_map(&maps.a_lo, a_lo, K, M, 1, 128)) != cudaSuccess) break;
        if ((e = make_gemm_map(&maps.b_hi, w_hi, K, N, 1, bn)) != cudaSuccess) break;
        if ((e = make_gemm_map(&maps.b_lo, w_lo, K, N, 1, bn)) != cudaSuccess) break;
        if ((e = launch_gemm(GEPI_STORE, plan, maps, g, s, false)) != cudaSuccess) break;
        if (iters > 0) {
            if ((e = cudaEventCreate(&e0)) != cudaSuccess) break;
            if ((e = cudaEventCreate(&e1)) != cudaSuccess) break;
            if ((e = cudaEventRecord(e0, s)) != cudaSuccess) break;
            for (int i = 0; i < iters && e == cudaSuccess; ++i)
                e = launch_gemm(GEPI_STORE, plan, maps, g, s, false);
            if (e != cudaSuccess) break;
            if ((e = cudaEventRecord(e1, s)) != cudaSuccess) break;
        }
        if ((e = cudaStreamSynchronize(s)) != cudaSuccess) break;
        if (iters > 0) {
            float t = 0.0f;
            if ((e = cudaEventElapsedTime(&t, e0, e1)) != cudaSuccess) break;
            *ms = t / iters;
        }
        int err = 0;
        if ((e = cudaMemcpy(&err, d_err, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess) break;
        if (err) rc = L2_ETIMEOUT;
    } while (0);
    if (e != cudaSuccess) rc = (e == cudaErrorInvalidValue) ? L2_EINVAL : L2_ECUDA;
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    cudaFree(buf);
    return rc;
}
