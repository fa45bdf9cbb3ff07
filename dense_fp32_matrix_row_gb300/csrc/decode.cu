// decode.cu -- SGEMM for M <= 16 rows (the decode regime).
//
// With M = batch the product is a matrix-vector-like pass that is bound by
// reading B once from HBM ("GPU GEMM 优化完全拆解（一）", section "LLM 推理本质上是
// GEMM 的串联": decode is memory-bound).  The kernel streams B with 128-bit
// loads that do not allocate in L1, keeps the few rows of A in shared memory,
// and splits K across the blocks of a thread-block cluster, the split-K idea
// of "CUDA 矩阵乘法优化：从朴素 Kernel 到接近 cuBLAS", section "10" -- but the
// partial sums are combined on chip instead of by a second reduction kernel:
//
//  * grid: (KS, ceil(N/128)); a cluster of KS blocks shares one 128-column
//    slice of B and C, block `rank` of the cluster takes rows
//    [rank*kslice, (rank+1)*kslice) of B;
//  * each lane owns 4 consecutive columns and MT accumulators per column; the
//    8 warps of a block take interleaved rows of the block's K range, so one
//    step of the block reads an 8x128 panel of B;
//  * partials are summed across warps through shared memory, then across the
//    cluster through distributed shared memory; both sums run in a fixed
//    order, so results do not depend on timing;
//  * block `rank` finishes outputs [rank*per, (rank+1)*per) of the 128*MT the
//    cluster owns and applies C = alpha*sum + beta*C (C read only if beta != 0).
#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace sgemm_gb300 {
namespace {

constexpr int DTHREADS = 256;
constexpr int DWARPS = DTHREADS / 32;
constexpr int DCOLS = 128;      // columns per cluster (32 lanes x 4)
constexpr int KCH = 512;        // rows of A staged in shared memory at a time
constexpr int UNROLL = 8;       // independent 128-bit B loads in flight per lane

template <int MT>
constexpr size_t decode_smem_bytes() {
    constexpr size_t stage = (size_t)KCH * MT * 4;
    constexpr size_t red = (size_t)DWARPS * MT * DCOLS * 4;
    return (stage > red ? stage : red) + (size_t)MT * DCOLS * 4;
}

// B[k, n0 .. n0+3] for one lane; columns >= N read as 0.
template <bool VEC>
__device__ __forceinline__ float4 load_b4(const float *__restrict__ brow, int64_t col, int64_t N,
                                          bool full4) {
    if (VEC && full4) return ldg_stream_f4(brow + col);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (col + 0 < N) v.x = ldg_stream_f1(brow + col + 0);
    if (col + 1 < N) v.y = ldg_stream_f1(brow + col + 1);
    if (col + 2 < N) v.z = ldg_stream_f1(brow + col + 2);
    if (col + 3 < N) v.w = ldg_stream_f1(brow + col + 3);
    return v;
}

template <int MT>
__device__ __forceinline__ void fma_row(float (&acc)[MT][4], const float *__restrict__ a,
                                        const float4 &b) {
    if constexpr (MT >= 4) {
#pragma unroll
        for (int m4 = 0; m4 < MT / 4; ++m4) {
            const float4 av = *reinterpret_cast<const float4 *>(a + 4 * m4);
            const float am[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float(&r)[4] = acc[4 * m4 + q];
                r[0] = fmaf(am[q], b.x, r[0]);
                r[1] = fmaf(am[q], b.y, r[1]);
                r[2] = fmaf(am[q], b.z, r[2]);
                r[3] = fmaf(am[q], b.w, r[3]);
            }
        }
    } else {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const float am = a[m];
            acc[m][0] = fmaf(am, b.x, acc[m][0]);
            acc[m][1] = fmaf(am, b.y, acc[m][1]);
            acc[m][2] = fmaf(am, b.z, acc[m][2]);
            acc[m][3] = fmaf(am, b.w, acc[m][3]);
        }
    }
}

template <int MT, bool VEC>
__global__ void __launch_bounds__(DTHREADS)
decode_kernel(int M, int64_t N, int64_t K, float alpha, const float *__restrict__ A, int64_t lda,
              const float *__restrict__ B, int64_t ldb, float beta, float *__restrict__ C,
              int64_t ldc, int64_t kslice) {
    extern __shared__ float4 smem4[];
    float *smem = reinterpret_cast<float *>(smem4);
    constexpr size_t STAGE_FLOATS = (size_t)KCH * MT;
    constexpr size_t RED_FLOATS = (size_t)DWARPS * MT * DCOLS;
    float *As = smem;                                   // [KCH][MT], A transposed
    float *red = smem;                                  // [DWARPS][MT][DCOLS], after the K loop
    float *part = smem + (STAGE_FLOATS > RED_FLOATS ? STAGE_FLOATS : RED_FLOATS);  // [MT][DCOLS]

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int ks = (int)cluster.num_blocks();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t n0 = (int64_t)blockIdx.y * DCOLS;
    const int64_t col = n0 + lane * 4;
    const bool full4 = col + 3 < N;
    const int64_t kbeg = (int64_t)rank * kslice;
    const int64_t kend = (kbeg + kslice < K) ? kbeg + kslice : K;

    float acc[MT][4];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.0f;

    for (int64_t kc0 = kbeg; kc0 < kend; kc0 += KCH) {
        const int klen = (int)((kend - kc0) < KCH ? (kend - kc0) : KCH);
        __syncthreads();   // readers of the previous chunk are done
        // Stage A[0..MT)[kc0 .. kc0+klen) as As[k][m]; coalesced along k.
        for (int idx = threadIdx.x; idx < klen * MT; idx += DTHREADS) {
            const int m = idx / klen, kl = idx - m * klen;
            As[kl * MT + m] = (m < M) ? A[(int64_t)m * lda + kc0 + kl] : 0.0f;
        }
        __syncthreads();
        if (col < N) {
            int kl = warp;
            for (; kl + DWARPS * (UNROLL - 1) < klen; kl += DWARPS * UNROLL) {
                float4 b[UNROLL];
#pragma unroll
                for (int u = 0; u < UNROLL; ++u)
                    b[u] = load_b4<VEC>(B + (kc0 + kl + DWARPS * u) * ldb, col, N, full4);
#pragma unroll
                for (int u = 0; u < UNROLL; ++u) fma_row<MT>(acc, As + (kl + DWARPS * u) * MT, b[u]);
            }
            for (; kl < klen; kl += DWARPS) {
                const float4 b = load_b4<VEC>(B + (kc0 + kl) * ldb, col, N, full4);
                fma_row<MT>(acc, As + kl * MT, b);
            }
        }
    }

    // Sum over warps in a fixed order.
    __syncthreads();   // As is no longer read; its space becomes `red`
#pragma unroll
    for (int m = 0; m < MT; ++m)
        *reinterpret_cast<float4 *>(&red[((size_t)warp * MT + m) * DCOLS + lane * 4]) =
            make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
    __syncthreads();
    for (int o = threadIdx.x; o < MT * DCOLS; o += DTHREADS) {
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < DWARPS; ++w) s += red[(size_t)w * MT * DCOLS + o];
        part[o] = s;
    }

    // Sum over the cluster's blocks in rank order, each block finishing a share.
    cluster.sync();
    const int per = (MT * DCOLS + ks - 1) / ks;
    const int obeg = rank * per;
    const int oend = (obeg + per < MT * DCOLS) ? obeg + per : MT * DCOLS;
    for (int o = obeg + threadIdx.x; o < oend; o += DTHREADS) {
        float s = 0.0f;
        for (int q = 0; q < ks; ++q) s += cluster.map_shared_rank(part, q)[o];
        const int m = o / DCOLS;
        const int64_t gn = n0 + (o - m * DCOLS);
        if (m < M && gn < N) {
            float *p = C + (int64_t)m * ldc + gn;
            const float v = alpha * s;
            *p = (beta != 0.0f) ? fmaf(beta, *p, v) : v;
        }
    }
    cluster.sync();   // keep this block's `part` alive until every peer has read it
}

template <int MT, bool VEC>
cudaError_t launch_mt(const GemmArgs &g) {
    constexpr size_t smem = decode_smem_bytes<MT>();
    auto kern = decode_kernel<MT, VEC>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // Split K over up to 8 blocks (a portable cluster), at least 64 rows each.
    int ks = (int)(g.K / 64);
    ks = ks < 1 ? 1 : (ks > 8 ? 8 : ks);
    const int64_t kslice = (g.K + ks - 1) / ks;
    const int64_t ncb = (g.N + DCOLS - 1) / DCOLS;
    if (ncb > 65535) return cudaErrorInvalidConfiguration;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ks, (unsigned)ncb, 1);
    cfg.blockDim = dim3(DTHREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = g.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, (int)g.M, (int64_t)g.N, (int64_t)g.K, g.alpha, g.A,
                              g.lda, g.B, g.ldb, g.beta, g.C, g.ldc, kslice);
}

template <int MT>
cudaError_t launch_vec(const GemmArgs &g) {
    const bool vec = ((reinterpret_cast<uintptr_t>(g.B) & 15) == 0) && (g.ldb % 4 == 0);
    return vec ? launch_mt<MT, true>(g) : launch_mt<MT, false>(g);
}

}  // namespace

cudaError_t launch_decode(const GemmArgs &g) {
    if (g.M <= 1) return launch_vec<1>(g);
    if (g.M <= 2) return launch_vec<2>(g);
    if (g.M <= 4) return launch_vec<4>(g);
    if (g.M <= 8) return launch_vec<8>(g);
    if (g.M <= 16) return launch_vec<16>(g);
    return cudaErrorInvalidValue;
}

}  // namespace sgemm_gb300
