// ffma_generic.cu -- the SGEMM kernel for operands the TMA path cannot take
// (pointers not 16-byte aligned, or a leading dimension not a multiple of 4),
// plus the C <- act(beta*C + bias) kernel used when K == 0 or alpha == 0.
//
// Method: shared-memory cache blocking with a per-thread register tile, as in
// "CUDA 矩阵乘法优化：从朴素 Kernel 到接近 cuBLAS", sections "3. Kernel 3"
// (stage a BMxBK slice of A and a BKxBN slice of B, synchronise, accumulate)
// and "6. Kernel 5" (each thread owns a TMxTN block of outputs and forms a
// register outer product per k).  Out-of-range tile elements are loaded as
// zero so the arithmetic loop has no branches ("GPU 基础原理", section 4.7,
// tile quantization), and the stores are guarded.
#include "common.cuh"

namespace sgemm_gb300 {
namespace {

constexpr int GBM = 64, GBN = 64, GBK = 16, GTM = 4, GTN = 4, GTHREADS = 256;

__global__ void __launch_bounds__(GTHREADS)
ffma_generic_kernel(int64_t M, int64_t N, int64_t K, Epilogue ep, const float *__restrict__ A,
                    int64_t lda, const float *__restrict__ B, int64_t ldb,
                    float *__restrict__ C, int64_t ldc) {
    // A is stored k-major (transposed) so that both operands are read as
    // float4 along the output dimension; +4 keeps rows 16-byte aligned.
    __shared__ __align__(16) float sA[GBK][GBM + 4];
    __shared__ __align__(16) float sB[GBK][GBN + 4];

    const int tid = threadIdx.x;
    const int tx = tid % (GBN / GTN);   // 0..15 -> columns
    const int ty = tid / (GBN / GTN);   // 0..15 -> rows
    const int64_t m0 = (int64_t)blockIdx.y * GBM;
    const int64_t n0 = (int64_t)blockIdx.x * GBN;

    float acc[GTM][GTN];
#pragma unroll
    for (int i = 0; i < GTM; ++i)
#pragma unroll
        for (int j = 0; j < GTN; ++j) acc[i][j] = 0.0f;

    for (int64_t k0 = 0; k0 < K; k0 += GBK) {
#pragma unroll
        for (int q = 0; q < (GBM * GBK) / GTHREADS; ++q) {
            const int idx = tid + q * GTHREADS;
            const int r = idx / GBK, c = idx % GBK;
            const int64_t gm = m0 + r, gk = k0 + c;
            sA[c][r] = (gm < M && gk < K) ? A[gm * lda + gk] : 0.0f;
        }
#pragma unroll
        for (int q = 0; q < (GBK * GBN) / GTHREADS; ++q) {
            const int idx = tid + q * GTHREADS;
            const int r = idx / GBN, c = idx % GBN;
            const int64_t gk = k0 + r, gn = n0 + c;
            sB[r][c] = (gk < K && gn < N) ? B[gk * ldb + gn] : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < GBK; ++k) {
            const float4 a = *reinterpret_cast<const float4 *>(&sA[k][ty * GTM]);
            const float4 b = *reinterpret_cast<const float4 *>(&sB[k][tx * GTN]);
            const float av[4] = {a.x, a.y, a.z, a.w};
            const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < GTM; ++i)
#pragma unroll
                for (int j = 0; j < GTN; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < GTM; ++i) {
        const int64_t gm = m0 + ty * GTM + i;
        if (gm >= M) continue;
#pragma unroll
        for (int j = 0; j < GTN; ++j) {
            const int64_t gn = n0 + tx * GTN + j;
            if (gn >= N) continue;
            float *p = C + gm * ldc + gn;
            const float v = ep.alpha * acc[i][j];
            *p = epilogue_tail(ep, (ep.beta != 0.0f) ? fmaf(ep.beta, *p, v) : v, gn);
        }
    }
}

// C <- act(beta * C + bias); beta == 0 does not read C.
__global__ void __launch_bounds__(256)
scale_c_kernel(int64_t M, int64_t N, Epilogue ep, float *__restrict__ C, int64_t ldc) {
    for (int64_t i = blockIdx.y; i < M; i += gridDim.y) {
        float *row = C + i * ldc;
        for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < N;
             j += (int64_t)gridDim.x * blockDim.x)
            row[j] = epilogue_tail(ep, (ep.beta != 0.0f) ? ep.beta * row[j] : 0.0f, j);
    }
}

}  // namespace

cudaError_t launch_ffma_generic(const GemmArgs &g) {
    const dim3 grid((unsigned)((g.N + GBN - 1) / GBN), (unsigned)((g.M + GBM - 1) / GBM));
    if (grid.y > 65535u) return cudaErrorInvalidConfiguration;
    ffma_generic_kernel<<<grid, GTHREADS, 0, g.stream>>>(g.M, g.N, g.K, g.epi(), g.A, g.lda, g.B,
                                                         g.ldb, g.C, g.ldc);
    return cudaGetLastError();
}

cudaError_t launch_scale_c(const GemmArgs &g) {
    const int64_t gx = (g.N + 255) / 256;
    const dim3 grid((unsigned)(gx < 64 ? gx : 64), (unsigned)(g.M < 65535 ? g.M : 65535));
    scale_c_kernel<<<grid, 256, 0, g.stream>>>(g.M, g.N, g.epi(), g.C, g.ldc);
    return cudaGetLastError();
}

}  // namespace sgemm_gb300
