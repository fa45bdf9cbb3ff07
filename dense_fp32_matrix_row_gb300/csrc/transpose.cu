// transpose.cu -- At[k][m] = A[m][k] for the FFMA kernel's A operand.
//
// The FFMA kernel reads A as K-major tiles ([k][m]: four consecutive rows in
// one 128-bit shared load), the layout the pages reach by transposing A on its
// way into shared memory ("CUDA 矩阵乘法优化：从朴素 Kernel 到接近 cuBLAS",
// section "7. Kernel 6"; "GPU 基础原理", section 4.3, load-and-transpose).  TMA
// cannot transpose 4-byte elements, so this memory-bound pass writes A^T once
// into a workspace, and every CTA then stages K-major A tiles with TMA.
//
// 32x32 tiles through padded shared memory: reads are coalesced along k, writes
// along m.  Any A alignment and any lda are accepted (plain 4-byte loads);
// the output row stride ldt is a multiple of 4 floats so TMA can read it.
#include "common.cuh"

namespace sgemm_gb300 {
namespace {

constexpr int TT = 32;       // tile edge
constexpr int TROWS = 8;     // block is TT x TROWS threads

__global__ void __launch_bounds__(TT *TROWS)
transpose_kernel(int64_t M, int64_t K, const float *__restrict__ A, int64_t lda,
                 float *__restrict__ At, int64_t ldt) {
    __shared__ float tile[TT][TT + 1];
    const int64_t k0 = (int64_t)blockIdx.x * TT, m0 = (int64_t)blockIdx.y * TT;
    const int tx = threadIdx.x, ty = threadIdx.y;
#pragma unroll
    for (int r = ty; r < TT; r += TROWS) {
        const int64_t m = m0 + r, k = k0 + tx;
        if (m < M && k < K) tile[r][tx] = A[m * lda + k];
    }
    __syncthreads();
#pragma unroll
    for (int r = ty; r < TT; r += TROWS) {
        const int64_t k = k0 + r, m = m0 + tx;
        if (m < M && k < K) At[k * ldt + m] = tile[tx][r];
    }
}

}  // namespace

cudaError_t launch_transpose(int64_t M, int64_t K, const float *A, int64_t lda, float *At,
                             int64_t ldt, cudaStream_t stream) {
    const int64_t gx = (K + TT - 1) / TT, gy = (M + TT - 1) / TT;
    if (gy > 65535 || gx > 0x7fffffff) return cudaErrorInvalidConfiguration;
    transpose_kernel<<<dim3((unsigned)gx, (unsigned)gy), dim3(TT, TROWS), 0, stream>>>(M, K, A, lda,
                                                                                      At, ldt);
    return cudaGetLastError();
}

}  // namespace sgemm_gb300
