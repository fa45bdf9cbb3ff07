// transpose.cu -- memory-bound operand preparation passes.
//
//  * launch_transpose:       At[k][m] = A[m][k] (the FFMA kernel's K-major A);
//  * launch_transpose_split: hi[n][k] = tf32(B[k][n]), lo[n][k] = tf32(B[k][n] - hi)
//                            (the TF32 kernels' K-major B; lo skipped when null);
//  * launch_split_rows:      hi[r][c] = tf32(X[r][c]), lo[r][c] = tf32(X[r][c] - hi)
//                            (the TF32 kernels' A; lo skipped when null);
//  * launch_bf16_rows / launch_bf16_transpose: the BF16 kernel's A ([M][K]) and
//                            B^T ([N][K]), rounded to nearest even.
//
// The FFMA kernel reads A as K-major tiles (four consecutive rows in one
// 128-bit shared load), the layout the pages reach by transposing A on its way
// into shared memory ("CUDA 矩阵乘法优化：从朴素 Kernel 到接近 cuBLAS", section
// "7. Kernel 6"; "GPU 基础原理", section 4.3, load-and-transpose).  TMA cannot
// transpose 4-byte elements, so these passes write the transposed operand once
// and every CTA then stages K-major tiles with TMA.
//
// Transposes go through 64 x 64 shared-memory tiles: 128-bit loads along the
// source rows, 128-bit stores along the destination rows, scalar accesses
// only where a source row is unaligned or a tile is cut by the matrix edge.
// Destination row strides are multiples of 4 floats.
#include <cuda_bf16.h>

#include "common.cuh"

namespace sgemm_gb300 {
namespace {

constexpr int TD = 64;            // tile edge
#ifndef ROWS_UNROLL
#define ROWS_UNROLL 4   // float4 groups per thread and pass in the BF16 row conversion
#endif
constexpr int TTHREADS = 256;     // 16 float4 columns x 16 rows per pass

__device__ __forceinline__ float tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// Output of a transposing pass.
enum : int { kOutCopy = 0, kOutTf32Split = 1, kOutBf16 = 2 };

// dst[c][r] from src[r][c], R x Cc source: a copy (kOutCopy), the TF32 hi /
// lo split into dst_hi / dst_lo (kOutTf32Split; lo skipped when null), or
// BF16 rounded to nearest even into dst_hi reinterpreted as bf16 (kOutBf16).
template <int OUT>
__global__ void __launch_bounds__(TTHREADS)
transpose_tile_kernel(int64_t R, int64_t Cc, const float *__restrict__ src, int64_t lds,
                      int src_vec, float *__restrict__ dst_hi, float *__restrict__ dst_lo,
                      int64_t ldd, unsigned *__restrict__ zero, int nzero) {
    constexpr bool SPLIT = OUT == kOutTf32Split;
    __shared__ float tile[TD][TD + 1];
    // the kernel that consumes this output may be launched now; it waits
    // for this grid to complete before it reads anything (pdl_wait)
    pdl_trigger();
    if (blockIdx.x == 0 && blockIdx.y == 0)
        for (int i = threadIdx.x; i < nzero; i += TTHREADS) zero[i] = 0u;
    const int64_t r0 = (int64_t)blockIdx.y * TD, c0 = (int64_t)blockIdx.x * TD;
    const int t = threadIdx.x;
    const int q = t & 15;         // float4 column within the tile
    const int row = t >> 4;       // 0..15
#pragma unroll
    for (int i = 0; i < TD / 16; ++i) {
        const int rr = row + 16 * i;
        const int64_t r = r0 + rr, c = c0 + 4 * q;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (r < R) {
            const float *p = src + r * lds + c;
            if (src_vec && c + 3 < Cc) {
                const float4 x = *reinterpret_cast<const float4 *>(p);
                v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (c + e < Cc) v[e] = p[e];
            }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) tile[rr][4 * q + e] = v[e];
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < TD / 16; ++i) {
        const int cc = row + 16 * i;          // destination row (source column)
        const int64_t c = c0 + cc, r = r0 + 4 * q;
        if (c >= Cc) continue;
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = tile[4 * q + e][cc];
        if constexpr (OUT == kOutBf16) {
            __nv_bfloat16 *pb = reinterpret_cast<__nv_bfloat16 *>(dst_hi) + c * ldd + r;
            if (r + 3 < R) {
                const __nv_bfloat162 lo2 = __floats2bfloat162_rn(v[0], v[1]);
                const __nv_bfloat162 hi2 = __floats2bfloat162_rn(v[2], v[3]);
                uint2 w;
                w.x = *reinterpret_cast<const uint32_t *>(&lo2);
                w.y = *reinterpret_cast<const uint32_t *>(&hi2);
                *reinterpret_cast<uint2 *>(pb) = w;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (r + e < R) pb[e] = __float2bfloat16_rn(v[e]);
            }
        } else {
            float h[4], l[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (SPLIT) {
                    h[e] = tf32_rna(v[e]);
                    l[e] = tf32_rna(v[e] - h[e]);
                } else {
                    h[e] = v[e];
                }
            }
            float *ph = dst_hi + c * ldd + r;
            const bool wlo = SPLIT && dst_lo != nullptr;
            float *pl = wlo ? dst_lo + c * ldd + r : nullptr;
            if (r + 3 < R) {
                *reinterpret_cast<float4 *>(ph) = make_float4(h[0], h[1], h[2], h[3]);
                if (wlo) *reinterpret_cast<float4 *>(pl) = make_float4(l[0], l[1], l[2], l[3]);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (r + e < R) {
                        ph[e] = h[e];
                        if (wlo) pl[e] = l[e];
                    }
                }
            }
        }
    }
}

// hi/lo split of an R x Cc row-major matrix into two [R][ldo] arrays.
__global__ void __launch_bounds__(256)
split_rows_kernel(int64_t R, int64_t Cc, const float *__restrict__ X, int64_t ldx, int x_vec,
                  float *__restrict__ hi, float *__restrict__ lo, int64_t ldo) {
    const int64_t c4n = (Cc + 3) / 4;
    for (int64_t r = blockIdx.y; r < R; r += gridDim.y) {
        for (int64_t c4 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c4 < c4n;
             c4 += (int64_t)gridDim.x * blockDim.x) {
            const int64_t c = 4 * c4;
            const float *p = X + r * ldx + c;
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            const bool full = c + 3 < Cc;
            if (x_vec && full) {
                const float4 x = *reinterpret_cast<const float4 *>(p);
                v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (c + e < Cc) v[e] = p[e];
            }
            float h[4], l[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                h[e] = tf32_rna(v[e]);
                l[e] = tf32_rna(v[e] - h[e]);
            }
            float *ph = hi + r * ldo + c;
            float *pl = lo != nullptr ? lo + r * ldo + c : nullptr;
            if (full) {
                *reinterpret_cast<float4 *>(ph) = make_float4(h[0], h[1], h[2], h[3]);
                if (pl) *reinterpret_cast<float4 *>(pl) = make_float4(l[0], l[1], l[2], l[3]);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (c + e < Cc) {
                        ph[e] = h[e];
                        if (pl) pl[e] = l[e];
                    }
            }
        }
    }
}

// out[r][c] = bf16(X[r][c]) (round to nearest even) for an R x Cc matrix.  A
// thread converts ROWS_UNROLL float4 groups of a row per pass, their loads
// issued together: with one 16-byte load in flight per thread the pass ran
// at 76% of the copy rate, with four at 87% (8192 x 8192: 78 -> 68 us).
__global__ void __launch_bounds__(256)
bf16_rows_kernel(int64_t R, int64_t Cc, const float *__restrict__ X, int64_t ldx, int x_vec,
                 __nv_bfloat16 *__restrict__ out, int64_t ldo) {
    const int64_t c4n = (Cc + 3) / 4;
    const int64_t step = (int64_t)gridDim.x * blockDim.x * ROWS_UNROLL;
    for (int64_t r = blockIdx.y; r < R; r += gridDim.y) {
        for (int64_t c40 = (int64_t)blockIdx.x * blockDim.x * ROWS_UNROLL + threadIdx.x; c40 < c4n;
             c40 += step) {
            float v[ROWS_UNROLL][4];
#pragma unroll
            for (int u = 0; u < ROWS_UNROLL; ++u) {
                const int64_t c = 4 * (c40 + (int64_t)u * blockDim.x);
                const float *p = X + r * ldx + c;
#pragma unroll
                for (int e = 0; e < 4; ++e) v[u][e] = 0.f;
                if (c >= Cc) continue;
                if (x_vec && c + 3 < Cc) {
                    const float4 x = *reinterpret_cast<const float4 *>(p);
                    v[u][0] = x.x; v[u][1] = x.y; v[u][2] = x.z; v[u][3] = x.w;
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (c + e < Cc) v[u][e] = p[e];
                }
            }
#pragma unroll
            for (int u = 0; u < ROWS_UNROLL; ++u) {
                const int64_t c = 4 * (c40 + (int64_t)u * blockDim.x);
                if (c >= Cc) continue;
                __nv_bfloat16 *po = out + r * ldo + c;
                if (c + 3 < Cc) {
                    const __nv_bfloat162 lo2 = __floats2bfloat162_rn(v[u][0], v[u][1]);
                    const __nv_bfloat162 hi2 = __floats2bfloat162_rn(v[u][2], v[u][3]);
                    uint2 w;
                    w.x = *reinterpret_cast<const uint32_t *>(&lo2);
                    w.y = *reinterpret_cast<const uint32_t *>(&hi2);
                    *reinterpret_cast<uint2 *>(po) = w;
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (c + e < Cc) po[e] = __float2bfloat16_rn(v[u][e]);
                }
            }
        }
    }
}

inline int vec_ok(const float *p, int64_t ld) {
    return ((reinterpret_cast<uintptr_t>(p) & 15) == 0) && (ld % 4 == 0);
}

template <int OUT>
cudaError_t launch_tile(int64_t R, int64_t Cc, const float *src, int64_t lds, float *hi, float *lo,
                        int64_t ldd, cudaStream_t stream, unsigned *zero = nullptr, int nzero = 0) {
    const int64_t gx = (Cc + TD - 1) / TD, gy = (R + TD - 1) / TD;
    if (gy > 65535 || gx > 0x7fffffff || nzero < 0 || nzero > 1024 || (nzero > 0 && zero == nullptr))
        return cudaErrorInvalidConfiguration;
    if (gx == 0 || gy == 0) {
        if (nzero > 0) return cudaMemsetAsync(zero, 0, (size_t)nzero * sizeof(unsigned), stream);
        return cudaSuccess;
    }
    transpose_tile_kernel<OUT><<<dim3((unsigned)gx, (unsigned)gy), TTHREADS, 0, stream>>>(
        R, Cc, src, lds, vec_ok(src, lds), hi, lo, ldd, zero, nzero);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_transpose(int64_t M, int64_t K, const float *A, int64_t lda, float *At,
                             int64_t ldt, cudaStream_t stream, unsigned *zero, int nzero) {
    return launch_tile<kOutCopy>(M, K, A, lda, At, nullptr, ldt, stream, zero, nzero);
}

cudaError_t launch_transpose_split(int64_t K, int64_t N, const float *B, int64_t ldb, float *hi,
                                   float *lo, int64_t ldo, cudaStream_t stream) {
    return launch_tile<kOutTf32Split>(K, N, B, ldb, hi, lo, ldo, stream);
}

cudaError_t launch_bf16_rows(int64_t R, int64_t Cc, const float *X, int64_t ldx, void *out,
                             int64_t ldo, cudaStream_t stream) {
    const int64_t c4n = (Cc + 3) / 4;
    const int64_t gx = (c4n + 256 * ROWS_UNROLL - 1) / (256 * ROWS_UNROLL);
    const dim3 grid((unsigned)(gx < 64 ? (gx > 0 ? gx : 1) : 64),
                    (unsigned)(R < 65535 ? (R > 0 ? R : 1) : 65535));
    bf16_rows_kernel<<<grid, 256, 0, stream>>>(R, Cc, X, ldx, vec_ok(X, ldx),
                                               static_cast<__nv_bfloat16 *>(out), ldo);
    return cudaGetLastError();
}

cudaError_t launch_bf16_transpose(int64_t K, int64_t N, const float *B, int64_t ldb, void *out,
                                  int64_t ldo, cudaStream_t stream) {
    return launch_tile<kOutBf16>(K, N, B, ldb, static_cast<float *>(out), nullptr, ldo, stream);
}

cudaError_t launch_split_rows(int64_t R, int64_t Cc, const float *X, int64_t ldx, float *hi,
                              float *lo, int64_t ldo, cudaStream_t stream) {
    const int64_t c4n = (Cc + 3) / 4;
    const int64_t gx = (c4n + 255) / 256;
    const dim3 grid((unsigned)(gx < 64 ? (gx > 0 ? gx : 1) : 64),
                    (unsigned)(R < 65535 ? (R > 0 ? R : 1) : 65535));
    split_rows_kernel<<<grid, 256, 0, stream>>>(R, Cc, X, ldx, vec_ok(X, ldx), hi, lo, ldo);
    return cudaGetLastError();
}

}  // namespace sgemm_gb300
