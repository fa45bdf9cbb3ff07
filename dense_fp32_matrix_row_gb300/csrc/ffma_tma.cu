// ffma_tma.cu -- the FP32 FFMA SGEMM kernel for 16-byte aligned operands.
//
// The tiling hierarchy of "CUDA 矩阵乘法优化：从朴素 Kernel 到接近 cuBLAS"
// (block tile -> warp tile -> thread tile; sections "6. Kernel 5" and
// "9. Kernel 10") with the staging its section "11" leaves as future work
// done by the Tensor Memory Accelerator:
//
//  * one producer warp issues 2-D TMA copies of a BMxBK slice of A and a
//    BKxBN slice of B into a STAGES-deep shared-memory ring; each stage has a
//    "full" mbarrier (TMA bytes landed) and an "empty" mbarrier (all consumer
//    warps finished reading), so copies run ahead of the arithmetic;
//  * eight consumer warps (4 along M x 2 along N) each own a 32x64 warp tile;
//    every lane owns an 8x8 thread tile and forms register outer products
//    (the page's "2D blocktiling"), with 128-bit shared loads for both
//    operands ("7. Kernel 6", vectorised access);
//  * A stays K-contiguous in shared memory as it is in global memory: one
//    128-bit load gives four consecutive k of one row, so no transpose is
//    needed.  The TMA 128-byte swizzle (16-byte chunk index XOR row mod 8)
//    puts the four rows a warp reads at one k in different banks, the
//    conflict-free layout the pages reach with padding or swizzling
//    ("GPU GEMM 优化完全拆解（一）", section "两种解法：Padding 与线性化");
//  * K tails and M/N edge tiles are zero-filled by TMA (out-of-range box
//    elements read as 0) and the epilogue guards its stores; the epilogue
//    applies C = alpha*acc + beta*C, reading C only when beta != 0.
#include "common.cuh"

namespace sgemm_gb300 {
namespace {

constexpr int BM = FfmaTmaShape::BM, BN = FfmaTmaShape::BN, BK = FfmaTmaShape::BK;
constexpr int STAGES = 4;
constexpr int CONSUMER_WARPS = 8;
constexpr int THREADS = (CONSUMER_WARPS + 1) * 32;
constexpr int A_STAGE = BM * BK;   // floats
constexpr int B_STAGE = BK * BN;   // floats
constexpr uint32_t STAGE_BYTES = (A_STAGE + B_STAGE) * 4;
constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + 2 * STAGES * sizeof(uint64_t);
constexpr uint64_t DRAIN_NS = 1000000000ull;   // in-flight copies finish in microseconds

static_assert(BK * 4 == 128, "A rows must be exactly one 128-byte swizzle span");
static_assert((A_STAGE * 4) % 1024 == 0, "stages must keep 1024-byte alignment for the swizzle");

__device__ __forceinline__ float comp(const float4 &v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

__global__ void __launch_bounds__(THREADS, 1)
ffma_tma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                int M, int N, int K, float alpha, float beta, float *__restrict__ C, int64_t ldc,
                int c_vec4, unsigned *err, uint64_t wait_ns) {
    extern __shared__ unsigned char smem_raw[];
    const uintptr_t base = (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023);
    float *sA = reinterpret_cast<float *>(base);
    float *sB = sA + STAGES * A_STAGE;
    uint64_t *full = reinterpret_cast<uint64_t *>(sB + STAGES * B_STAGE);
    uint64_t *empty = full + STAGES;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int ktiles = (K + BK - 1) / BK;

    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), CONSUMER_WARPS);
        }
        mbar_fence_init();
    }
    __syncthreads();

    // ---------------------------------------------------------------- producer
    if (warp == CONSUMER_WARPS) {
        if (lane != 0) return;
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        int kt = 0;
        for (; kt < ktiles; ++kt) {
            const int s = kt % STAGES;
            const uint32_t use = kt / STAGES;
            if (use > 0 && !mbar_wait(smem_u32(&empty[s]), (use - 1) & 1, wait_ns)) break;
            const uint32_t fb = smem_u32(&full[s]);
            mbar_arrive_expect_tx(fb, STAGE_BYTES);
            tma_load_2d(smem_u32(sA + s * A_STAGE), &tmA, fb, kt * BK, m0);
            tma_load_2d(smem_u32(sB + s * B_STAGE), &tmB, fb, n0, kt * BK);
        }
        if (kt < ktiles) {
            // The consumers stopped releasing stages.  Record it, then wait for
            // the copies already issued so none lands after this block exits.
            record_error(err, kErrWaitTimeout);
            for (int q = (kt > STAGES ? kt - STAGES : 0); q < kt; ++q)
                mbar_wait(smem_u32(&full[q % STAGES]), (q / STAGES) & 1, DRAIN_NS);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int wm = warp >> 1, wn = warp & 1;
    const int ty = lane >> 3, tx = lane & 7;
    const int rowbase = wm * 32 + ty;        // thread rows: rowbase + 4*i, i < 8
    const int colbase = wn * 64 + tx * 4;    // thread cols: colbase + {0..3}, +32 + {0..3}

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

    for (int kt = 0; kt < ktiles; ++kt) {
        const int s = kt % STAGES;
        if (!mbar_wait(smem_u32(&full[s]), (kt / STAGES) & 1, wait_ns)) {
            record_error(err, kErrWaitTimeout);
            return;
        }
        const float *a_st = sA + s * A_STAGE + rowbase * BK;
        const float *b_st = sB + s * B_STAGE + colbase;
#pragma unroll
        for (int kc = 0; kc < BK / 4; ++kc) {
            // Row r = rowbase + 4i has (r & 7) = ty for even i and ty ^ 4 for odd i;
            // its k-chunk kc sits at 16-byte chunk kc ^ (r & 7).
            const int sw_even = (kc ^ ty) << 2;
            const int sw_odd = (kc ^ ty ^ 4) << 2;
            float4 a[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                a[i] = *reinterpret_cast<const float4 *>(a_st + i * 4 * BK +
                                                         ((i & 1) ? sw_odd : sw_even));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const float *brow = b_st + (kc * 4 + kk) * BN;
                const float4 b0 = *reinterpret_cast<const float4 *>(brow);
                const float4 b1 = *reinterpret_cast<const float4 *>(brow + 32);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float av = comp(a[i], kk);
                    acc[i][0] = fmaf(av, b0.x, acc[i][0]);
                    acc[i][1] = fmaf(av, b0.y, acc[i][1]);
                    acc[i][2] = fmaf(av, b0.z, acc[i][2]);
                    acc[i][3] = fmaf(av, b0.w, acc[i][3]);
                    acc[i][4] = fmaf(av, b1.x, acc[i][4]);
                    acc[i][5] = fmaf(av, b1.y, acc[i][5]);
                    acc[i][6] = fmaf(av, b1.z, acc[i][6]);
                    acc[i][7] = fmaf(av, b1.w, acc[i][7]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    }

    // ---------------------------------------------------------------- epilogue
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int gm = m0 + rowbase + 4 * i;
        if (gm >= M) continue;
        float *crow = C + (int64_t)gm * ldc;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int gn = n0 + colbase + 32 * h;
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] = alpha * acc[i][4 * h + e];
            if (c_vec4 && gn + 3 < N) {
                float4 *p = reinterpret_cast<float4 *>(crow + gn);
                if (beta != 0.0f) {
                    const float4 o = *p;
                    v[0] = fmaf(beta, o.x, v[0]);
                    v[1] = fmaf(beta, o.y, v[1]);
                    v[2] = fmaf(beta, o.z, v[2]);
                    v[3] = fmaf(beta, o.w, v[3]);
                }
                *p = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (gn + e < N) {
                        float *p = crow + gn + e;
                        *p = (beta != 0.0f) ? fmaf(beta, *p, v[e]) : v[e];
                    }
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_ffma_tma(const GemmArgs &g, const CUtensorMap &tmA, const CUtensorMap &tmB) {
    // The attribute is per device, so it is set on every launch (a host-side call).
    cudaError_t e = cudaFuncSetAttribute(ffma_tma_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((g.N + BN - 1) / BN), (unsigned)((g.M + BM - 1) / BM));
    if (grid.y > 65535u) return cudaErrorInvalidConfiguration;
    const int c_vec4 = ((reinterpret_cast<uintptr_t>(g.C) & 15) == 0) && (g.ldc % 4 == 0);
    ffma_tma_kernel<<<grid, THREADS, SMEM_BYTES, g.stream>>>(
        tmA, tmB, (int)g.M, (int)g.N, (int)g.K, g.alpha, g.beta, g.C, g.ldc, c_vec4, g.err,
        g.wait_ns);
    return cudaGetLastError();
}

}  // namespace sgemm_gb300
