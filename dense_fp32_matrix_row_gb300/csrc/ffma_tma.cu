// ffma_tma.cu -- the FP32 FFMA SGEMM kernel for 16-byte aligned operands.
//
// The tiling hierarchy of "CUDA 矩阵乘法优化：从朴素 Kernel 到接近 cuBLAS"
// (block tile -> warp tile -> thread tile; sections "6. Kernel 5" and
// "9. Kernel 10") with the staging its section "11" leaves as future work
// done by the Tensor Memory Accelerator:
//
//  * 2-D TMA copies of a BMxBK slice of A and a BKxBN slice of B fill a
//    STAGES-deep shared-memory ring; each stage has a "full" mbarrier (TMA
//    bytes landed) and an arrival counter.  There is no producer warp (a
//    ninth warp would take a third of one sub-partition's registers): each
//    warp bumps the stage's counter when it has read the stage, and the warp
//    that arrives last issues the copy that refills it, STAGES k-tiles ahead;
//  * WM x WN consumer warps each own a (4*TM) x (8*TN) warp tile; a lane
//    (4 rows x 8 columns of lanes per warp) owns a TM x TN thread tile and
//    forms register outer products (the page's "2D blocktiling"), with
//    128-bit shared loads for both operands ("7. Kernel 6");
//  * A stays K-contiguous in shared memory as it is in global memory: one
//    128-bit load gives four consecutive k of one row, so no transpose is
//    needed.  The TMA 128-byte swizzle (16-byte chunk index XOR row mod 8)
//    puts the rows a warp reads at one k in different banks, the
//    conflict-free layout the pages reach with padding or swizzling
//    ("GPU GEMM 优化完全拆解（一）", section "两种解法：Padding 与线性化");
//  * K tails and M/N edge tiles are zero-filled by TMA (out-of-range box
//    elements read as 0) and the epilogue guards its stores; the epilogue
//    applies C = alpha*acc + beta*C, reading C only when beta != 0.
//
// Lane (ty, tx) of warp (wm, wn) owns rows  wm*4*TM + ty + 4*i  (i < TM)
//                              and columns wn*8*TN + tx*4 + 32*h + e  (h < TN/4, e < 4).
#include "common.cuh"

#ifndef FFMA_TM
#define FFMA_TM 8
#endif
#ifndef FFMA_TN
#define FFMA_TN 8
#endif
#ifndef FFMA_WM
#define FFMA_WM 4
#endif
#ifndef FFMA_WN
#define FFMA_WN 2
#endif
#ifndef FFMA_STAGES
#define FFMA_STAGES 4
#endif
#ifndef FFMA_SNAKE
#define FFMA_SNAKE 1
#endif

namespace sgemm_gb300 {
namespace {

constexpr uint64_t DRAIN_NS = 1000000000ull;   // in-flight copies finish in microseconds

template <int TM_, int TN_, int WM_, int WN_, int STAGES_>
struct Cfg {
    static constexpr int TM = TM_, TN = TN_, WM = WM_, WN = WN_, STAGES = STAGES_;
    static constexpr int BM = WM * 4 * TM, BN = WN * 8 * TN, BK = 32;
    static constexpr int CONSUMER_WARPS = WM * WN;
    static constexpr int THREADS = CONSUMER_WARPS * 32;
    static constexpr int A_STAGE = BM * BK;   // floats
    static constexpr int B_STAGE = BK * BN;   // floats
    static constexpr uint32_t STAGE_BYTES = (A_STAGE + B_STAGE) * 4;
    static constexpr size_t SMEM = 1024 + (size_t)STAGES * STAGE_BYTES + STAGES * 16;
    static constexpr int B_BOX = BN > 256 ? 256 : BN;   // TMA box is at most 256 wide
    static constexpr int B_BOXES = BN / B_BOX;
    static_assert(TN % 4 == 0, "thread tile columns come in float4 groups");
    static_assert(BK * 4 == 128, "A rows must be exactly one 128-byte swizzle span");
    static_assert((A_STAGE * 4) % 1024 == 0 && (B_STAGE * 4) % 1024 == 0,
                  "stages must keep 1024-byte alignment for the swizzle");
    static_assert(BM <= 256 && BN % B_BOX == 0, "TMA box limits");
    static_assert(SMEM <= 227 * 1024, "shared memory per block");
};

using Default = Cfg<FFMA_TM, FFMA_TN, FFMA_WM, FFMA_WN, FFMA_STAGES>;

__device__ __forceinline__ float comp(const float4 &v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
ffma_tma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                int M, int N, int K, float alpha, float beta, float *__restrict__ Cm, int64_t ldc,
                int c_vec4, unsigned *err, uint64_t wait_ns) {
    constexpr int TM = C::TM, TN = C::TN, BK = C::BK, BN = C::BN, STAGES = C::STAGES;
    extern __shared__ unsigned char smem_raw[];
    const uintptr_t base = (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023);
    float *sA = reinterpret_cast<float *>(base);
    float *sB = sA + STAGES * C::A_STAGE;
    uint64_t *full = reinterpret_cast<uint64_t *>(sB + STAGES * C::B_STAGE);
    unsigned *arrived = reinterpret_cast<unsigned *>(full + STAGES);   // warps done with a stage
    int *issued = reinterpret_cast<int *>(arrived + STAGES);           // k-tile last copied in

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.y * C::BM, n0 = blockIdx.x * C::BN;
    const int ktiles = (K + BK - 1) / BK;

    // Copy k-tile kt into stage kt % STAGES (one thread).
    auto issue = [&](int kt) {
        const int s = kt % STAGES;
        issued[s] = kt;
        const uint32_t fb = smem_u32(&full[s]);
        mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
        tma_load_2d(smem_u32(sA + s * C::A_STAGE), &tmA, fb, kt * BK, m0);
#pragma unroll
        for (int q = 0; q < C::B_BOXES; ++q)
            tma_load_2d(smem_u32(sB + s * C::B_STAGE + q * C::B_BOX * BK), &tmB, fb,
                        n0 + q * C::B_BOX, kt * BK);
    };
    // After a failed wait: wait for every copy issued so far, so that none
    // lands in this block's shared memory after the block has exited.
    auto drain = [&]() {
        for (int s = 0; s < STAGES; ++s) {
            const int kt = *reinterpret_cast<volatile int *>(&issued[s]);
            if (kt >= 0) mbar_wait(smem_u32(&full[s]), (kt / STAGES) & 1, DRAIN_NS);
        }
    };

    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            arrived[s] = 0;
            issued[s] = -1;
        }
        mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        for (int kt = 0; kt < STAGES && kt < ktiles; ++kt) issue(kt);
    }

    // ---------------------------------------------------------------- main loop
    const int wm = warp / C::WN, wn = warp % C::WN;
    const int ty = lane >> 3, tx = lane & 7;
    const int rowbase = wm * 4 * TM + ty;        // thread rows: rowbase + 4*i
    const int colbase = wn * 8 * TN + tx * 4;    // thread cols: colbase + 32*h + e
    // B is stored as B_BOXES boxes of [BK][B_BOX]; column c lives in box c / B_BOX.

    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;

    for (int kt = 0; kt < ktiles; ++kt) {
        const int s = kt % STAGES;
        if (!mbar_wait(smem_u32(&full[s]), (kt / STAGES) & 1, wait_ns)) {
            if (lane == 0) {
                record_error(err, kErrWaitTimeout);
                drain();
            }
            return;
        }
        const float *a_st = sA + s * C::A_STAGE + rowbase * BK;
        const float *b_st = sB + s * C::B_STAGE;
#pragma unroll
        for (int kc = 0; kc < BK / 4; ++kc) {
            // Row r = rowbase + 4i has (r & 7) = ty for even i and ty ^ 4 for odd i;
            // its k-chunk kc sits at 16-byte chunk kc ^ (r & 7).
            const int sw_even = (kc ^ ty) << 2;
            const int sw_odd = (kc ^ ty ^ 4) << 2;
            float4 a[TM];
#pragma unroll
            for (int i = 0; i < TM; ++i)
                a[i] = *reinterpret_cast<const float4 *>(a_st + i * 4 * BK +
                                                         ((i & 1) ? sw_odd : sw_even));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int k = kc * 4 + kk;
                float4 b[TN / 4];
#pragma unroll
                for (int h = 0; h < TN / 4; ++h) {
                    const int c = colbase + 32 * h;
                    b[h] = *reinterpret_cast<const float4 *>(
                        b_st + (c / C::B_BOX) * (C::B_BOX * BK) + k * C::B_BOX + (c % C::B_BOX));
                }
#pragma unroll
                for (int i = 0; i < TM; ++i) {
                    const float av = comp(a[i], kk);
                    // Odd rows walk the columns backwards, so consecutive FFMAs
                    // share an operand across the row change.
#pragma unroll
                    for (int jj = 0; jj < TN; ++jj) {
                        const int j = (FFMA_SNAKE && (i & 1)) ? TN - 1 - jj : jj;
                        acc[i][j] = fmaf(av, comp(b[j / 4], j % 4), acc[i][j]);
                    }
                }
            }
        }
        // Release the stage; the last warp to do so refills it STAGES k-tiles ahead.
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            if (atomicAdd(&arrived[s], 1u) == C::CONSUMER_WARPS - 1) {
                arrived[s] = 0;
                if (kt + STAGES < ktiles) {
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    issue(kt + STAGES);
                }
            }
        }
    }

    // ---------------------------------------------------------------- epilogue
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int gm = m0 + rowbase + 4 * i;
        if (gm >= M) continue;
        float *crow = Cm + (int64_t)gm * ldc;
#pragma unroll
        for (int h = 0; h < TN / 4; ++h) {
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

template <class C>
cudaError_t launch_cfg(const GemmArgs &g) {
    alignas(64) CUtensorMap tmA, tmB;
    if (!encode_tma_2d(g.encode, &tmA, g.A, g.K, g.M, g.lda, C::BK, C::BM,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tma_2d(g.encode, &tmB, g.B, g.N, g.K, g.ldb, C::B_BOX, C::BK,
                       CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    // The attribute is per device, so it is set on every launch (a host-side call).
    cudaError_t e = cudaFuncSetAttribute(ffma_tma_kernel<C>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((g.N + C::BN - 1) / C::BN), (unsigned)((g.M + C::BM - 1) / C::BM));
    if (grid.y > 65535u) return cudaErrorInvalidConfiguration;
    const int c_vec4 = ((reinterpret_cast<uintptr_t>(g.C) & 15) == 0) && (g.ldc % 4 == 0);
    ffma_tma_kernel<C><<<grid, C::THREADS, C::SMEM, g.stream>>>(
        tmA, tmB, (int)g.M, (int)g.N, (int)g.K, g.alpha, g.beta, g.C, g.ldc, c_vec4, g.err,
        g.wait_ns);
    return cudaGetLastError();
}

}  // namespace

int64_t ffma_tma_max_m() { return (int64_t)65535 * Default::BM; }

cudaError_t launch_ffma_tma(const GemmArgs &g) { return launch_cfg<Default>(g); }

}  // namespace sgemm_gb300
