// ffma_tma.cu -- the FP32 FFMA SGEMM kernel (TMA-staged, warp-tiled).
//
// The tiling hierarchy of "CUDA 矩阵乘法优化：从朴素 Kernel 到接近 cuBLAS"
// (block tile -> warp tile -> thread tile; sections "6. Kernel 5" and
// "9. Kernel 10") with the staging its section "11" leaves as future work
// done by the Tensor Memory Accelerator:
//
//  * both operands are staged K-major: a BKxBM slice of A^T (A transposed
//    once into a workspace by transpose.cu) and a BKxBN slice of B, so one
//    128-bit shared load gives four consecutive rows (A) or columns (B) at a
//    single k -- "7. Kernel 6"'s transposed As.  This matters on sm_103: the
//    four operands of a load land in four consecutive registers, so the
//    eight A and eight B operands of a k-step spread over the register banks
//    (K-contiguous A put all eight A operands of a k-step in one bank and
//    capped the inner loop near 70% of the FFMA rate);
//  * 2-D TMA copies fill a STAGES-deep shared-memory ring; each stage has a
//    "full" mbarrier (TMA bytes landed) and an arrival counter.  There is no
//    producer warp: each warp bumps the stage's counter when it has read the
//    stage, and the warp that arrives last issues the copy that refills it,
//    STAGES k-tiles ahead;
//  * WM x WN warps each own a (4*TM) x (8*TN) warp tile; a lane (4 rows x 8
//    columns of lanes per warp) owns a TM x TN thread tile and forms register
//    outer products ("6. Kernel 5", 2D blocktiling).  Odd rows walk the
//    columns backwards so consecutive FFMAs share an operand;
//  * reads of a k row are contiguous float4s, so the shared-memory accesses
//    are free of bank conflicts without padding or swizzle ("GPU GEMM 优化完全
//    拆解（一）", section "共享内存的内部结构：32 个 bank");
//  * K tails and M/N edge tiles are zero-filled by TMA (out-of-range box
//    elements read as 0) and the epilogue guards its stores; the epilogue
//    applies C = act(alpha*acc + beta*C + bias), reading C only when beta != 0;
//  * the grid is a 1-D list of work units: whole tiles for the full waves of
//    CTA slots, then the tail divided by work -- equal runs of k-tile
//    iterations, summed through partial tiles in a fixed order (the split-K
//    of "CUDA 矩阵乘法优化：从朴素 Kernel 到接近 cuBLAS", section "10", see
//    TailPlan and plan_units) by a second kernel over all tail tiles;
//  * the kernel is launched as a programmatic dependent of the transpose that
//    writes its A^T, so its set-up overlaps the transpose's tail.
//
// Lane (ty, tx) of warp (wm, wn) owns rows    wm*4*TM + 16*(i/4) + 4*ty + i%4   (i < TM)
//                                 and columns wn*8*TN + 32*(j/4) + 4*tx + j%4   (j < TN).
#include <algorithm>
#include <atomic>
#include <mutex>

#include "common.cuh"

#ifndef FFMA_TAIL_SPLIT
#define FFMA_TAIL_SPLIT 1
#endif
#ifndef FFMA_PDL
#define FFMA_PDL 1   // launch the tile kernel as a programmatic dependent of the transpose
#endif
#ifndef FFMA_PACKED
#define FFMA_PACKED 1
#endif
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
#define FFMA_STAGES 2
#endif
#ifndef FFMA_BK
#define FFMA_BK 48   // k-steps per k-tile of the default configuration
#endif
#ifndef FFMA_MINB
#define FFMA_MINB 2
#endif
// the 32-row configuration (index 4): k-tile depth, stages, CTAs per SM
#ifndef FFMA_SK_BK
#define FFMA_SK_BK 32
#endif
#ifndef FFMA_SK_STAGES
#define FFMA_SK_STAGES 2
#endif
#ifndef FFMA_SK_MINB
#define FFMA_SK_MINB 3
#endif

namespace sgemm_gb300 {
namespace {

constexpr uint64_t DRAIN_NS = 1000000000ull;   // in-flight copies finish in microseconds

template <int TM_, int TN_, int WM_, int WN_, int BK_, int STAGES_, int MINB_>
struct Cfg {
    static constexpr int TM = TM_, TN = TN_, WM = WM_, WN = WN_, BK = BK_, STAGES = STAGES_;
    static constexpr int MINB = MINB_;
    static constexpr int BM = WM * 4 * TM, BN = WN * 8 * TN;
    static constexpr int WARPS = WM * WN;
    static constexpr int THREADS = WARPS * 32;
    static constexpr int A_STAGE = BK * BM;   // floats, [BK][BM]
    static constexpr int B_STAGE = BK * BN;   // floats, [BK][BN]
    static constexpr uint32_t STAGE_BYTES = (A_STAGE + B_STAGE) * 4;
    static constexpr size_t SMEM = 128 + (size_t)STAGES * STAGE_BYTES + STAGES * 16;
    static_assert(TM % 4 == 0 && TN % 4 == 0, "thread tiles come in float4 groups");
    static_assert(BM <= 256 && BN <= 256, "TMA box is at most 256 elements wide");
    static_assert(SMEM * MINB <= 227 * 1024, "shared memory per SM");
};

// The tile configurations compiled into the library (the search space of the
// tuning script, dense_fp32_matrix_row_gb300/autotune.py).  Index 0 is the
// default; ffma_tuning.inc maps shape classes to an index.
using Default = Cfg<FFMA_TM, FFMA_TN, FFMA_WM, FFMA_WN, FFMA_BK, FFMA_STAGES, FFMA_MINB>;   // 128 x 128, BK 48
using Wide = Cfg<8, 8, 2, 4, 32, 2, 2>;                                         // 64 x 256
using Narrow = Cfg<8, 8, 4, 1, 32, 2, 4>;                                       // 128 x 64
using ShallowK = Cfg<8, 8, 4, 2, 16, 4, 2>;                                     // 128 x 128, BK 16
using Skinny = Cfg<8, 8, 1, 4, FFMA_SK_BK, FFMA_SK_STAGES, FFMA_SK_MINB>;          // 32 x 256
using Base32 = Cfg<8, 8, 4, 2, 32, 2, 2>;                                       // 128 x 128, BK 32
constexpr int kFfmaConfigs = 6;

// f(C{}) for the configuration with index `idx`.
template <class F>
decltype(auto) with_config(int idx, F &&f) {
    switch (idx) {
        case 1: return f(Wide{});
        case 2: return f(Narrow{});
        case 3: return f(ShallowK{});
        case 4: return f(Skinny{});
        case 5: return f(Base32{});
        default: return f(Default{});
    }
}

struct FfmaTuneEntry {
    int64_t m_lo, m_max, n_lo, n_max, k_lo, k_max;   // applies inside these bounds on M, N, K
    int config;
};
#include "ffma_tuning.inc"

std::atomic<int> g_force_config{-1};
std::atomic<int> g_force_tail_sum{-1};   // sgemm_ffma_force_tail_sum

// sgemm_kernel_timing: event pairs around the tile-kernel launches.
constexpr int kTimingSlots = 4096;
std::mutex g_timing_mu;
std::atomic<int> g_timing_on{0};
int g_timing_used = 0;
cudaEvent_t g_timing_ev[kTimingSlots][2] = {};
int g_timing_dev[kTimingSlots] = {};

// The event pair for the next launch (created on first use), or false when
// recording is off or every slot is taken.
bool timing_slot(cudaEvent_t &e0, cudaEvent_t &e1) {
    if (!g_timing_on.load(std::memory_order_relaxed)) return false;
    std::lock_guard<std::mutex> lock(g_timing_mu);
    if (g_timing_used >= kTimingSlots) return false;
    const int i = g_timing_used;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    for (int k = 0; k < 2; ++k) {
        // events belong to the device that was current when they were made
        if (g_timing_ev[i][k] != nullptr && g_timing_dev[i] != dev) {
            (void)cudaEventDestroy(g_timing_ev[i][k]);
            g_timing_ev[i][k] = nullptr;
        }
        if (g_timing_ev[i][k] == nullptr && cudaEventCreate(&g_timing_ev[i][k]) != cudaSuccess) {
            (void)cudaGetLastError();
            g_timing_ev[i][k] = nullptr;
            return false;
        }
    }
    g_timing_dev[i] = dev;
    e0 = g_timing_ev[i][0];
    e1 = g_timing_ev[i][1];
    ++g_timing_used;
    return true;
}

__device__ __forceinline__ float comp(const float4 &v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// acc += the stage's BK-deep outer products for this lane (see the layout above).
template <class C>
__device__ __forceinline__ void compute_stage(float (&acc)[C::TM][C::TN], const float *a_st,
                                              const float *b_st) {
    constexpr int TM = C::TM, TN = C::TN, BM = C::BM, BN = C::BN;
#pragma unroll
    for (int k = 0; k < C::BK; ++k) {
        float4 a[TM / 4], b[TN / 4];
#pragma unroll
        for (int q = 0; q < TM / 4; ++q)
            a[q] = *reinterpret_cast<const float4 *>(a_st + k * BM + 16 * q);
#pragma unroll
        for (int h = 0; h < TN / 4; ++h)
            b[h] = *reinterpret_cast<const float4 *>(b_st + k * BN + 32 * h);
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const float av = comp(a[i / 4], i % 4);
#if FFMA_PACKED
            // two FP32 lanes per instruction (each lane one fused multiply-add,
            // rounded once, exactly as fmaf): half the issue slots of scalar FFMA
            const float2 a2 = make_float2(av, av);
#pragma unroll
            for (int qq = 0; qq < TN / 2; ++qq) {
                const int q = (i & 1) ? TN / 2 - 1 - qq : qq;
                const float4 &bh = b[q / 2];
                const float2 b2 = (q & 1) ? make_float2(bh.z, bh.w) : make_float2(bh.x, bh.y);
                const float2 d = __ffma2_rn(a2, b2, make_float2(acc[i][2 * q], acc[i][2 * q + 1]));
                acc[i][2 * q] = d.x;
                acc[i][2 * q + 1] = d.y;
            }
#else
#pragma unroll
            for (int jj = 0; jj < TN; ++jj) {
                const int j = (i & 1) ? TN - 1 - jj : jj;
                acc[i][j] = fmaf(av, comp(b[j / 4], j % 4), acc[i][j]);
            }
#endif
        }
    }
}

// C = act(alpha*acc + beta*C + bias) for this lane's outputs of the tile at
// (m0, n0); C is read only when beta != 0, stores are guarded at the matrix edge.
template <class C>
__device__ __forceinline__ void store_tile(const float (&acc)[C::TM][C::TN], int m0, int n0,
                                           int arow, int bcol, int M, int N, const Epilogue &ep,
                                           float *__restrict__ Cm, int64_t ldc, int c_vec4) {
    constexpr int TM = C::TM, TN = C::TN;
    const bool tail = ep.bias != nullptr || ep.act != kActNone;
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int gm = m0 + arow + 16 * (i / 4) + (i % 4);
        if (gm >= M) continue;
        float *crow = Cm + (int64_t)gm * ldc;
#pragma unroll
        for (int h = 0; h < TN / 4; ++h) {
            const int gn = n0 + bcol + 32 * h;
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] = ep.alpha * acc[i][4 * h + e];
            if (c_vec4 && gn + 3 < N) {
                float4 *p = reinterpret_cast<float4 *>(crow + gn);
                if (ep.beta != 0.0f) {
                    const float4 o = *p;
                    v[0] = fmaf(ep.beta, o.x, v[0]);
                    v[1] = fmaf(ep.beta, o.y, v[1]);
                    v[2] = fmaf(ep.beta, o.z, v[2]);
                    v[3] = fmaf(ep.beta, o.w, v[3]);
                }
                if (tail) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) v[e] = epilogue_tail(ep, v[e], gn + e);
                }
                *p = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (gn + e < N) {
                        float *p = crow + gn + e;
                        float w = (ep.beta != 0.0f) ? fmaf(ep.beta, *p, v[e]) : v[e];
                        if (tail) w = epilogue_tail(ep, w, gn + e);
                        *p = w;
                    }
                }
            }
        }
    }
}

// Work units.  Units 0 .. full-1 are whole tiles, tile t = unit t, in
// row-major tile order (tiles_x tiles along N).  The tiles after the last
// full wave of CTA slots -- all tiles, when they do not fill one wave -- form
// the tail.  When plan_units finds it cheaper, the tail is divided by work
// rather than by tile: its rem x ktiles k-tile iterations, taken tile by tile
// in k order, are dealt out in contiguous runs of `span` iterations to units
// full, full + 1, ..., so every tail unit gets the same amount of work
// whatever the tile count (the "stream-K" division).  A unit's run may end
// part of one tile and start the next.  For each tile it touches without
// covering it whole, the unit writes its partial tile to a slot of
// `partials`.  By default (reduce_pass) that is all: ffma_tail_reduce_kernel,
// launched right after the tile kernel, sums every tail tile's partial tiles
// in unit order and runs the epilogue.  The alternative, selectable with
// sgemm_ffma_force_tail_sum and giving the same bits, sums inside this
// kernel: each unit counts the tile's arrival in counters[tile - full]
// (zeroed before the launch) and the unit that completes the count sums the
// tile's partial tiles in unit order.  No unit waits for another, and the
// sum order does not depend on timing.
struct TailPlan {
    int tiles_x;
    int full;             // whole-tile units
    int span;             // k-tile iterations per tail unit; 0: no tail division
    int tail_iters;       // rem * ktiles
    float *partials;      // two slots per tail unit, each [TM * TN / 4][THREADS] float4
    unsigned *counters;   // [rem]
    int reduce_pass;      // 1: every tail unit only writes its partial tiles; a second
                          // kernel (ffma_tail_reduce_kernel) sums them
};

// Slot of tail unit v's partial tile of tail tile t: 2v + 1 when v's run ends
// in t (inside it or at its end), 2v when v's run goes on past t.  A run is
// shorter than a tile, so it touches at most two tiles and they get
// different slots.
__device__ __forceinline__ int partial_slot(int v, int t, int span, int ktiles, int iters) {
    const int end = min((v + 1) * span, iters);
    return 2 * v + (end <= (t + 1) * ktiles ? 1 : 0);
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, C::MINB)
ffma_tma_kernel(const __grid_constant__ CUtensorMap tmAt, const __grid_constant__ CUtensorMap tmB,
                int M, int N, int K, Epilogue ep, float *__restrict__ Cm, int64_t ldc,
                int c_vec4, TailPlan tp, unsigned *err, uint64_t wait_ns) {
    constexpr int TM = C::TM, TN = C::TN, BK = C::BK, BM = C::BM, BN = C::BN, STAGES = C::STAGES;
    constexpr int NV = TM * TN / 4;   // float4s of a lane's partial tile
    extern __shared__ unsigned char smem_raw[];
    __shared__ unsigned s_prev;
    const uintptr_t base = (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127);
    float *sA = reinterpret_cast<float *>(base);
    float *sB = sA + STAGES * C::A_STAGE;
    uint64_t *full = reinterpret_cast<uint64_t *>(sB + STAGES * C::B_STAGE);
    unsigned *arrived = reinterpret_cast<unsigned *>(full + STAGES);   // warps done with a stage
    int *issued = reinterpret_cast<int *>(arrived + STAGES);           // local k-tile last copied in

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ktiles = (K + BK - 1) / BK;
    // This unit's k-tile iterations j = 0 .. n-1: k-tile j of tile blockIdx.x,
    // or, for a tail unit v = blockIdx.x - full, iteration v*span + j of the
    // tail (tile full + i/ktiles, k-tile i%ktiles for i = v*span + j).
    const bool in_tail = (int)blockIdx.x >= tp.full;
    const int n = in_tail ? min(tp.span, tp.tail_iters - ((int)blockIdx.x - tp.full) * tp.span) : ktiles;
    // Where the copies of local k-tile j go, kept in shared memory rather than
    // in every thread's registers (only the issuing thread reads them): tile
    // origin (m0, n0) and first k-tile of the unit's first tile, the j at
    // which its second tile starts (n if none), and that tile's origin.
    __shared__ int s_iss[6];
    auto issue = [&](int j) {
        const int s = j % STAGES;
        issued[s] = j;
        const volatile int *q = s_iss;
        const bool second = j >= q[3];
        const int m0 = second ? q[4] : q[0], n0 = second ? q[5] : q[1];
        const int kt = second ? j - q[3] : q[2] + j;
        const uint32_t fb = smem_u32(&full[s]);
        mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
        tma_load_2d(smem_u32(sA + s * C::A_STAGE), &tmAt, fb, m0, kt * BK);
        tma_load_2d(smem_u32(sB + s * C::B_STAGE), &tmB, fb, n0, kt * BK);
    };
    // After a failed wait: wait for every copy issued so far, so that none
    // lands in this block's shared memory after the block has exited.
    auto drain = [&]() {
        for (int s = 0; s < STAGES; ++s) {
            const int j = *reinterpret_cast<volatile int *>(&issued[s]);
            if (j >= 0) mbar_wait(smem_u32(&full[s]), (j / STAGES) & 1, DRAIN_NS);
        }
    };

    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            arrived[s] = 0;
            issued[s] = -1;
        }
        int t0 = blockIdx.x, kt0 = 0, jsw = n, t1 = 0;
        if (in_tail) {
            const int i0 = ((int)blockIdx.x - tp.full) * tp.span;
            t0 = tp.full + i0 / ktiles;
            kt0 = i0 % ktiles;
            jsw = min(n, ktiles - kt0);
            t1 = t0 + 1;
        }
        s_iss[0] = (t0 / tp.tiles_x) * BM;
        s_iss[1] = (t0 % tp.tiles_x) * BN;
        s_iss[2] = kt0;
        s_iss[3] = jsw;
        s_iss[4] = (t1 / tp.tiles_x) * BM;
        s_iss[5] = (t1 % tp.tiles_x) * BN;
        mbar_fence_init();
        tma_prefetch_desc(&tmAt);
        tma_prefetch_desc(&tmB);
    }
    // Launched as a programmatic dependent of the transpose: everything above
    // overlaps its tail; A^T, and the tail counters it zeroes, are read only
    // after it has completed.
    pdl_wait();
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int j = 0; j < STAGES && j < n; ++j) issue(j);
    }

    const int wm = warp / C::WN, wn = warp % C::WN;
    const int ty = lane >> 3, tx = lane & 7;
    const int arow = wm * 4 * TM + 4 * ty;     // + 16*q + r
    const int bcol = wn * 8 * TN + 4 * tx;     // + 32*h + e

    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int jj = 0; jj < TN; ++jj) acc[i][jj] = 0.0f;

    // Segments: the k-tiles a unit computes for one tile (a whole-tile unit
    // has one; a tail unit one or two).  The k loop of a segment is the
    // kernel's hot loop; segment ends are block-wide (a failed wait in any
    // warp is seen there and skips every later store).
    bool any_failed = false;
    for (int j0 = 0; j0 < n;) {
        const int j1 = j0 == 0 ? s_iss[3] : n;   // the first tile's k-tiles, then the rest
        bool failed = false;
        for (int j = j0; j < j1; ++j) {
            const int s = j % STAGES;
            if (!mbar_wait(smem_u32(&full[s]), (j / STAGES) & 1, wait_ns)) {
                failed = true;
                if (lane == 0) record_error(err, kErrWaitTimeout);
                break;
            }
            compute_stage<C>(acc, sA + s * C::A_STAGE + arow, sB + s * C::B_STAGE + bcol);
            // Release the stage; the last warp to do so refills it STAGES k-tiles ahead.
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();
                if (atomicAdd(&arrived[s], 1u) == C::WARPS - 1) {
                    arrived[s] = 0;
                    if (j + STAGES < n) {
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        issue(j + STAGES);
                    }
                }
            }
        }
        any_failed = __syncthreads_or(failed) != 0;
        if (any_failed) break;

        const int m0 = s_iss[j0 == 0 ? 0 : 4], n0 = s_iss[j0 == 0 ? 1 : 5];
        if (j1 - j0 == ktiles) {
            store_tile<C>(acc, m0, n0, arow, bcol, M, N, ep, Cm, ldc, c_vec4);
        } else {
            // partial tile, thread-interleaved so that each warp writes whole lines
            const int v = (int)blockIdx.x - tp.full;
            const int t = (v * tp.span + j0) / ktiles;   // tail tile of this segment
            float4 *mine = reinterpret_cast<float4 *>(tp.partials) +
                           (size_t)partial_slot(v, t, tp.span, ktiles, tp.tail_iters) * NV * C::THREADS;
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int h = 0; h < TN / 4; ++h)
                    __stcg(mine + (size_t)(i * (TN / 4) + h) * C::THREADS + threadIdx.x,
                           make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2],
                                       acc[i][4 * h + 3]));
            // with a reduce pass the partial tile is all this unit contributes
            if (!tp.reduce_pass) {
                __threadfence();
                __syncthreads();
                if (threadIdx.x == 0) s_prev = atomicAdd(&tp.counters[t], 1u);
                __syncthreads();
                const int v0 = t * ktiles / tp.span, v1 = ((t + 1) * ktiles - 1) / tp.span;
                if (s_prev == (unsigned)(v1 - v0)) {
                    // last one in: sum the partial tiles of units v0 .. v1 in that
                    // order (this unit's included), whichever unit arrived last
                    __threadfence();
                    for (int w = v0; w <= v1; ++w) {
                        const float4 *src = reinterpret_cast<const float4 *>(tp.partials) +
                                            (size_t)partial_slot(w, t, tp.span, ktiles, tp.tail_iters) * NV *
                                                C::THREADS;
#pragma unroll
                        for (int i = 0; i < TM; ++i)
#pragma unroll
                            for (int h = 0; h < TN / 4; ++h) {
                                const float4 q = __ldcg(src + (size_t)(i * (TN / 4) + h) * C::THREADS + threadIdx.x);
                                if (w == v0) {
                                    acc[i][4 * h] = q.x; acc[i][4 * h + 1] = q.y;
                                    acc[i][4 * h + 2] = q.z; acc[i][4 * h + 3] = q.w;
                                } else {
                                    acc[i][4 * h] += q.x; acc[i][4 * h + 1] += q.y;
                                    acc[i][4 * h + 2] += q.z; acc[i][4 * h + 3] += q.w;
                                }
                            }
                    }
                    store_tile<C>(acc, m0, n0, arow, bcol, M, N, ep, Cm, ldc, c_vec4);
                }
            }
        }
        j0 = j1;
        if (j0 < n) {
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int jj = 0; jj < TN; ++jj) acc[i][jj] = 0.0f;
        }
    }
    // Every warp is past its k loop, so `issued` no longer changes.
    if (any_failed && threadIdx.x == 0) drain();
}

// The tail's partial tiles summed by a kernel of their own (TailPlan::
// reduce_pass): one thread per float4 of a tail tile, the partials of units
// v0 .. v1 added in that order and the epilogue applied -- the same
// arithmetic, in the same order, as the last unit to arrive would do, spread
// over the whole GPU instead of one CTA per tile.  Launched as a
// programmatic dependent of the tile kernel.
template <class C>
__global__ void __launch_bounds__(256)
ffma_tail_reduce_kernel(TailPlan tp, int ktiles, int M, int N, Epilogue ep, float *__restrict__ Cm,
                        int64_t ldc, int c_vec4) {
    constexpr int TM = C::TM, TN = C::TN, NV = TM * TN / 4;
    constexpr int PER_TILE = NV * C::THREADS;   // float4s of one partial tile
    pdl_wait();
    const int t = blockIdx.y;                   // tail tile
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= PER_TILE) return;
    // the tile kernel's thread (tid) and register (i, h) this float4 came from
    const int tid = e % C::THREADS, q = e / C::THREADS;
    const int i = q / (TN / 4), h = q % (TN / 4);
    const int warp = tid >> 5, lane = tid & 31;
    const int wm = warp / C::WN, wn = warp % C::WN;
    const int gt = tp.full + t;
    const int gm = (gt / tp.tiles_x) * C::BM + wm * 4 * TM + 4 * (lane >> 3) + 16 * (i / 4) + (i % 4);
    const int64_t gn = (int64_t)(gt % tp.tiles_x) * C::BN + wn * 8 * TN + 4 * (lane & 7) + 32 * h;
    if (gm >= M || gn >= N) return;
    const int v0 = t * ktiles / tp.span, v1 = ((t + 1) * ktiles - 1) / tp.span;
    const float4 *P = reinterpret_cast<const float4 *>(tp.partials);
    float4 sum = __ldcg(P + (size_t)partial_slot(v0, t, tp.span, ktiles, tp.tail_iters) * PER_TILE + e);
#pragma unroll 4
    for (int w = v0 + 1; w <= v1; ++w) {
        const float4 x = __ldcg(P + (size_t)partial_slot(w, t, tp.span, ktiles, tp.tail_iters) * PER_TILE + e);
        sum.x += x.x; sum.y += x.y; sum.z += x.z; sum.w += x.w;
    }
    float v[4] = {ep.alpha * sum.x, ep.alpha * sum.y, ep.alpha * sum.z, ep.alpha * sum.w};
    float *crow = Cm + (int64_t)gm * ldc;
    const bool tail = ep.bias != nullptr || ep.act != kActNone;
    if (c_vec4 && gn + 3 < N) {
        float4 *p = reinterpret_cast<float4 *>(crow + gn);
        if (ep.beta != 0.0f) {
            const float4 o = *p;
            v[0] = fmaf(ep.beta, o.x, v[0]);
            v[1] = fmaf(ep.beta, o.y, v[1]);
            v[2] = fmaf(ep.beta, o.z, v[2]);
            v[3] = fmaf(ep.beta, o.w, v[3]);
        }
        if (tail) {
#pragma unroll
            for (int k = 0; k < 4; ++k) v[k] = epilogue_tail(ep, v[k], gn + k);
        }
        *p = make_float4(v[0], v[1], v[2], v[3]);
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (gn + k < N) {
                float *p = crow + gn + k;
                float w = (ep.beta != 0.0f) ? fmaf(ep.beta, *p, v[k]) : v[k];
                if (tail) w = epilogue_tail(ep, w, gn + k);
                *p = w;
            }
        }
    }
}

// CTAs of the kernel one SM holds, per device (0 until asked).
template <class C>
int ctas_per_sm() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaFuncSetAttribute(ffma_tma_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::SMEM) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, ffma_tma_kernel<C>, C::THREADS, C::SMEM) !=
            cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

// The work list for one call (see TailPlan).  The tail -- the tiles left
// after the last full wave of CTA slots, all tiles when they do not fill one
// wave -- is divided by work when that is cheaper under a simple model: run
// as whole tiles, it takes one wave of ktiles k-tiles plus a fixed cost per
// unit (pipeline fill, epilogue); divided, one wave of `span` k-tiles plus two
// fixed costs (a unit may end one tile and start the next), where span is
// the tail's iterations over the CTA slots, at least four k-tiles and fewer
// than ktiles.  The fixed cost is FFMA_SPLIT_C0 k-steps.  The partial tiles
// (two slots per tail unit) must fit in `capacity` floats of workspace beside
// A^T; a longer span (fewer units) is taken when they do not.
#ifndef FFMA_SPLIT_C0
#define FFMA_SPLIT_C0 64
#endif
struct Plan {
    int tiles_x = 0;
    int64_t tiles = 0, full = 0;
    int span = 0;              // 0: whole tiles only
    bool reduce_pass = false;  // partial tiles summed by ffma_tail_reduce_kernel
    int64_t tail_units = 0;
    int64_t rem() const { return tiles - full; }
    int64_t units() const { return full + tail_units; }
};
constexpr int64_t kCounterFloats = 1024;   // counters reserved after A^T
constexpr int64_t kMinSpan = 4;            // k-tiles per tail unit, at least

template <class C>
int64_t partial_floats(const Plan &p) {
    return p.span > 0 ? kCounterFloats + 2 * p.tail_units * (int64_t)C::BM * C::BN : 0;
}

template <class C>
Plan plan_units(const GemmArgs &g, int64_t at_floats, int64_t capacity) {
    Plan p;
    p.tiles_x = (int)((g.N + C::BN - 1) / C::BN);
    p.tiles = (int64_t)p.tiles_x * ((g.M + C::BM - 1) / C::BM);
    p.full = p.tiles;
    const int64_t slots = (int64_t)ctas_per_sm<C>() * g.sm_count;
    const int64_t ktiles = (g.K + C::BK - 1) / C::BK;
    if (slots <= 0 || !FFMA_TAIL_SPLIT) return p;
    const int64_t rem = p.tiles % slots;
    if (rem == 0 || rem > kCounterFloats) return p;
    const int64_t iters = rem * ktiles;
    const int64_t whole_cost = ktiles * C::BK + FFMA_SPLIT_C0;
    Plan q = p;
    q.full = p.tiles - rem;
    for (int64_t span = std::max(kMinSpan, (iters + slots - 1) / slots); span < ktiles; ++span) {
        if (span * C::BK + 2 * FFMA_SPLIT_C0 >= whole_cost) break;   // no cheaper than whole tiles
        q.span = (int)span;
        q.tail_units = (iters + span - 1) / span;
        // The last unit to arrive at a tile would read the others' partial
        // tiles one after another; a separate kernel sums every tile's
        // partials at once, which measured as fast or faster on every shape.
        const int forced = g_force_tail_sum.load(std::memory_order_relaxed);
        q.reduce_pass = forced != 0;
        if (at_floats + partial_floats<C>(q) <= capacity) return q;   // the shortest span that fits
    }
    return p;
}

template <class C>
cudaError_t launch_cfg(const GemmArgs &g, const float *At, int64_t ldt, const Plan &p, float *extra) {
    alignas(64) CUtensorMap tmAt, tmB;
    if (!encode_tma_2d(g.encode, &tmAt, At, g.M, g.K, ldt, C::BM, C::BK, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_tma_2d(g.encode, &tmB, g.B, g.N, g.K, g.ldb, C::BN, C::BK, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    // The attribute is per device, so it is set on every launch (a host-side call).
    cudaError_t e = cudaFuncSetAttribute(ffma_tma_kernel<C>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e != cudaSuccess) return e;
    if (p.units() > 0x7fffffff) return cudaErrorInvalidConfiguration;
    TailPlan tp;
    tp.tiles_x = p.tiles_x;
    tp.full = (int)p.full;
    tp.span = p.span;
    tp.tail_iters = (int)(p.rem() * ((g.K + C::BK - 1) / C::BK));
    tp.counters = reinterpret_cast<unsigned *>(extra);
    tp.partials = extra != nullptr ? extra + kCounterFloats : nullptr;
    tp.reduce_pass = p.span > 0 && p.reduce_pass ? 1 : 0;
    const int c_vec4 = ((reinterpret_cast<uintptr_t>(g.C) & 15) == 0) && (g.ldc % 4 == 0);
    // a programmatic dependent of the transpose launched just before it
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.units(), 1, 1);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = g.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = FFMA_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaEvent_t t0 = nullptr, t1 = nullptr;
    const bool timed = timing_slot(t0, t1);
    if (timed && (e = cudaEventRecord(t0, g.stream)) != cudaSuccess) return e;
    e = cudaLaunchKernelEx(&cfg, ffma_tma_kernel<C>, tmAt, tmB, (int)g.M, (int)g.N, (int)g.K, g.epi(),
                           g.C, g.ldc, c_vec4, tp, g.err, g.wait_ns);
    if (e == cudaSuccess && timed) e = cudaEventRecord(t1, g.stream);
    if (e != cudaSuccess || !tp.reduce_pass) return e;
    constexpr int per_tile = C::TM * C::TN / 4 * C::THREADS;
    cudaLaunchConfig_t rcfg = cfg;
    rcfg.gridDim = dim3((unsigned)((per_tile + 255) / 256), (unsigned)p.rem(), 1);
    rcfg.blockDim = dim3(256, 1, 1);
    rcfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&rcfg, ffma_tail_reduce_kernel<C>, tp, (int)((g.K + C::BK - 1) / C::BK),
                              (int)g.M, (int)g.N, g.epi(), g.C, g.ldc, c_vec4);
}

}  // namespace

int64_t ffma_tma_max_m() { return (int64_t)65535 * Default::BM; }

int64_t ffma_tma_at_ld(int64_t M) { return (M + 3) / 4 * 4; }

int ffma_config_for(int64_t M, int64_t N, int64_t K) {
    const int forced = g_force_config.load(std::memory_order_relaxed);
    if (forced >= 0 && forced < kFfmaConfigs) return forced;
    for (const FfmaTuneEntry &e : kFfmaTune)
        if (e.m_lo <= M && M <= e.m_max && e.n_lo <= N && N <= e.n_max && e.k_lo <= K && K <= e.k_max)
            return (e.config >= 0 && e.config < kFfmaConfigs) ? e.config : 0;
    return 0;
}

int ffma_config_count() { return kFfmaConfigs; }

void ffma_tma_plan_info(const GemmArgs &g, int64_t *units, int *span, int *tail_sum) {
    const int64_t at = g.K * ffma_tma_at_ld(g.M);
    with_config(ffma_config_for(g.M, g.N, g.K), [&](auto c) {
        using C = decltype(c);
        const Plan p = plan_units<C>(g, at, INT64_MAX);
        *units = p.units();
        *span = p.span;
        *tail_sum = p.span > 0 && p.reduce_pass ? 1 : 0;
        return 0;
    });
}

int kernel_timing(int enable) {
    if (enable != 0 && enable != 1) return -2;
    std::lock_guard<std::mutex> lock(g_timing_mu);
    if (enable) g_timing_used = 0;
    return g_timing_on.exchange(enable);
}

bool kernel_timing_result(double *total_ms, int64_t *launches) {
    std::lock_guard<std::mutex> lock(g_timing_mu);
    double sum = 0.0;
    int cur = 0;
    if (cudaGetDevice(&cur) != cudaSuccess) return false;
    bool ok = true;
    for (int i = 0; i < g_timing_used && ok; ++i) {
        float ms = 0.0f;
        ok = cudaSetDevice(g_timing_dev[i]) == cudaSuccess &&
             cudaEventSynchronize(g_timing_ev[i][1]) == cudaSuccess &&
             cudaEventElapsedTime(&ms, g_timing_ev[i][0], g_timing_ev[i][1]) == cudaSuccess;
        sum += ms;
    }
    if (cudaSetDevice(cur) != cudaSuccess) ok = false;
    if (!ok) {
        (void)cudaGetLastError();
        return false;
    }
    *total_ms = sum;
    *launches = g_timing_used;
    return true;
}

int ffma_force_tail_sum(int mode) {
    if (mode < -1 || mode > 1) return -2;
    return g_force_tail_sum.exchange(mode);
}

int ffma_force_config(int idx) {
    if (idx < -1 || idx >= kFfmaConfigs) return -2;
    return g_force_config.exchange(idx);
}

bool ffma_config_info(int idx, int *bm, int *bn, int *bk, int *stages, int *threads, int *minb) {
    if (idx < 0 || idx >= kFfmaConfigs) return false;
    with_config(idx, [&](auto c) {
        using C = decltype(c);
        *bm = C::BM; *bn = C::BN; *bk = C::BK; *stages = C::STAGES; *threads = C::THREADS;
        *minb = C::MINB;
        return 0;
    });
    return true;
}

int64_t ffma_tma_workspace_floats(const GemmArgs &g, int64_t capacity) {
    const int64_t at = g.K * ffma_tma_at_ld(g.M);
    return with_config(ffma_config_for(g.M, g.N, g.K), [&](auto c) -> int64_t {
        using C = decltype(c);
        return at + partial_floats<C>(plan_units<C>(g, at, capacity));
    });
}

cudaError_t launch_ffma_tma(const GemmArgs &g, float *workspace, int64_t capacity) {
    const int64_t ldt = ffma_tma_at_ld(g.M);
    const int64_t at = g.K * ldt;
    return with_config(ffma_config_for(g.M, g.N, g.K), [&](auto c) -> cudaError_t {
        using C = decltype(c);
        const Plan p = plan_units<C>(g, at, capacity);
        float *extra = p.span > 0 ? workspace + at : nullptr;
        cudaError_t e = launch_transpose(g.M, g.K, g.A, g.lda, workspace, ldt, g.stream,
                                         reinterpret_cast<unsigned *>(extra),
                                         (int)(p.span > 0 ? p.rem() : 0));
        if (e != cudaSuccess) return e;
        return launch_cfg<C>(g, workspace, ldt, p, extra);
    });
}

}  // namespace sgemm_gb300
