// decode.cu -- SGEMM for M <= 16 rows (the decode regime).
//
// With M = batch the product is a matrix-vector-like pass that is bound by
// reading B once from HBM ("GPU GEMM 优化完全拆解（一）", section "LLM 推理本质上是
// GEMM 的串联": decode is memory-bound).  The kernel streams B with 128-bit
// loads that do not allocate in L1, keeps the few rows of A in shared memory,
// and splits K across the blocks of a thread-block cluster, the split-K idea
// of "CUDA 矩阵乘法优化：从朴素 Kernel 到接近 cuBLAS", section "10" -- but the
// partial sums are combined on chip instead of by a second reduction kernel.
// Three kernels share that plan: decode_outer_kernel (TMA-staged outer
// products, every shape whose A and B are 16-byte aligned with ld % 4 == 0;
// see there), decode_tma_kernel (A unaligned) and, for unaligned B, the
// plain-load kernel described here:
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
//    cluster owns and applies C = act(alpha*sum + beta*C + bias) (C read only
//    if beta != 0).
#include <cooperative_groups.h>

#include <atomic>
#include <cmath>

#include "common.cuh"

namespace cg = cooperative_groups;

// Packed two-lane FMAs and per-warp transposed A (see decode_outer_kernel):
// *_16 for the 16-row tile (M = 9..16), the others for M <= 8.
#ifndef DECODE_PACKED
#define DECODE_PACKED 0
#endif
#ifndef DECODE_PACKED_16
#define DECODE_PACKED_16 1
#endif

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

// acc[m][c] += A[m][k] * B[k][col + c] for one k row: a is the K-major A row
// (MT values), b the lane's four columns.
template <int MT>
__device__ __forceinline__ void fma_row(float (&acc)[MT][4], const float *__restrict__ a,
                                        const float4 &b) {
    float am[MT];
    if constexpr (MT >= 4) {
#pragma unroll
        for (int m4 = 0; m4 < MT / 4; ++m4) {
            const float4 av = *reinterpret_cast<const float4 *>(a + 4 * m4);
            am[4 * m4 + 0] = av.x;
            am[4 * m4 + 1] = av.y;
            am[4 * m4 + 2] = av.z;
            am[4 * m4 + 3] = av.w;
        }
    } else {
#pragma unroll
        for (int m = 0; m < MT; ++m) am[m] = a[m];
    }
    const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[m][c] = fmaf(am[m], bv[c], acc[m][c]);
}

template <int MT, bool VEC>
__global__ void __launch_bounds__(DTHREADS)
decode_kernel(int M, int64_t N, int64_t K, Epilogue ep, const float *__restrict__ A, int64_t lda,
              const float *__restrict__ B, int64_t ldb, float *__restrict__ C,
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
            const float v = ep.alpha * s;
            *p = epilogue_tail(ep, (ep.beta != 0.0f) ? fmaf(ep.beta, *p, v) : v, gn);
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
    return cudaLaunchKernelEx(&cfg, kern, (int)g.M, (int64_t)g.N, (int64_t)g.K, g.epi(), g.A,
                              g.lda, g.B, g.ldb, g.C, g.ldc, kslice);
}

// ---------------------------------------------------------------- TMA-streamed variant
// B 16-byte aligned with ldb % 4 == 0: B panels of TKB rows x
// (128*TNV) columns stream through a TSTAGES-deep ring of 2-D TMA copies (one
// "full" mbarrier per stage), so every block keeps TSTAGES-1 panels in flight
// independently of its arithmetic.  Each lane owns TNV float4 column groups
// (columns lane*4 + 128*v), so each broadcast A value it loads from shared
// memory feeds 4*TNV FFMAs: at M = 16 the shared-memory bytes per byte of B
// fall from 5 (one float4 per lane) to 3.  Each of the DW warps reads rows
// warp, warp+DW, ... of a panel; the last warp to release a stage issues the
// copy that refills it (as in the FFMA kernel).  A's K-slice is staged K-major
// in shared memory in chunks of KCH rows.  The reduction over warps and over
// the cluster is the same fixed-order one as above.
#ifndef DECODE_TKB
#define DECODE_TKB 32
#endif
#ifndef DECODE_MINB
#define DECODE_MINB 1
#endif
constexpr int TKB = DECODE_TKB;   // rows of B per stage
constexpr uint64_t DRAIN_NS = 1000000000ull;

template <int MT, int TNV, int DW, int TSTAGES>
struct TmaCfg {
    static constexpr int COLS = 128 * TNV;                                  // columns per cluster
    static constexpr int THREADS = DW * 32;
    static constexpr size_t B_STAGE = (size_t)TKB * COLS;                   // floats
    static constexpr size_t B_RING = TSTAGES * B_STAGE;                     // floats
    static constexpr size_t RED = (size_t)DW * MT * COLS;                   // floats, aliases the ring
    static constexpr size_t REGION0 = B_RING > RED ? B_RING : RED;
    static constexpr size_t AS = (size_t)KCH * MT;                          // floats
    static constexpr size_t PART = (size_t)MT * COLS;                       // floats
    static constexpr size_t FLOATS = REGION0 + AS + PART;
    static constexpr size_t BYTES = 128 + FLOATS * 4 + TSTAGES * 16;
    static_assert(KCH % TKB == 0 && TKB % DW == 0, "A chunks hold whole B panels");
    static_assert(COLS <= 256, "TMA box is at most 256 elements wide");
    static_assert(BYTES <= 227 * 1024, "shared memory per block");
};

template <class T, int MT, int TNV, int DW, int TSTAGES>
__global__ void __launch_bounds__(DW * 32, DECODE_MINB)
decode_tma_kernel(const __grid_constant__ CUtensorMap tmB, int M, int64_t N, int64_t K,
                  Epilogue ep, const float *__restrict__ A, int64_t lda,
                  float *__restrict__ C, int64_t ldc, int64_t kslice, unsigned *err,
                  uint64_t wait_ns) {
    using L = T;
    constexpr int COLS = L::COLS;
    extern __shared__ unsigned char smem_raw[];
    float *smem = reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                            ~uintptr_t(127));
    float *sB = smem;                      // [TSTAGES][TKB][COLS]
    float *red = smem;                     // [DW][MT][COLS], after the K loop
    float *As = smem + L::REGION0;         // [KCH][MT]
    float *part = As + L::AS;              // [MT][COLS]
    uint64_t *full = reinterpret_cast<uint64_t *>(part + L::PART);
    unsigned *arrived = reinterpret_cast<unsigned *>(full + TSTAGES);
    int *issued = reinterpret_cast<int *>(arrived + TSTAGES);

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int ks = (int)cluster.num_blocks();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t n0 = (int64_t)blockIdx.y * COLS;
    const int64_t kbeg = (int64_t)rank * kslice;
    const int64_t kend = (kbeg + kslice < K) ? kbeg + kslice : K;
    const int nst = kend > kbeg ? (int)((kend - kbeg + TKB - 1) / TKB) : 0;

    auto issue = [&](int st) {
        const int s = st % TSTAGES;
        issued[s] = st;
        const uint32_t fb = smem_u32(&full[s]);
        mbar_arrive_expect_tx(fb, (uint32_t)(L::B_STAGE * 4));
        tma_load_2d(smem_u32(sB + s * L::B_STAGE), &tmB, fb, (int32_t)n0,
                    (int32_t)(kbeg + (int64_t)st * TKB));
    };
    auto drain = [&]() {
        for (int s = 0; s < TSTAGES; ++s) {
            const int st = *reinterpret_cast<volatile int *>(&issued[s]);
            if (st >= 0) mbar_wait(smem_u32(&full[s]), (st / TSTAGES) & 1, DRAIN_NS);
        }
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < TSTAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            arrived[s] = 0;
            issued[s] = -1;
        }
        mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmB);
        for (int st = 0; st < TSTAGES && st < nst; ++st) issue(st);
    }

    float acc[TNV][MT][4];
#pragma unroll
    for (int v = 0; v < TNV; ++v)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[v][m][0] = acc[v][m][1] = acc[v][m][2] = acc[v][m][3] = 0.0f;
    bool failed = false;

    for (int st = 0; st < nst; ++st) {
        const int64_t kc = kbeg + (int64_t)st * TKB;
        const int64_t chunk0 = kbeg + ((int64_t)st * TKB) / KCH * KCH;
        if (kc == chunk0) {
            // Next chunk of A, K-major: As[k - chunk0][m]; rows past kend are zero.
            __syncthreads();
            const int64_t clen64 = (kend - chunk0) < KCH ? (kend - chunk0) : KCH;
            const int clen = (int)clen64;
            for (int idx = threadIdx.x; idx < KCH * MT; idx += L::THREADS) {
                const int m = idx / KCH, kl = idx - m * KCH;
                As[kl * MT + m] = (m < M && kl < clen) ? A[(int64_t)m * lda + chunk0 + kl] : 0.0f;
            }
            __syncthreads();
        }
        const int s = st % TSTAGES;
        if (!failed && !mbar_wait(smem_u32(&full[s]), (st / TSTAGES) & 1, wait_ns)) {
            failed = true;
            if (lane == 0) {
                record_error(err, kErrWaitTimeout);
                drain();
            }
        }
        if (failed) continue;   // keep reaching the block barriers; skip the stage
        const float *bst = sB + s * L::B_STAGE + lane * 4;
        const float *ast = As + (kc - chunk0) * MT;
#pragma unroll
        for (int j = 0; j < TKB / DW; ++j) {
            const int r = warp + DW * j;
#pragma unroll
            for (int v = 0; v < TNV; ++v) {
                const float4 b = *reinterpret_cast<const float4 *>(bst + r * COLS + 128 * v);
                fma_row<MT>(acc[v], ast + r * MT, b);
            }
        }
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            if (atomicAdd(&arrived[s], 1u) == DW - 1) {
                arrived[s] = 0;
                if (st + TSTAGES < nst) {
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    issue(st + TSTAGES);
                }
            }
        }
    }

    // Sum over warps in a fixed order; the ring is free once every stage was
    // read.  (After a time-out, wait for any copy still in flight first.)
    if (threadIdx.x == 0) drain();
    const bool any_failed = __syncthreads_or(failed) != 0;
#pragma unroll
    for (int v = 0; v < TNV; ++v)
#pragma unroll
        for (int m = 0; m < MT; ++m)
            *reinterpret_cast<float4 *>(&red[((size_t)warp * MT + m) * COLS + 128 * v + lane * 4]) =
                make_float4(acc[v][m][0], acc[v][m][1], acc[v][m][2], acc[v][m][3]);
    __syncthreads();
    for (int o = threadIdx.x; o < MT * COLS; o += L::THREADS) {
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < DW; ++w) sum += red[(size_t)w * MT * COLS + o];
        part[o] = sum;
    }

    cluster.sync();
    const int per = (MT * COLS + ks - 1) / ks;
    const int obeg = rank * per;
    const int oend = (obeg + per < MT * COLS) ? obeg + per : MT * COLS;
    for (int o = obeg + threadIdx.x; o < oend; o += L::THREADS) {
        // the (up to 8) remote loads are independent: issue them together,
        // then add in rank order
        float pv[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) pv[q] = q < ks ? cluster.map_shared_rank(part, q)[o] : 0.0f;
        float sum = 0.0f;
#pragma unroll
        for (int q = 0; q < 8; ++q) sum += pv[q];
        const int m = o / COLS;
        const int64_t gn = n0 + (o - m * COLS);
        if (!any_failed && m < M && gn < N) {
            float *p = C + (int64_t)m * ldc + gn;
            const float v = ep.alpha * sum;
            *p = epilogue_tail(ep, (ep.beta != 0.0f) ? fmaf(ep.beta, *p, v) : v, gn);
        }
    }
    cluster.sync();
}

// acc[j] += a * b[j] for j < 8; `rev` walks the columns backwards
// (alternating rows keep operands of neighbouring FMAs apart).  PACKED: two
// FP32 lanes per instruction, `a` duplicated into a register pair (each lane
// one fused multiply-add rounded once, as fmaf).
template <bool PACKED>
__device__ __forceinline__ void fma_row8(float (&acc)[8], float a, const float (&b)[8], bool rev) {
    if constexpr (!PACKED) {
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
            const int j = rev ? 7 - jj : jj;
            acc[j] = fmaf(a, b[j], acc[j]);
        }
        return;
    }
    const float2 a2 = make_float2(a, a);
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
        const int q = rev ? 3 - qq : qq;
        const float2 d = __ffma2_rn(a2, make_float2(b[2 * q], b[2 * q + 1]),
                                    make_float2(acc[2 * q], acc[2 * q + 1]));
        acc[2 * q] = d.x;
        acc[2 * q + 1] = d.y;
    }
}

// ---------------------------------------------------------------- outer-product variant (M >= 5)
// A block owns an MT x 256 tile of C.  Each stage of its TMA ring carries
// both operands of TKB k-steps: the TKB x 256 panel of B ([k][n]) and
// the MT x TKB panel of A ([m][k], rows past M zero-filled by the copy),
// so the K loop has no block barrier and no global load of its own.  Needs
// A and B 16-byte aligned with lda % 4 == 0 and ldb % 4 == 0.
//
// The four warps split the tile into RG row groups and every stage's k-steps
// into KG = 4/RG interleaved k groups.  A lane owns the MT/RG rows of its
// row group and eight columns (lane*4 + {0..3} and 128 + lane*4 + {0..3}):
// an (MT/RG) x 8 outer product per k.  Per k a lane loads 8 floats of B (two
// 128-bit loads) and MT/RG broadcast floats of A, so shared memory delivers
// (MT/RG + 8) floats per lane for 8*MT/RG FFMAs: 0.25 wavefronts per FFMA
// at MT/RG = 8, against 0.375 with 4 rows per lane.  At M = 16 a byte of B
// carries four FFMAs, so streaming B at the copy rate needs the FMA pipe
// about two thirds busy, and with 4 rows per lane the shared-memory pipe
// saturated first.
//
// After the K loop the k groups' partial tiles are summed in a fixed order
// in shared memory, then across the cluster.
//
// The kernel is launched as a programmatic dependent of whatever precedes it
// on the stream: its blocks may become resident and initialise their
// barriers while that work finishes, and wait (pdl_wait) before the first
// copy.  Once past its K loop a block lets the next such kernel launch, so
// back-to-back decode products (a model's layers) overlap one kernel's
// reduction with the next one's launch.
#ifndef DECODE_PDL
#define DECODE_PDL 1   // programmatic dependent launch of the outer-product tile
#endif
#ifndef DECODE_DO_TKB
#define DECODE_DO_TKB 16      // k-steps per TMA stage, 8-row tile
#endif
#ifndef DECODE_DO_TKB_16
#define DECODE_DO_TKB_16 16   // k-steps per TMA stage, 16-row tile
#endif
constexpr int DO_COLS = 256, DO_WARPS = 4, DO_THREADS = DO_WARPS * 32;
#ifndef DECODE_DO_STAGES
#define DECODE_DO_STAGES 2      // TMA stages of the 8-row tile
#endif
#ifndef DECODE_DO_STAGES_16
#define DECODE_DO_STAGES_16 3   // TMA stages of the 16-row tile
#endif
#ifndef DECODE_DO_MINB
#define DECODE_DO_MINB 0   // blocks per SM the registers are sized for; 0: by row count
#endif
#ifndef DECODE_DO_KS
#define DECODE_DO_KS 0
#endif
#ifndef DECODE_AT
#define DECODE_AT 0
#endif
#ifndef DECODE_AT_16
#define DECODE_AT_16 1
#endif
constexpr int DO_KSMAX = 16;   // cluster size limit (16 is non-portable)

template <int MT, int RG>
struct DoCfg {
    // 64 accumulators per lane at MT/RG = 8: five blocks per SM (96 registers)
    // suit M <= 8; at M = 16, four blocks (128 registers) measured faster.
    static constexpr int MINB = DECODE_DO_MINB > 0 ? DECODE_DO_MINB : (MT <= 8 ? 5 : 4);
    // Stages: at four blocks per SM the 16-row tile has room for a third
    // (measured 4.82 -> 4.98 TB/s at M = 16); a third stage would cost the
    // 8-row tile its fifth block (5.99 -> 5.48 at M = 8).
    static constexpr int STAGES = MT > 8 ? DECODE_DO_STAGES_16 : DECODE_DO_STAGES;
    static constexpr int TKB = MT > 8 ? DECODE_DO_TKB_16 : DECODE_DO_TKB;   // a multiple of 4 (TMA x)
    static constexpr int KG = DO_WARPS / RG;                               // k groups
    static constexpr int MTL = MT / RG;                                    // rows per lane
    static constexpr int RPW = TKB / KG;                                // k-steps per warp per stage
    static constexpr size_t B_PANEL = (size_t)TKB * DO_COLS;            // floats, [k][n]
    static constexpr size_t A_PANEL = (size_t)MT * TKB;                 // floats, [m][k]
    static constexpr size_t STAGE = B_PANEL + A_PANEL;
    static constexpr size_t RING = STAGES * STAGE;
    static constexpr size_t RED = (size_t)KG * MT * DO_COLS;              // aliases the ring
    static constexpr size_t REGION0 = RING > RED ? RING : RED;
    // The 16-row tile: each warp transposes its A values of a stage to [k][m]
    // (128-bit A loads, a third fewer instructions per k-step) and uses
    // packed FMAs; measured at M = 16, eager: 4.42 TB/s scalar, 4.52 with
    // both; at M = 8 either costs 1-4%.
    static constexpr bool TRANSPOSE_A = MT > 8 ? DECODE_AT_16 : DECODE_AT;
    static constexpr bool PACKED = MT > 8 ? DECODE_PACKED_16 : DECODE_PACKED;
    static constexpr size_t AT = TRANSPOSE_A ? (size_t)DO_WARPS * RPW * MTL : 0;   // [warp][k][m]
    static constexpr size_t BYTES = 128 + (REGION0 + AT) * 4 + STAGES * 16;
    static_assert(DO_WARPS % RG == 0 && MT % RG == 0 && TKB % KG == 0 && TKB % 4 == 0, "warp split");
    static_assert(!TRANSPOSE_A || (RPW * MTL) % 32 == 0, "whole lanes in the A transpose");
    static_assert(MTL % 4 == 0, "A rows come in float4 groups");
    static_assert((STAGE * 4) % 128 == 0, "stage offsets stay 128-byte aligned");
    static_assert((MT * DO_COLS) % (4 * DO_THREADS) == 0, "whole float4 sweeps in the group sum");
};

template <int MT, int RG>
__global__ void __launch_bounds__(DO_THREADS, DoCfg<MT, RG>::MINB)
decode_outer_kernel(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmA,
                    int M, int64_t N, int64_t K, Epilogue ep, float *__restrict__ C,
                    int64_t ldc, int64_t kslice, unsigned *err, uint64_t wait_ns) {
    using L = DoCfg<MT, RG>;
    constexpr int KG = L::KG, MTL = L::MTL, DO_STAGES = L::STAGES, TKB = L::TKB;
    extern __shared__ unsigned char smem_raw[];
    float *smem = reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                            ~uintptr_t(127));
    float *ring = smem;                    // [STAGES][B panel | A panel]
    float *red = smem;                     // [KG][MT][DO_COLS], after the K loop
    float *at = smem + L::REGION0 + (size_t)(threadIdx.x >> 5) * L::RPW * MTL;   // this warp's A^T
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::REGION0 + L::AT);
    unsigned *arrived = reinterpret_cast<unsigned *>(full + DO_STAGES);
    int *issued = reinterpret_cast<int *>(arrived + DO_STAGES);

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int ks = (int)cluster.num_blocks();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rg = warp / KG, kg = warp % KG;
    const int64_t n0 = (int64_t)blockIdx.y * DO_COLS;
    const int64_t kbeg = (int64_t)rank * kslice;
    const int64_t kend = (kbeg + kslice < K) ? kbeg + kslice : K;
    const int nst = kend > kbeg ? (int)((kend - kbeg + TKB - 1) / TKB) : 0;

    auto issue = [&](int st) {
        const int s = st % DO_STAGES;
        issued[s] = st;
        const uint32_t fb = smem_u32(&full[s]);
        const int32_t kc = (int32_t)(kbeg + (int64_t)st * TKB);
        float *stg = ring + s * L::STAGE;
        mbar_arrive_expect_tx(fb, (uint32_t)(L::STAGE * 4));
        tma_load_2d(smem_u32(stg), &tmB, fb, (int32_t)n0, kc);
        tma_load_2d(smem_u32(stg + L::B_PANEL), &tmA, fb, kc, 0);
    };
    auto drain = [&]() {
        for (int s = 0; s < DO_STAGES; ++s) {
            const int st = *reinterpret_cast<volatile int *>(&issued[s]);
            if (st >= 0) mbar_wait(smem_u32(&full[s]), (st / DO_STAGES) & 1, DRAIN_NS);
        }
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < DO_STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            arrived[s] = 0;
            issued[s] = -1;
        }
        mbar_fence_init();
    }
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmA);
    }
#if DECODE_PDL
    // Launched as a programmatic dependent of the work before it on the
    // stream: everything above overlaps that work's tail; A, B and C are
    // touched only after it has completed.
    pdl_wait();
#endif
    __syncthreads();
    if (threadIdx.x == 0)
        for (int st = 0; st < DO_STAGES && st < nst; ++st) issue(st);

    float acc[MTL][8];
#pragma unroll
    for (int m = 0; m < MTL; ++m)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[m][j] = 0.0f;
    bool failed = false;

    for (int st = 0; st < nst; ++st) {
        const int s = st % DO_STAGES;
        if (!mbar_wait(smem_u32(&full[s]), (st / DO_STAGES) & 1, wait_ns)) {
            failed = true;
            if (lane == 0) {
                record_error(err, kErrWaitTimeout);
                drain();
            }
            break;
        }
        const float *stg = ring + s * L::STAGE;
        const float *bst = stg + lane * 4;
        const float *ast = stg + L::B_PANEL + (size_t)rg * MTL * TKB;
        if constexpr (L::TRANSPOSE_A) {
            // this warp's A values of the stage, transposed to [k][m] so that
            // a k-step's MTL values are float4 loads
#pragma unroll
            for (int e = lane; e < L::RPW * MTL; e += 32) {
                const int rr = e / MTL, m = e % MTL;
                at[e] = ast[m * TKB + kg + KG * rr];
            }
            __syncwarp();
        }
#pragma unroll
        for (int rr = 0; rr < L::RPW; ++rr) {
            const int r = kg + KG * rr;
            const float4 b0 = *reinterpret_cast<const float4 *>(bst + r * DO_COLS);
            const float4 b1 = *reinterpret_cast<const float4 *>(bst + r * DO_COLS + 128);
            const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
            if constexpr (L::TRANSPOSE_A) {
                float av[MTL];
#pragma unroll
                for (int q = 0; q < MTL / 4; ++q) {
                    const float4 a4 = *reinterpret_cast<const float4 *>(at + rr * MTL + 4 * q);
                    av[4 * q] = a4.x;
                    av[4 * q + 1] = a4.y;
                    av[4 * q + 2] = a4.z;
                    av[4 * q + 3] = a4.w;
                }
#pragma unroll
                for (int m = 0; m < MTL; ++m) fma_row8<L::PACKED>(acc[m], av[m], bv, m & 1);
            } else {
#pragma unroll
                for (int m = 0; m < MTL; ++m)
                    fma_row8<L::PACKED>(acc[m], ast[m * TKB + r], bv, m & 1);
            }
        }
        if constexpr (L::TRANSPOSE_A) __syncwarp();   // lanes are done with `at` before it is rewritten
        __syncwarp();
        if (lane == 0) {
            // release: this warp's reads of the stage happen before its arrival;
            // acquire: the last warp to arrive sees every other warp's release
            // before it lets the copy engine overwrite the stage
            unsigned prev;
            asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;"
                         : "=r"(prev)
                         : "r"(smem_u32(&arrived[s]))
                         : "memory");
            if (prev == DO_WARPS - 1) {
                arrived[s] = 0;
                if (st + DO_STAGES < nst) {
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    issue(st + DO_STAGES);
                }
            }
        }
    }

    if (threadIdx.x == 0) drain();
    const bool any_failed = __syncthreads_or(failed) != 0;
#if DECODE_PDL
    // the next kernel on the stream may launch once every block is here (it
    // waits for this grid to complete before touching memory)
    pdl_trigger();
#endif
    // k-group partials to shared memory (the ring is free now), then their
    // sum in k-group order into group 0's slot.
#pragma unroll
    for (int m = 0; m < MTL; ++m) {
        float *pr = red + ((size_t)kg * MT + rg * MTL + m) * DO_COLS + lane * 4;
        *reinterpret_cast<float4 *>(pr) = make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
        *reinterpret_cast<float4 *>(pr + 128) = make_float4(acc[m][4], acc[m][5], acc[m][6], acc[m][7]);
    }
    __syncthreads();
    constexpr int TOTAL4 = MT * DO_COLS / 4;
    if constexpr (KG > 1) {
#pragma unroll
        for (int it = 0; it < TOTAL4 / DO_THREADS; ++it) {
            const int o4 = threadIdx.x + it * DO_THREADS;
            float4 v = reinterpret_cast<const float4 *>(red)[o4];
#pragma unroll
            for (int w = 1; w < KG; ++w) {
                const float4 u = reinterpret_cast<const float4 *>(red + (size_t)w * MT * DO_COLS)[o4];
                v.x += u.x; v.y += u.y; v.z += u.z; v.w += u.w;
            }
            reinterpret_cast<float4 *>(red)[o4] = v;
        }
    }
    cluster.sync();
    // Block `rank` finishes float4 groups [rank*per4, (rank+1)*per4) of the
    // cluster's MT x 256 tile: the ks partials in rank order, then alpha/beta.
    const int per4 = (TOTAL4 + ks - 1) / ks;
    const int obeg = rank * per4;
    const int oend = (obeg + per4 < TOTAL4) ? obeg + per4 : TOTAL4;
    for (int o4 = obeg + threadIdx.x; o4 < oend; o4 += DO_THREADS) {
        // four remote loads in flight at a time; the sum stays in rank order
        float4 sum = reinterpret_cast<const float4 *>(cluster.map_shared_rank(red, 0))[o4];
        for (int q0 = 1; q0 < ks; q0 += 4) {
            float4 pv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (q0 + u < ks)
                    pv[u] = reinterpret_cast<const float4 *>(cluster.map_shared_rank(red, q0 + u))[o4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (q0 + u < ks) {
                    sum.x += pv[u].x; sum.y += pv[u].y; sum.z += pv[u].z; sum.w += pv[u].w;
                }
        }
        const int m = (4 * o4) / DO_COLS;
        const int64_t gn = n0 + (4 * o4 - m * DO_COLS);
        if (!any_failed && m < M) {
            const float sv[4] = {sum.x, sum.y, sum.z, sum.w};
            float *p = C + (int64_t)m * ldc + gn;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (gn + e < N) {
                    const float v = ep.alpha * sv[e];
                    p[e] = epilogue_tail(ep, (ep.beta != 0.0f) ? fmaf(ep.beta, p[e], v) : v, gn + e);
                }
            }
        }
    }
    cluster.sync();
}

// Cluster size: K split over ks blocks (<= 8, a portable cluster), chosen so
// the grid fills whole waves of resident blocks as nearly as possible.
inline int choose_ks(int64_t K, int64_t ncb, int slots) {
    int best = 1;
    double best_eff = -1.0;
    for (int ks = 1; ks <= 8; ks *= 2) {
        if (ks > 1 && K / ks < TKB) break;
        const double waves = (double)(ncb * ks) / slots;
        const double eff = waves / std::ceil(waves);
        // more blocks hide latency better, so prefer larger ks unless clearly worse
        if (eff > best_eff + 0.02 || (eff > best_eff - 0.02 && ks > best)) {
            best = ks;
            best_eff = eff > best_eff ? eff : best_eff;
        }
    }
    return best;
}

template <int MT, int TNV, int DW, int TSTAGES>
cudaError_t launch_tma(const GemmArgs &g) {
    using L = TmaCfg<MT, TNV, DW, TSTAGES>;
    alignas(64) CUtensorMap tmB;
    if (!encode_tma_2d(g.encode, &tmB, g.B, g.N, g.K, g.ldb, L::COLS, TKB, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    auto kern = decode_tma_kernel<L, MT, TNV, DW, TSTAGES>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::BYTES);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, L::THREADS, L::BYTES);
    if (e != cudaSuccess) return e;
    const int64_t ncb = (g.N + L::COLS - 1) / L::COLS;
    if (ncb > 65535) return cudaErrorInvalidConfiguration;
    const int ks = choose_ks(g.K, ncb, (per_sm > 0 ? per_sm : 1) * (g.sm_count > 0 ? g.sm_count : 148));
    int64_t kslice = (g.K + ks - 1) / ks;
    kslice = (kslice + TKB - 1) / TKB * TKB;   // whole panels per block

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ks, (unsigned)ncb, 1);
    cfg.blockDim = dim3(L::THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::BYTES;
    cfg.stream = g.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmB, (int)g.M, (int64_t)g.N, (int64_t)g.K, g.epi(), g.A,
                              g.lda, g.C, g.ldc, kslice, g.err, g.wait_ns);
}

#ifndef DECODE_TNV
#define DECODE_TNV 2
#endif
#ifndef DECODE_DW
#define DECODE_DW 8
#endif
#ifndef DECODE_OUTER_MIN_M
#define DECODE_OUTER_MIN_M 1
#endif
#ifndef DECODE_STAGES
#define DECODE_STAGES 3
#endif
#ifndef DECODE_TMA_MIN_M
#define DECODE_TMA_MIN_M 1
#endif

// Largest number of clusters of `ks` blocks of `kern` the GPU holds at once,
// cached per device and cluster size (0: this cluster size cannot launch).
template <typename Kern>
int max_clusters(Kern kern, int ks, cudaLaunchConfig_t cfg, std::atomic<int> (&cache)[64][17]) {
    int dev = 0;
    if (ks < 1 || ks > 16 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    const int hit = cache[dev][ks].load(std::memory_order_relaxed);
    if (hit > 0) return hit - 1;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)ks, 1, 1);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
    }
    cache[dev][ks].store(n + 1, std::memory_order_relaxed);
    return n;
}

// Cluster size for a K split over the blocks of a cluster: among sizes
// 1..ksmax that leave each block at least `min_k` k-steps, the one whose
// grid (ncb clusters) fills its waves best; within 2% of the best, the
// largest (more blocks in flight hide more memory latency).
template <typename Kern>
int choose_cluster(Kern kern, int64_t K, int64_t ncb, int ksmax, int min_k, const cudaLaunchConfig_t &cfg,
                   std::atomic<int> (&cache)[64][17]) {
    int ks = 1;
    double best_eff = -1.0;
    for (int c = 1; c <= ksmax; ++c) {
        if (c > 1 && K / c < min_k) break;
        const int nclu = max_clusters(kern, c, cfg, cache);
        if (nclu <= 0) continue;
        const double waves = (double)ncb / nclu;
        const double eff = waves / std::ceil(waves);
        if (eff > best_eff + 0.02 || (eff > best_eff - 0.02 && c > ks)) {
            ks = c;
            best_eff = eff > best_eff ? eff : best_eff;
        }
    }
    return ks;
}

template <int MT, int RG>
cudaError_t launch_outer(const GemmArgs &g) {
    using L = DoCfg<MT, RG>;
    static std::atomic<int> cache[64][17];
    alignas(64) CUtensorMap tmB, tmA;
    if (!encode_tma_2d(g.encode, &tmB, g.B, g.N, g.K, g.ldb, DO_COLS, L::TKB, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    if (!encode_tma_2d(g.encode, &tmA, g.A, g.K, g.M, g.lda, L::TKB, MT, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    auto kern = decode_outer_kernel<MT, RG>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::BYTES);
    if (e != cudaSuccess) return e;
    int ksmax = 8;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess)
        ksmax = DO_KSMAX;
    else
        (void)cudaGetLastError();
    const int64_t ncb = (g.N + DO_COLS - 1) / DO_COLS;
    if (ncb > 65535) return cudaErrorInvalidConfiguration;

    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(DO_THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::BYTES;
    cfg.stream = g.stream;
    int ks = choose_cluster(kern, g.K, ncb, ksmax, L::TKB, cfg, cache);
    if (DECODE_DO_KS > 0 && g.K >= (int64_t)DECODE_DO_KS * L::TKB) ks = DECODE_DO_KS;
    int64_t kslice = (g.K + ks - 1) / ks;
    kslice = (kslice + L::TKB - 1) / L::TKB * L::TKB;

    cfg.gridDim = dim3((unsigned)ks, (unsigned)ncb, 1);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = DECODE_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, tmB, tmA, (int)g.M, (int64_t)g.N, (int64_t)g.K, g.epi(),
                              g.C, g.ldc, kslice, g.err, g.wait_ns);
}

template <int MT>
cudaError_t launch_vec(const GemmArgs &g) {
    if (g.M >= DECODE_OUTER_MIN_M && ((reinterpret_cast<uintptr_t>(g.B) & 15) == 0) &&
        (g.ldb % 4 == 0) && ((reinterpret_cast<uintptr_t>(g.A) & 15) == 0) && (g.lda % 4 == 0)) {
        // fewer than 8 rows run the 8-row tile (the copy zero-fills the rows past M)
        if constexpr (MT <= 8)
            return launch_outer<8, 1>(g);
        else
            return launch_outer<MT, 2>(g);
    }
    const bool vec = ((reinterpret_cast<uintptr_t>(g.B) & 15) == 0) && (g.ldb % 4 == 0);
    if (vec && g.M >= DECODE_TMA_MIN_M)
        return launch_tma<MT, DECODE_TNV, DECODE_DW, DECODE_STAGES>(g);
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
