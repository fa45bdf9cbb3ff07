// tf32x3.cu -- FP32-accurate GEMM on the tcgen05 tensor cores (3xTF32).
//
// Each operand element x is split into two TF32 numbers,
//     hi = tf32(x)   and   lo = tf32(x - hi)   (round to nearest),
// so x = hi + lo up to the 2^-22 relative error of lo; the product is
// accumulated as  hi*hi + hi*lo + lo*hi  in FP32 (the lo*lo term, below
// FP32 precision, is dropped) -- the error-compensated "3xTF32" split of
// Ootomo and Yokota (2022).  The pages only name tensor cores and TF32
// ("CUDA 矩阵乘法优化：从朴素 Kernel 到接近 cuBLAS", results-table note;
// "GPU GEMM 优化完全拆解（一）", series outline); this kernel is the FP32-accuracy
// tensor path the benchmark asks for.
//
// Two passes:
//  1. split kernels (memory-bound) write A_hi, A_lo as [M][K] and B_hi, B_lo
//     transposed as [N][K] into the workspace, so both MMA operands are
//     K-major -- the canonical UMMA layout;
//  2. the MMA kernel, persistent (one CTA per SM walking its tiles), on one
//     SM per 128 x 256 tile (tf32_mma_kernel) or, for M >= 256, on a pair of
//     SMs per 256 x 256 tile with tcgen05 cta_group::2 (tf32_mma2_kernel, see
//     there).  Warp 8 streams 16-wide K slices of the four operand tiles into
//     a shared-memory ring with TMA (64-byte swizzle; the one-term kinds below
//     stream 128-byte K rows with the 128-byte swizzle); one thread of warp 9
//     issues, per 8-wide k step, three tcgen05.mma kind::tf32 (hi*lo, lo*hi,
//     hi*hi) into an FP32 accumulator of 128 lanes x 256 columns in tensor
//     memory and releases each stage with tcgen05.commit; warps 0-7 read the
//     accumulator back with tcgen05.ld (each warp 32 lanes = rows, half the
//     columns), add it into FP32 registers chunk by chunk (see
//     tf32_mma_kernel) and finally apply C = alpha*acc + beta*C, reading C
//     only when beta != 0.
//
// Every wait is bounded.  On a time-out the kernel records the error, waits
// (bounded) for its own TMA copies and MMAs in flight, frees its tensor
// memory and exits without storing.
#include <cuda_bf16.h>

#include <atomic>

#include "common.cuh"

namespace sgemm_gb300 {
namespace {

constexpr int TBM = 128, TBN = 256;
#ifndef TF_KC3
#define TF_KC3 6
#endif
// 3xTF32: k-tiles per accumulation chunk (96 k).  Shorter chunks keep the
// tensor-memory accumulation error lower but make the MMAs wait for the
// epilogue warps of both SMs between chunks; measured at 8192^3 (two-SM
// tiles): 64 k 290 TFLOP/s, 96 k 321, 128 k 327, with the mean relative
// error 4.7e-7 at 64 k and 9.1e-7 at 128 k (FP32 FFMA: 2e-7 .. 4e-7).
constexpr int KC_TILES = TF_KC3;
// One-term kinds: 1024 k (TF32) / 2048 k (BF16) per chunk.  A 64 k chunk is
// only 8 MMAs, about as long as the epilogue warps take to drain a 128 x 256
// accumulator from tensor memory, so the MMAs waited on the drain.  Measured
// at 8192^3 (TFLOP/s / normwise error against the rounded-operand product,
// TF32 and BF16): 64 k 463 / 1.0e-8 and 814 / 7e-9; 256 k 557 / 1.5e-8 and
// 959 / 9e-9 (64-byte rows, one CTA per tile); persistent, 128-byte rows:
// 256 k 718 and 1240, 512 k 741 / 2.4e-8 and 1282 / 1.7e-8; two-SM tiles:
// 512 k 767 and 1286, 1024 k 807 / 4.4e-8 and 1364 / 4.1e-8.
#ifndef TF_KC1
#define TF_KC1 64   // in 64-byte k-tiles (1024 k TF32, 2048 k BF16); scaled to the row width used
#endif
// Swizzle span (= bytes of K per operand row of a stage) of the one-term
// kinds.  128-byte rows move each stage in half as many TMA requests as
// 64-byte rows; the one-term kinds are bound by operand delivery, the
// 3-term kind by the tensor pipe, so only the former use them.
#ifndef TF_SW1
#define TF_SW1 128
#endif
#ifndef TF_PAIR
#define TF_PAIR 1   // two-SM (cta_group::2) tiles for M >= 256
#endif
#ifndef TF_PERSIST
#define TF_PERSIST 1
#endif
#ifndef TF_SW3
#define TF_SW3 64   // measured at 8192^3: 128-byte rows (two 96 KB stages) 271 vs 297 TFLOP/s
#endif
constexpr int EPI_WARPS = 8;                    // two warpgroups: 32 rows x 128 columns each
constexpr int PRODUCER_WARP = EPI_WARPS, MMA_WARP = EPI_WARPS + 1;
constexpr int THREADS = (EPI_WARPS + 2) * 32;
constexpr int EPI_COLS = TBN / (EPI_WARPS / 4); // columns per epilogue thread
constexpr int RASTER_GROUP = 16;                // M tiles walked together (L2 reuse)
constexpr uint32_t TMEM_COLS = 2 * TBN;                    // two 128 x 256 FP32 accumulators

// Per-stage layout: the A parts, then the B parts (hi, then lo for 3 terms),
// each tile rows x SWB bytes of K.  3 terms (64-byte rows): 48 KB stages, 4
// deep; 1 term (128-byte rows): 48 KB stages, 4 deep (192 KB both).
// Operand kinds: FP32 bit patterns read as TF32 (kind::tf32), or BF16
// (kind::f16 with both operands BF16).
enum : int { kTf32 = 0, kBf16 = 1 };

template <int TERMS, int KIND = kTf32>
struct TfCfg {
    static constexpr int PARTS = TERMS == 3 ? 2 : 1;
    static constexpr int SWB = TERMS == 3 ? TF_SW3 : TF_SW1;      // bytes of K per tile row
    static constexpr uint32_t A_TILE = TBM * SWB, B_TILE = TBN * SWB;
    static constexpr uint32_t STAGE_BYTES = PARTS * (A_TILE + B_TILE);
    static constexpr int TSTG = (192 * 1024) / STAGE_BYTES;
    static constexpr size_t SMEM = 1024 + (size_t)TSTG * STAGE_BYTES + 256;
    // K elements in one row of a tile, and per MMA instruction (32 bytes)
    static constexpr int KT = KIND == kTf32 ? SWB / 4 : SWB / 2;
    static constexpr int MMA_K = KIND == kTf32 ? 8 : 16;
    // k-tiles per accumulation chunk: 64 k (3 terms), TF_KC1 64-byte k-tiles (1 term)
    static constexpr int KC = TERMS == 3 ? KC_TILES : TF_KC1 * 64 / SWB;
    static_assert(SWB == 64 || SWB == 128, "64- or 128-byte swizzle");
    static_assert(A_TILE % 1024 == 0 && B_TILE % 1024 == 0, "tiles keep 1024-byte alignment");
    static_assert(KC >= 1 && TSTG >= 2, "chunk and ring depth");
    static_assert(TERMS == 1 || TERMS == 3, "1xTF32 or 3xTF32");
    static_assert(KIND == kTf32 || TERMS == 1, "BF16 is one term");
    static_assert(SMEM <= 227 * 1024, "shared memory per block");
};
constexpr uint64_t DRAIN_NS = 1000000000ull;
static_assert(EPI_WARPS % 4 == 0 && EPI_COLS % 16 == 0, "epilogue covers all lanes and columns");

// Instruction descriptor of tcgen05.mma kind::tf32: D format F32 (bits 4-5 = 1),
// A and B format TF32 (bits 7-9 and 10-12 = 2), both K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t IDESC = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(TBN >> 3) << 17) |
                           ((uint32_t)(TBM >> 4) << 24);
// kind::f16 with BF16 operands: the same fields, A and B format BF16 (1),
// both taken from one constant so that they can never differ.
constexpr uint32_t BF16_FORMAT = 1;
constexpr uint32_t IDESC_BF16 = (1u << 4) | (BF16_FORMAT << 7) | (BF16_FORMAT << 10) |
                                ((uint32_t)(TBN >> 3) << 17) | ((uint32_t)(TBM >> 4) << 24);

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with the SWB-byte swizzle: rows of SWB bytes, 8-row core groups 8*SWB
// bytes apart (stride byte offset), descriptor version 1, layout
// SWIZZLE_64B (4) or SWIZZLE_128B (2).  A k-offset inside the row is added
// to the start address; the swizzle is a function of the address bits.
template <int SWB>
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
    static_assert(SWB == 64 || SWB == 128, "64- or 128-byte swizzle");
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);               // start address
    d |= (uint64_t)1 << 16;                                // leading byte offset (unused here)
    d |= (uint64_t)(((8u * SWB) >> 4) & 0x3FFFu) << 32;    // stride byte offset
    d |= (uint64_t)1 << 46;                                // version
    d |= (uint64_t)(SWB == 128 ? 2 : 4) << 61;             // layout
    return d;
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(IDESC), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(IDESC_BF16), "r"(accumulate)
        : "memory");
}

// The mbarrier completes once every tcgen05 operation this thread issued so far is done.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// One epilogue thread's row of a tile: C[gm][gn0 .. gn0 + EPI_COLS) =
// act(alpha*acc + beta*C + bias), C read only when beta != 0; rows past M
// and columns past N are skipped.
__device__ __forceinline__ void store_row(const float (&acc)[EPI_COLS], const Epilogue &ep,
                                          float *__restrict__ C, int64_t ldc, int gm, int gn0,
                                          int M, int N, int c_vec4) {
    if (gm >= M) return;
    const bool tail = ep.bias != nullptr || ep.act != kActNone;
    float *crow = C + (int64_t)gm * ldc;
#pragma unroll
    for (int q = 0; q < EPI_COLS / 4; ++q) {
        const int gn = gn0 + 4 * q;
        float o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) o[e] = ep.alpha * acc[4 * q + e];
        if (c_vec4 && gn + 3 < N) {
            float4 *p = reinterpret_cast<float4 *>(crow + gn);
            if (ep.beta != 0.0f) {
                const float4 cv = *p;
                o[0] = fmaf(ep.beta, cv.x, o[0]);
                o[1] = fmaf(ep.beta, cv.y, o[1]);
                o[2] = fmaf(ep.beta, cv.z, o[2]);
                o[3] = fmaf(ep.beta, cv.w, o[3]);
            }
            if (tail) {
#pragma unroll
                for (int e = 0; e < 4; ++e) o[e] = epilogue_tail(ep, o[e], gn + e);
            }
            *p = make_float4(o[0], o[1], o[2], o[3]);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (gn + e < N) {
                    float *p = crow + gn + e;
                    const float w = (ep.beta != 0.0f) ? fmaf(ep.beta, *p, o[e]) : o[e];
                    *p = tail ? epilogue_tail(ep, w, gn + e) : w;
                }
            }
        }
    }
}

// Chunked accumulation.  A tensor-core MMA adds its products into the FP32
// accumulator with an error of a fraction of an ulp of the accumulator, so a
// single accumulator over all of K loses accuracy linearly in K (measured:
// relative error 1.8e-6 at K = 256 growing to 5.7e-5 at K = 8192).  The MMA
// thread therefore restarts the accumulator every KC_TILES k-tiles, in two
// alternating tensor-memory buffers, and the epilogue warps add each chunk
// into FP32 registers (round to nearest) while the next chunk is computed.
template <int TERMS, int KIND>
__global__ void __launch_bounds__(THREADS, 1)
tf32_mma_kernel(const __grid_constant__ CUtensorMap tmAhi, const __grid_constant__ CUtensorMap tmAlo,
                const __grid_constant__ CUtensorMap tmBhi, const __grid_constant__ CUtensorMap tmBlo,
                int M, int N, int K, Epilogue ep, float *__restrict__ C, int64_t ldc,
                int c_vec4, unsigned *err, uint64_t wait_ns) {
    using L = TfCfg<TERMS, KIND>;
    constexpr int TSTG = L::TSTG;
    constexpr int KT = L::KT;
    constexpr uint32_t STAGE_BYTES = L::STAGE_BYTES;
    extern __shared__ unsigned char smem_raw[];
    const uintptr_t base = (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023);
    unsigned char *ring = reinterpret_cast<unsigned char *>(base);
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + (size_t)TSTG * STAGE_BYTES);
    uint64_t *empty = full + TSTG;
    uint64_t *cfull = empty + TSTG;     // [2] chunk in tensor memory buffer b is complete
    uint64_t *cempty = cfull + 2;       // [2] epilogue has read buffer b
    uint64_t *drainbar = cempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drainbar + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Persistent: CTA b takes tiles b, b + gridDim.x, ...  Grouped
    // rasterisation: RASTER_GROUP M-tiles x all N-tiles per group, so the
    // tiles in flight at one time share a few A and B panels through L2.
    const int num_m = (M + TBM - 1) / TBM, num_n = (N + TBN - 1) / TBN;
    const int tiles = num_m * num_n;
    const int per_group = RASTER_GROUP * num_n;
    auto tile_origin = [&](int t, int &m0, int &n0) {
        const int first_m = (t / per_group) * RASTER_GROUP;
        const int gsz = (num_m - first_m) < RASTER_GROUP ? (num_m - first_m) : RASTER_GROUP;
        m0 = (first_m + (t % per_group) % gsz) * TBM;
        n0 = ((t % per_group) / gsz) * TBN;
    };
    const int ktiles = (K + KT - 1) / KT;
    const int nchunks = (ktiles + L::KC - 1) / L::KC;
    auto stage_ptr = [&](int s, int which) -> uint32_t {   // 0 A_hi, 1 A_lo, 2 B_hi, 3 B_lo
        constexpr int P = L::PARTS;
        const uint32_t off =
            which < 2 ? which * L::A_TILE : P * L::A_TILE + (which - 2) * L::B_TILE;
        return smem_u32(ring + (size_t)s * STAGE_BYTES + off);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < TSTG; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&cfull[b]), 1);
            mbar_init(smem_u32(&cempty[b]), EPI_WARPS);
        }
        mbar_init(smem_u32(drainbar), 1);
        mbar_fence_init();
    }
    if (warp == 0) {   // one full warp allocates the accumulator columns
        __syncwarp();
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(tmem_slot);

    if (warp == PRODUCER_WARP) {
        if (lane == 0) {
            tma_prefetch_desc(&tmAhi);
            tma_prefetch_desc(&tmBhi);
            if (TERMS == 3) {
                tma_prefetch_desc(&tmAlo);
                tma_prefetch_desc(&tmBlo);
            }
            uint32_t g = 0;   // k-tiles issued by this CTA, over all its tiles
            bool ok = true;
            for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
                int m0, n0;
                tile_origin(t, m0, n0);
                for (int kt = 0; kt < ktiles; ++kt) {
                    const int s = (int)(g % TSTG);
                    const uint32_t use = g / TSTG;
                    if (use > 0 && !mbar_wait(smem_u32(&empty[s]), (use - 1) & 1, wait_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&full[s]);
                    mbar_arrive_expect_tx(fb, STAGE_BYTES);
                    tma_load_2d(stage_ptr(s, 0), &tmAhi, fb, kt * KT, m0);
                    tma_load_2d(stage_ptr(s, 2), &tmBhi, fb, kt * KT, n0);
                    if (TERMS == 3) {
                        tma_load_2d(stage_ptr(s, 1), &tmAlo, fb, kt * KT, m0);
                        tma_load_2d(stage_ptr(s, 3), &tmBlo, fb, kt * KT, n0);
                    }
                    ++g;
                }
            }
            if (!ok) {
                record_error(err, kErrWaitTimeout);
                for (uint32_t q = (g > TSTG ? g - TSTG : 0); q < g; ++q)
                    mbar_wait(smem_u32(&full[q % TSTG]), (q / TSTG) & 1, DRAIN_NS);
            }
        }
    } else if (warp == MMA_WARP) {
        if (lane == 0) {
            bool ok = true;
            bool issued_any = false;
            uint32_t g = 0;    // k-tiles consumed, over all tiles
            uint32_t gc = 0;   // accumulation chunks issued, over all tiles
            for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
                for (int c = 0; c < nchunks && ok; ++c, ++gc) {
                    const int b = (int)(gc & 1);
                    if (gc >= 2) {   // the epilogue must have read this buffer's previous chunk
                        if (!mbar_wait(smem_u32(&cempty[b]), ((gc >> 1) - 1) & 1, wait_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    const uint32_t d = tmem + (uint32_t)(b * TBN);
                    const int kt_end = (c + 1) * L::KC < ktiles ? (c + 1) * L::KC : ktiles;
                    for (int kt = c * L::KC; kt < kt_end; ++kt) {
                        const int s = (int)(g % TSTG);
                        if (!mbar_wait(smem_u32(&full[s]), (g / TSTG) & 1, wait_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < KT / L::MMA_K; ++kk) {
                            const uint32_t koff = kk * 32;   // 8 TF32 or 16 BF16 = 32 bytes along K
                            const uint64_t ahi = smem_desc<L::SWB>(stage_ptr(s, 0) + koff);
                            const uint64_t bhi = smem_desc<L::SWB>(stage_ptr(s, 2) + koff);
                            const uint32_t acc_in = (kt != c * L::KC || kk != 0) ? 1u : 0u;
                            if (TERMS == 3) {
                                const uint64_t alo = smem_desc<L::SWB>(stage_ptr(s, 1) + koff);
                                const uint64_t blo = smem_desc<L::SWB>(stage_ptr(s, 3) + koff);
                                tc_mma_tf32(d, ahi, blo, acc_in);
                                tc_mma_tf32(d, alo, bhi, 1u);
                                tc_mma_tf32(d, ahi, bhi, 1u);
                            } else if (KIND == kBf16) {
                                tc_mma_bf16(d, ahi, bhi, acc_in);
                            } else {
                                tc_mma_tf32(d, ahi, bhi, acc_in);
                            }
                        }
                        issued_any = true;
                        tc_commit(smem_u32(&empty[s]));   // the stage is free once these MMAs are done
                        ++g;
                    }
                    if (ok) tc_commit(smem_u32(&cfull[b]));
                }
            }
            if (!ok) {
                record_error(err, kErrWaitTimeout);
                if (issued_any) {   // wait for the MMAs already issued
                    tc_commit(smem_u32(drainbar));
                    mbar_wait(smem_u32(drainbar), 0, DRAIN_NS);
                }
            }
        }
    } else {
        // Epilogue warp w: tensor-memory lanes (rows) 32*(w%4) .. +31,
        // columns (w/4)*EPI_COLS .. +EPI_COLS.  The store of one tile runs
        // while the MMAs of the next tile fill the other accumulator buffer.
        const int lane_base = (warp & 3) * 32;
        const int col_base = (warp >> 2) * EPI_COLS;
        bool ok = true;
        uint32_t gc = 0;   // chunks drained, over all tiles
        for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
            int m0, n0;
            tile_origin(t, m0, n0);
            float acc[EPI_COLS];
#pragma unroll
            for (int j = 0; j < EPI_COLS; ++j) acc[j] = 0.0f;
            for (int c = 0; c < nchunks; ++c, ++gc) {
                const int b = (int)(gc & 1);
                // tcgen05.ld is warp-collective: lane 0 decides for the warp whether
                // the chunk is ready; the others then see the completed phase at once.
                bool ready =
                    lane == 0 ? mbar_wait(smem_u32(&cfull[b]), (gc >> 1) & 1, wait_ns) : false;
                ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
                if (!ready) {
                    ok = false;
                    break;
                }
                mbar_wait(smem_u32(&cfull[b]), (gc >> 1) & 1, DRAIN_NS);
                tc_fence_after();
                const uint32_t taddr =
                    tmem + ((uint32_t)lane_base << 16) + (uint32_t)(b * TBN + col_base);
#pragma unroll
                for (int piece = 0; piece < EPI_COLS / 16; ++piece) {
                    float v[16];
                    __syncwarp();
                    tc_ld16(taddr + (uint32_t)(piece * 16), v);
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[piece * 16 + i] += v[i];
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&cempty[b]));
            }
            if (!ok) break;
            const int gm = m0 + lane_base + lane;
            store_row(acc, ep, C, ldc, gm, n0 + col_base, M, N, c_vec4);
        }
        if (!ok && lane == 0) record_error(err, kErrWaitTimeout);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(TMEM_COLS)
                     : "memory");
    }
}


// ---------------------------------------------------------------------------
// Two-SM tiles (tcgen05 cta_group::2).  A cluster of two CTAs on two SMs owns
// a 256 x 256 tile of C.  Each CTA stages its own 128 rows of A and half of
// the tile's B (128 of the 256 columns); one thread of the even CTA issues
// tcgen05.mma.cta_group::2 with M = 256, which reads A and B from both CTAs'
// shared memory at the same offsets and writes each CTA's 128 rows of the
// accumulator into that CTA's tensor memory.  Per SM this moves a third fewer
// operand bytes per MMA than the one-SM 128 x 256 tile, so the same 192 KB
// ring holds six stages instead of four.
//
// Synchronisation (all barriers at the same offsets in both CTAs):
//   full[s]    even CTA: both CTAs' TMA bytes of stage s landed (the odd
//              CTA's copies complete on it through the cta_group::2 form)
//   empty[s]   both: the MMAs reading stage s are done (multicast commit)
//   cfull[b]   both: accumulator buffer b holds a finished chunk (multicast commit)
//   cempty[b]  even CTA: all 16 epilogue warps of the pair have read buffer b
// Every wait is bounded; a time-out is recorded and the roles wind down.

template <int TERMS, int KIND>
struct PairCfg {
    using One = TfCfg<TERMS, KIND>;
    static constexpr int PARTS = One::PARTS, SWB = One::SWB, KT = One::KT, MMA_K = One::MMA_K,
                         KC = One::KC;
    static constexpr int HALF_N = TBN / 2;                       // B columns held per CTA
    static constexpr uint32_t A_TILE = TBM * SWB, B_TILE = HALF_N * SWB;
    static constexpr uint32_t STAGE_BYTES = PARTS * (A_TILE + B_TILE);
    static constexpr int TSTG = (192 * 1024) / STAGE_BYTES;
    // SLACK after the ring keeps any operand read that starts inside the ring
    // (a tile of up to 256 rows) inside this CTA's shared memory.
    static constexpr uint32_t SLACK = PARTS * B_TILE;
    static constexpr size_t SMEM = 1024 + (size_t)TSTG * STAGE_BYTES + SLACK + 512;
    static_assert(A_TILE % 1024 == 0 && B_TILE % 1024 == 0, "tiles keep 1024-byte alignment");
    static_assert(SMEM <= 227 * 1024, "shared memory per block");
};

// Instruction descriptors with M = 256 (the pair's rows).
constexpr uint32_t IDESC2 = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(TBN >> 3) << 17) |
                            ((uint32_t)(256 >> 4) << 24);
constexpr uint32_t IDESC2_BF16 = (1u << 4) | (BF16_FORMAT << 7) | (BF16_FORMAT << 10) |
                                 ((uint32_t)(TBN >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);

__device__ __forceinline__ void tc2_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate, bool bf16) {
    if (bf16)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
}

// Arrive on the barrier at offset `bar` in both CTAs of the pair once every
// tcgen05 operation this thread issued so far is done.
__device__ __forceinline__ void tc2_commit_both(uint32_t bar) {
    const uint16_t mask = 0x3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
        "[%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}

// 2-D TMA load into this CTA's shared memory that completes its bytes on a
// barrier that may belong to the peer CTA of the pair (`bar` a shared::cluster
// address, e.g. from mapa).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                                 int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ uint32_t cluster_addr(uint32_t bar, uint32_t cta) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(bar), "r"(cta));
    return remote;
}

// Arrive (release, cluster scope) on the barrier at offset `bar` of CTA `cta`.
__device__ __forceinline__ void mbar_arrive_cta(uint32_t bar, uint32_t cta) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(bar), "r"(cta));
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote)
                 : "memory");
}

// Bounded wait with cluster-scope acquire (for barriers other CTAs arrive on).
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    auto try_once = [&]() {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        return ok != 0;
    };
    if (try_once()) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (try_once()) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

template <int TERMS, int KIND>
__global__ void __launch_bounds__(THREADS, 1)
tf32_mma2_kernel(const __grid_constant__ CUtensorMap tmAhi, const __grid_constant__ CUtensorMap tmAlo,
                 const __grid_constant__ CUtensorMap tmBhi, const __grid_constant__ CUtensorMap tmBlo,
                 int M, int N, int K, Epilogue ep, float *__restrict__ C, int64_t ldc,
                 int c_vec4, unsigned *err, uint64_t wait_ns) {
    using L = PairCfg<TERMS, KIND>;
    constexpr int TSTG = L::TSTG;
    constexpr int KT = L::KT;
    constexpr uint32_t STAGE_BYTES = L::STAGE_BYTES;
    extern __shared__ unsigned char smem_raw[];
    const uintptr_t base = (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023);
    unsigned char *ring = reinterpret_cast<unsigned char *>(base);
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + (size_t)TSTG * STAGE_BYTES + L::SLACK);
    uint64_t *empty = full + TSTG;
    uint64_t *cfull = empty + TSTG;
    uint64_t *cempty = cfull + 2;
    uint64_t *drainbar = cempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drainbar + 1);

    uint32_t rank;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    const bool lead = rank == 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Persistent over pair tiles: cluster p takes tiles p, p + #clusters, ...
    const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);
    const int num_m = (M + 2 * TBM - 1) / (2 * TBM), num_n = (N + TBN - 1) / TBN;
    const int tiles = num_m * num_n;
    const int per_group = RASTER_GROUP * num_n;
    auto tile_origin = [&](int t, int &m0, int &n0) {
        const int first_m = (t / per_group) * RASTER_GROUP;
        const int gsz = (num_m - first_m) < RASTER_GROUP ? (num_m - first_m) : RASTER_GROUP;
        m0 = (first_m + (t % per_group) % gsz) * (2 * TBM);
        n0 = ((t % per_group) / gsz) * TBN;
    };
    const int ktiles = (K + KT - 1) / KT;
    const int nchunks = (ktiles + L::KC - 1) / L::KC;
    auto stage_ptr = [&](int s, int which) -> uint32_t {   // 0 A_hi, 1 A_lo, 2 B_hi, 3 B_lo
        constexpr int P = L::PARTS;
        const uint32_t off =
            which < 2 ? which * L::A_TILE : P * L::A_TILE + (which - 2) * L::B_TILE;
        return smem_u32(ring + (size_t)s * STAGE_BYTES + off);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < TSTG; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&cfull[b]), 1);
            mbar_init(smem_u32(&cempty[b]), 2 * EPI_WARPS);
        }
        mbar_init(smem_u32(drainbar), 1);
        mbar_fence_init();
    }
    if (warp == 0) {   // one warp of each CTA: the pair allocates its columns together
        __syncwarp();
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();   // both CTAs' barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(tmem_slot);

    if (warp == PRODUCER_WARP) {
        if (lane == 0) {
            tma_prefetch_desc(&tmAhi);
            tma_prefetch_desc(&tmBhi);
            if (TERMS == 3) {
                tma_prefetch_desc(&tmAlo);
                tma_prefetch_desc(&tmBlo);
            }
            uint32_t g = 0;
            bool ok = true;
            for (int t = pair; t < tiles && ok; t += npairs) {
                int m0, n0;
                tile_origin(t, m0, n0);
                const int ya = m0 + TBM * (int)rank, yb = n0 + L::HALF_N * (int)rank;
                for (int kt = 0; kt < ktiles; ++kt) {
                    const int s = (int)(g % TSTG);
                    const uint32_t use = g / TSTG;
                    if (use > 0 && !mbar_wait(smem_u32(&empty[s]), (use - 1) & 1, wait_ns)) {
                        ok = false;
                        break;
                    }
                    // both CTAs' bytes complete on the even CTA's full[s]
                    const uint32_t fb = cluster_addr(smem_u32(&full[s]), 0);
                    if (lead) mbar_arrive_expect_tx(smem_u32(&full[s]), 2 * STAGE_BYTES);
                    tma_load_2d_pair(stage_ptr(s, 0), &tmAhi, fb, kt * KT, ya);
                    tma_load_2d_pair(stage_ptr(s, 2), &tmBhi, fb, kt * KT, yb);
                    if (TERMS == 3) {
                        tma_load_2d_pair(stage_ptr(s, 1), &tmAlo, fb, kt * KT, ya);
                        tma_load_2d_pair(stage_ptr(s, 3), &tmBlo, fb, kt * KT, yb);
                    }
                    ++g;
                }
            }
            if (!ok) {
                record_error(err, kErrWaitTimeout);
                if (lead) {   // the odd CTA's copies complete on these barriers too
                    for (uint32_t q = (g > TSTG ? g - TSTG : 0); q < g; ++q)
                        mbar_wait(smem_u32(&full[q % TSTG]), (q / TSTG) & 1, DRAIN_NS);
                } else {
                    // The odd CTA cannot wait on its copies (they complete on the
                    // even CTA's barriers, possibly in phases the even CTA gave up
                    // on): give them time to land before the CTA can exit.
                    const uint64_t t0 = globaltimer_ns();
                    while (globaltimer_ns() - t0 < 200000ull) {
                    }
                }
            }
        }
    } else if (warp == MMA_WARP) {
        if (lane == 0 && lead) {
            bool ok = true;
            bool issued_any = false;
            uint32_t g = 0, gc = 0;
            constexpr uint32_t idesc = KIND == kBf16 ? IDESC2_BF16 : IDESC2;
            for (int t = pair; t < tiles && ok; t += npairs) {
                for (int c = 0; c < nchunks && ok; ++c, ++gc) {
                    const int b = (int)(gc & 1);
                    if (gc >= 2) {   // both CTAs' epilogues must have read this buffer
                        if (!mbar_wait_cluster(smem_u32(&cempty[b]), ((gc >> 1) - 1) & 1, wait_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    const uint32_t d = tmem + (uint32_t)(b * TBN);
                    const int kt_end = (c + 1) * L::KC < ktiles ? (c + 1) * L::KC : ktiles;
                    for (int kt = c * L::KC; kt < kt_end; ++kt) {
                        const int s = (int)(g % TSTG);
                        if (!mbar_wait_cluster(smem_u32(&full[s]), (g / TSTG) & 1, wait_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < KT / L::MMA_K; ++kk) {
                            const uint32_t koff = kk * 32;
                            const uint64_t ahi = smem_desc<L::SWB>(stage_ptr(s, 0) + koff);
                            const uint64_t bhi = smem_desc<L::SWB>(stage_ptr(s, 2) + koff);
                            const uint32_t acc_in = (kt != c * L::KC || kk != 0) ? 1u : 0u;
                            if (TERMS == 3) {
                                const uint64_t alo = smem_desc<L::SWB>(stage_ptr(s, 1) + koff);
                                const uint64_t blo = smem_desc<L::SWB>(stage_ptr(s, 3) + koff);
                                tc2_mma(d, ahi, blo, idesc, acc_in, false);
                                tc2_mma(d, alo, bhi, idesc, 1u, false);
                                tc2_mma(d, ahi, bhi, idesc, 1u, false);
                            } else {
                                tc2_mma(d, ahi, bhi, idesc, acc_in, KIND == kBf16);
                            }
                        }
                        issued_any = true;
                        tc2_commit_both(smem_u32(&empty[s]));   // both CTAs may refill stage s
                        ++g;
                    }
                    if (ok) tc2_commit_both(smem_u32(&cfull[b]));
                }
            }
            if (!ok) {
                record_error(err, kErrWaitTimeout);
                if (issued_any) {
                    asm volatile(
                        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                            smem_u32(drainbar))
                        : "memory");
                    mbar_wait(smem_u32(drainbar), 0, DRAIN_NS);
                }
            }
        }
    } else {
        // Epilogue warp w of CTA r: rows m0 + 128 r + 32 (w % 4) + lane (this
        // CTA's tensor-memory lanes), columns (w / 4) * EPI_COLS .. + EPI_COLS.
        const int lane_base = (warp & 3) * 32;
        const int col_base = (warp >> 2) * EPI_COLS;
        bool ok = true;
        uint32_t gc = 0;
        for (int t = pair; t < tiles && ok; t += npairs) {
            int m0, n0;
            tile_origin(t, m0, n0);
            float acc[EPI_COLS];
#pragma unroll
            for (int j = 0; j < EPI_COLS; ++j) acc[j] = 0.0f;
            for (int c = 0; c < nchunks; ++c, ++gc) {
                const int b = (int)(gc & 1);
                bool ready =
                    lane == 0 ? mbar_wait(smem_u32(&cfull[b]), (gc >> 1) & 1, wait_ns) : false;
                ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
                if (!ready) {
                    ok = false;
                    break;
                }
                mbar_wait(smem_u32(&cfull[b]), (gc >> 1) & 1, DRAIN_NS);
                tc_fence_after();
                const uint32_t taddr =
                    tmem + ((uint32_t)lane_base << 16) + (uint32_t)(b * TBN + col_base);
#pragma unroll
                for (int piece = 0; piece < EPI_COLS / 16; ++piece) {
                    float v[16];
                    __syncwarp();
                    tc_ld16(taddr + (uint32_t)(piece * 16), v);
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[piece * 16 + i] += v[i];
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cta(smem_u32(&cempty[b]), 0);
            }
            if (!ok) break;
            const int gm = m0 + TBM * (int)rank + lane_base + lane;
            store_row(acc, ep, C, ldc, gm, n0 + col_base, M, N, c_vec4);
        }
        if (!ok && lane == 0) record_error(err, kErrWaitTimeout);
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();   // the pair is done with each other's memory and barriers
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(TMEM_COLS)
                     : "memory");
    }
}


int64_t tf32_ld(int64_t K) { return (K + 3) / 4 * 4; }

template <int TERMS, int KIND>
cudaError_t launch_mma(const GemmArgs &g, const CUtensorMap &tAhi, const CUtensorMap &tAlo,
                       const CUtensorMap &tBhi, const CUtensorMap &tBlo) {
    using L = TfCfg<TERMS, KIND>;
    cudaError_t e = cudaFuncSetAttribute(tf32_mma_kernel<TERMS, KIND>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::SMEM);
    if (e != cudaSuccess) return e;
    const int64_t tiles = ((g.N + TBN - 1) / TBN) * ((g.M + TBM - 1) / TBM);
    if (tiles > 0x7fffffff) return cudaErrorInvalidConfiguration;
    // Persistent: one CTA per SM (the 192 KB ring allows one), each walking
    // its share of the tiles; TF_PERSIST=0 launches one CTA per tile instead.
    const int64_t ctas = TF_PERSIST && g.sm_count > 0 && g.sm_count < tiles ? g.sm_count : tiles;
    const dim3 grid((unsigned)ctas);
    const int c_vec4 = ((reinterpret_cast<uintptr_t>(g.C) & 15) == 0) && (g.ldc % 4 == 0);
    tf32_mma_kernel<TERMS, KIND><<<grid, THREADS, L::SMEM, g.stream>>>(
        tAhi, tAlo, tBhi, tBlo, (int)g.M, (int)g.N, (int)g.K, g.epi(), g.C, g.ldc, c_vec4,
        g.err, g.wait_ns);
    return cudaGetLastError();
}

// Two-SM tiles: clusters of two CTAs, as many as fit at once (one CTA per
// SM), each walking its share of the 256 x 256 tiles.  Returns
// cudaErrorNotSupported (nothing launched) when no cluster fits.
template <int TERMS, int KIND>
cudaError_t launch_mma2(const GemmArgs &g, const CUtensorMap &tAhi, const CUtensorMap &tAlo,
                        const CUtensorMap &tBhi, const CUtensorMap &tBlo) {
    using L = PairCfg<TERMS, KIND>;
    static std::atomic<int> max_pairs[64];   // per device, +1 (0: not yet known)
    auto kern = tf32_mma2_kernel<TERMS, KIND>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::SMEM);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::SMEM;
    cfg.stream = g.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int np = max_pairs[dev].load(std::memory_order_relaxed) - 1;
    if (np < 0) {
        cfg.gridDim = dim3(2, 1, 1);
        if (cudaOccupancyMaxActiveClusters(&np, kern, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            np = 0;
        }
        max_pairs[dev].store(np + 1, std::memory_order_relaxed);
    }
    if (np <= 0) return cudaErrorNotSupported;

    const int64_t tiles = ((g.N + TBN - 1) / TBN) * ((g.M + 2 * TBM - 1) / (2 * TBM));
    const int64_t pairs = tiles < np ? tiles : np;
    cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
    const int c_vec4 = ((reinterpret_cast<uintptr_t>(g.C) & 15) == 0) && (g.ldc % 4 == 0);
    return cudaLaunchKernelEx(&cfg, kern, tAhi, tAlo, tBhi, tBlo, (int)g.M, (int)g.N, (int)g.K,
                              g.epi(), g.C, g.ldc, c_vec4, g.err, g.wait_ns);
}

// Whether a product runs on two-SM tiles: at least one full pair of rows.
bool use_pairs(int64_t M) { return TF_PAIR && M >= 2 * TBM; }

int64_t bf16_ld(int64_t K) { return (K + 7) / 8 * 8; }

template <int TERMS>
cudaError_t launch_terms(const GemmArgs &g, float *ws) {
    using L = TfCfg<TERMS>;
    const int64_t ldk = tf32_ld(g.K);
    const int64_t asz = (g.M * ldk + 63) / 64 * 64, bsz = (g.N * ldk + 63) / 64 * 64;
    // workspace: A_hi, B_hi, then (3 terms) A_lo, B_lo
    float *ahi = ws, *bhi = ws + asz;
    float *alo = TERMS == 3 ? ws + asz + bsz : nullptr;
    float *blo = TERMS == 3 ? ws + 2 * asz + bsz : nullptr;

    // round / split A (rows stay rows), round / split + transpose B
    cudaError_t e = launch_split_rows(g.M, g.K, g.A, g.lda, ahi, alo, ldk, g.stream);
    if (e != cudaSuccess) return e;
    e = launch_transpose_split(g.K, g.N, g.B, g.ldb, bhi, blo, ldk, g.stream);
    if (e != cudaSuccess) return e;

    alignas(64) CUtensorMap tAhi, tAlo, tBhi, tBlo;
    const CUtensorMapSwizzle sw = L::SWB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    constexpr uint32_t kt = L::KT;
    for (int pass = use_pairs(g.M) ? 0 : 1; pass < 2; ++pass) {
        // pass 0: two-SM tiles (each CTA holds half of B's 256 columns); pass 1: one-SM tiles
        const uint32_t brows = pass == 0 ? TBN / 2 : TBN;
        if (!encode_tma_2d(g.encode, &tAhi, ahi, g.K, g.M, ldk, kt, TBM, sw) ||
            !encode_tma_2d(g.encode, &tBhi, bhi, g.K, g.N, ldk, kt, brows, sw))
            return cudaErrorInvalidValue;
        if (TERMS == 3) {
            if (!encode_tma_2d(g.encode, &tAlo, alo, g.K, g.M, ldk, kt, TBM, sw) ||
                !encode_tma_2d(g.encode, &tBlo, blo, g.K, g.N, ldk, kt, brows, sw))
                return cudaErrorInvalidValue;
        } else {
            tAlo = tAhi;   // never read
            tBlo = tBhi;
        }
        if (pass == 0) {
            e = launch_mma2<TERMS, kTf32>(g, tAhi, tAlo, tBhi, tBlo);
            if (e != cudaErrorNotSupported) return e;
        }
    }
    return launch_mma<TERMS, kTf32>(g, tAhi, tAlo, tBhi, tBlo);
}

// BF16: A and B^T rounded to BF16 (nearest even) as [M][ldk] and [N][ldk]
// 16-bit arrays, ldk = K rounded up to 8 (16-byte rows).
cudaError_t launch_bf16_terms(const GemmArgs &g, float *ws) {
    const int64_t ldk = bf16_ld(g.K);
    const int64_t asz = (g.M * ldk + 127) / 128 * 128;
    __nv_bfloat16 *a = reinterpret_cast<__nv_bfloat16 *>(ws), *b = a + asz;
    cudaError_t e = launch_bf16_rows(g.M, g.K, g.A, g.lda, a, ldk, g.stream);
    if (e != cudaSuccess) return e;
    e = launch_bf16_transpose(g.K, g.N, g.B, g.ldb, b, ldk, g.stream);
    if (e != cudaSuccess) return e;
    alignas(64) CUtensorMap tA, tB;
    using L = TfCfg<1, kBf16>;
    const CUtensorMapSwizzle sw = L::SWB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    constexpr uint32_t kt = L::KT;
    for (int pass = use_pairs(g.M) ? 0 : 1; pass < 2; ++pass) {
        const uint32_t brows = pass == 0 ? TBN / 2 : TBN;
        if (!encode_tma_2d_bf16(g.encode, &tA, a, g.K, g.M, ldk, kt, TBM, sw) ||
            !encode_tma_2d_bf16(g.encode, &tB, b, g.K, g.N, ldk, kt, brows, sw))
            return cudaErrorInvalidValue;
        if (pass == 0) {
            e = launch_mma2<1, kBf16>(g, tA, tA, tB, tB);
            if (e != cudaErrorNotSupported) return e;
        }
    }
    return launch_mma<1, kBf16>(g, tA, tA, tB, tB);
}

}  // namespace

size_t tf32_workspace_floats(int64_t M, int64_t N, int64_t K, int terms) {
    if (terms == 0) {   // BF16: two 16-bit arrays
        const int64_t ldk = bf16_ld(K);
        const int64_t a = (M * ldk + 127) / 128 * 128, b = (N * ldk + 127) / 128 * 128;
        return (size_t)((a + b) / 2);
    }
    const int64_t ldk = tf32_ld(K);
    const int64_t a = (M * ldk + 63) / 64 * 64, b = (N * ldk + 63) / 64 * 64;
    return (size_t)((terms == 3 ? 2 : 1) * (a + b));
}

bool tf32x3_can_run(int64_t M, int64_t N, int64_t K) {
    const int64_t lim = int64_t(1) << 31;
    // the tile index (plus one grid stride) stays an int
    return M < lim && N < lim && K < lim && ((M + TBM - 1) / TBM) * ((N + TBN - 1) / TBN) <= 0x7fff0000 &&
           (K + 31) / 32 <= 65535;
}

cudaError_t launch_tf32(const GemmArgs &g, float *ws, int terms) {
    if (terms == 3) return launch_terms<3>(g, ws);
    if (terms == 1) return launch_terms<1>(g, ws);
    if (terms == 0) return launch_bf16_terms(g, ws);
    return cudaErrorInvalidValue;
}

}  // namespace sgemm_gb300
