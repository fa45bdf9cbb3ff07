// common.cuh -- internal helpers shared by the sm_103a kernels of the SGEMM
// library: launch descriptions, mbarrier and TMA wrappers (inline PTX), and
// the bounded wait every kernel uses.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sgemm_gb300 {

// Bit set in the per-device error word when a bounded wait runs out.
constexpr unsigned kErrWaitTimeout = 1u;

// The driver's cuTensorMapEncodeTiled, looked up at run time.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Everything a kernel launcher needs.
// Activations of the fused epilogue (the SGEMM_ACT_* values of the C ABI).
enum : int { kActNone = 0, kActRelu = 1, kActGelu = 2, kActSilu = 3 };

// What every kernel's store applies to an accumulated dot product `acc`:
//     C = act(alpha*acc + beta*C + bias[col])
// C is read only when beta != 0; bias == nullptr adds nothing.
struct Epilogue {
    float alpha, beta;
    const float *bias;
    int act;
};

struct GemmArgs {
    int64_t M, N, K;
    float alpha, beta;
    const float *A; int64_t lda;
    const float *B; int64_t ldb;
    float *C; int64_t ldc;
    cudaStream_t stream;
    unsigned *err;          // device pointer to the error word
    uint64_t wait_ns;       // bounded-wait limit in nanoseconds
    int sm_count;
    EncodeTiledFn encode;   // tensor-map encoder
    const float *bias = nullptr;   // fused epilogue: N floats, or none
    int act = kActNone;            // fused epilogue activation
    Epilogue epi() const { return Epilogue{alpha, beta, bias, act}; }
};

// 2-D fp32 tensor map over a row-major matrix: `inner` contiguous elements
// per row, `rows` rows, row stride `ld` elements, box box_inner x box_rows,
// out-of-range elements read as zero.  Returns false if the driver refuses.
bool encode_tma_2d(EncodeTiledFn enc, CUtensorMap *map, const float *base, int64_t inner,
                   int64_t rows, int64_t ld, uint32_t box_inner, uint32_t box_rows,
                   CUtensorMapSwizzle swz);
// The same over 16-bit BF16 elements (ld and the box in elements).
bool encode_tma_2d_bf16(EncodeTiledFn enc, CUtensorMap *map, const void *base, int64_t inner,
                        int64_t rows, int64_t ld, uint32_t box_inner, uint32_t box_rows,
                        CUtensorMapSwizzle swz);

// ---- launchers (one translation unit each) ------------------------------------
cudaError_t launch_scale_c(const GemmArgs &g);
cudaError_t launch_ffma_generic(const GemmArgs &g);
// FFMA kernel: transposes A into `workspace` (K rows of ffma_tma_at_ld(M)
// floats, 16-byte aligned), then runs the TMA-staged kernel on A^T and B.
// `capacity` is the workspace's size in floats: at least K * ffma_tma_at_ld(M);
// whatever ffma_tma_workspace_floats(g, capacity) asks beyond that holds the
// partial tiles of the split last wave.
cudaError_t launch_ffma_tma(const GemmArgs &g, float *workspace, int64_t capacity);
int64_t ffma_tma_workspace_floats(const GemmArgs &g, int64_t capacity);
// Tile configurations of the FFMA kernel: the one a shape runs (the tuning
// table, or the forced one), their number, forcing one (-1: the table;
// returns the previous setting, -2 for a bad index), and their parameters.
int ffma_config_for(int64_t M, int64_t N, int64_t K);
int ffma_config_count();
int ffma_force_config(int idx);
int ffma_force_tail_sum(int mode);   // -1 default, 0 last arriver, 1 separate kernel; -2 if invalid
// The work list an sgemm() call of g's shape runs on the FFMA-TMA path:
// units (CTAs), span (k-tiles per tail unit, 0 when the tail is not
// divided) and whether a separate kernel sums the tail (1) or not (0).
void ffma_tma_plan_info(const GemmArgs &g, int64_t *units, int *span, int *tail_sum);
// sgemm_kernel_timing: start (1, clearing earlier records) or stop (0) the
// event pairs around FFMA tile-kernel launches; -2 for another value.
int kernel_timing(int enable);
// Summed elapsed time of the recorded tile kernels (waits for them).
bool kernel_timing_result(double *total_ms, int64_t *launches);
bool ffma_config_info(int idx, int *bm, int *bn, int *bk, int *stages, int *threads, int *minb);
int64_t ffma_tma_at_ld(int64_t M);
// Largest M the TMA FFMA kernel's grid can cover.
int64_t ffma_tma_max_m();
// At[k*ldt + m] = A[m*lda + k] for m < M, k < K (ldt % 4 == 0, At 16-byte aligned);
// also sets zero[0 .. nzero) to 0 (nzero <= 1024).
cudaError_t launch_transpose(int64_t M, int64_t K, const float *A, int64_t lda, float *At,
                             int64_t ldt, cudaStream_t stream, unsigned *zero = nullptr,
                             int nzero = 0);
// TF32 hi/lo split of B (K x N) written transposed: hi[n*ldo + k], lo[n*ldo + k]
// (lo == nullptr: the rounded hi part only).
cudaError_t launch_transpose_split(int64_t K, int64_t N, const float *B, int64_t ldb, float *hi,
                                   float *lo, int64_t ldo, cudaStream_t stream);
// TF32 hi/lo split of X (R x Cc) in place of layout: hi[r*ldo + c], lo[r*ldo + c]
// (lo == nullptr: the rounded hi part only).
cudaError_t launch_split_rows(int64_t R, int64_t Cc, const float *X, int64_t ldx, float *hi,
                              float *lo, int64_t ldo, cudaStream_t stream);
// BF16 (round to nearest even) copies for the BF16 tensor-core kernel:
// out[r*ldo + c] = bf16(X[r][c]) and out[n*ldo + k] = bf16(B[k][n]); `out` is
// bf16 storage, ldo in elements, a multiple of 4.
cudaError_t launch_bf16_rows(int64_t R, int64_t Cc, const float *X, int64_t ldx, void *out,
                             int64_t ldo, cudaStream_t stream);
cudaError_t launch_bf16_transpose(int64_t K, int64_t N, const float *B, int64_t ldb, void *out,
                                  int64_t ldo, cudaStream_t stream);
cudaError_t launch_decode(const GemmArgs &g);
cudaError_t launch_selftest_wait(unsigned *err, uint64_t wait_ns, cudaStream_t stream);
// Tensor-core kernels.  terms == 3 (3xTF32): splits A and B into TF32
// hi/lo parts in `workspace`, then accumulates hi*lo + lo*hi + hi*hi with
// tcgen05 MMAs.  terms == 1 (1xTF32): rounds A and B to TF32 (the hi parts
// only) and accumulates hi*hi.  terms == 0 (BF16): rounds A and B to BF16
// and accumulates their products (kind::f16).  The workspace holds
// tf32_workspace_floats(M, N, K, terms) floats.
cudaError_t launch_tf32(const GemmArgs &g, float *workspace, int terms);
size_t tf32_workspace_floats(int64_t M, int64_t N, int64_t K, int terms);
bool tf32x3_can_run(int64_t M, int64_t N, int64_t K);
// Frees the buffers, streams and events of sgemm_host's pipelines (after
// waiting for them); false if a CUDA call failed.
bool release_host_paths();
// Fills g.err, g.wait_ns, g.sm_count and g.encode for the current device
// (setting the device up on first use); returns an SGEMM_* status.
int fill_device_args(GemmArgs &g);


#ifdef __CUDACC__

// act(v + bias[col]): the part of the epilogue after alpha*acc + beta*C.
// GELU is the tanh form x/2 * (1 + tanh(sqrt(2/pi) * (x + 0.044715 x^3))),
// SiLU is x / (1 + e^-x); CUDA's tanhf and expf.  ReLU keeps NaN.
__device__ __forceinline__ float epilogue_tail(const Epilogue &e, float v, int64_t col) {
    if (e.bias != nullptr) v += __ldg(e.bias + col);
    switch (e.act) {
        case kActRelu: return v < 0.0f ? 0.0f : v;
        case kActGelu:
            return 0.5f * v * (1.0f + tanhf(0.7978845608028654f * fmaf(0.044715f * v, v * v, v)));
        case kActSilu: return v / (1.0f + expf(-v));
        default: return v;
    }
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make initialised barriers visible to the async (TMA) proxy and the cluster.
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait until the barrier phase with parity `parity` has completed, giving up
// after `limit_ns` nanoseconds.  Returns false on time-out; the caller records
// the error and leaves without touching the stage.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

__device__ __forceinline__ void record_error(unsigned *err, unsigned bits) {
    if (err) atomicOr(err, bits);
}

// 2-D tiled TMA load of one box into shared memory, completing on `bar`.
// x is the innermost (contiguous) coordinate, y the row coordinate.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Programmatic dependent launch.  A kernel launched with the programmatic
// stream-serialization attribute may start while the kernel before it on the
// stream is still running; pdl_wait() blocks until that kernel has completed
// and its writes are visible (it returns at once without such a launch).
// pdl_trigger() in the earlier kernel lets the dependent grid launch once every
// CTA of the earlier grid has triggered or exited.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 128-bit streaming load that does not allocate in L1 (data used once).
__device__ __forceinline__ float4 ldg_stream_f4(const float *p) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float ldg_stream_f1(const float *p) {
    float v;
    asm volatile("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

#endif  // __CUDACC__

}  // namespace sgemm_gb300
