// api.cu -- the C ABI declared in include/sgemm_gb300.h: argument checks,
// quick returns, kernel choice, TMA descriptor encoding and the per-device
// kernel error word.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "sgemm_gb300.h"

using namespace sgemm_gb300;

namespace {

// Kernels set bits here when a bounded wait runs out; sgemm_status() reads and
// clears it.  One word per device (a __device__ variable lives in each
// device's copy of this module).
__device__ unsigned g_err_word;

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    int status = SGEMM_OK;
    unsigned *err = nullptr;
    int sm_count = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
std::atomic<int> g_force{SGEMM_KERNEL_AUTO};
std::atomic<int64_t> g_wait_ns{2000000000LL};   // 2 s

EncodeTiledFn g_encode = nullptr;

// Workspace (A^T for the FFMA kernel): one buffer per (device, stream), grown
// and freed in stream order, so calls on one stream reuse it safely and calls
// on different streams never share it.
std::mutex g_ws_mu;
std::map<std::pair<int, uintptr_t>, std::pair<void *, size_t>> g_ws;

int workspace(size_t bytes, cudaStream_t s, float **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_ws_mu);
    auto &w = g_ws[{dev, reinterpret_cast<uintptr_t>(s)}];
    if (w.second < bytes) {
        // An allocation made while `s` is captured would belong to the graph.
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
            (void)cudaGetLastError();
            return SGEMM_ERR_CUDA;
        }
        if (cs != cudaStreamCaptureStatusNone) return SGEMM_ERR_CAPTURE;
        const size_t grow = std::max(bytes, w.second + w.second / 2);
        const size_t nb = (grow + (size_t(2) << 20) - 1) & ~((size_t(2) << 20) - 1);
        if (w.first != nullptr) {
            if (cudaFreeAsync(w.first, s) != cudaSuccess) return SGEMM_ERR_CUDA;
            w = {nullptr, 0};
        }
        void *p = nullptr;
        if (cudaMallocAsync(&p, nb, s) != cudaSuccess) {
            (void)cudaGetLastError();
            return SGEMM_ERR_CUDA;
        }
        w = {p, nb};
    }
    *out = static_cast<float *>(w.first);
    return SGEMM_OK;
}

// Per-device set-up: check the architecture, find the error word, look up
// the driver's tensor-map encoder.  Returns a status code.
int device_state(DeviceState **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SGEMM_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &st = g_dev[dev];
    if (!st.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SGEMM_ERR_CUDA;
        if (major != 10 || minor != 3) {
            st.status = SGEMM_ERR_DEVICE;
        } else {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return SGEMM_ERR_CUDA;
            if (cudaMemset(p, 0, sizeof(unsigned)) != cudaSuccess) return SGEMM_ERR_CUDA;
            if (cudaDeviceSynchronize() != cudaSuccess) return SGEMM_ERR_CUDA;
            if (!g_encode) {
                void *fn = nullptr;
                cudaDriverEntryPointQueryResult q;
                if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q) != cudaSuccess ||
                    q != cudaDriverEntryPointSuccess || fn == nullptr)
                    return SGEMM_ERR_CUDA;
                g_encode = reinterpret_cast<EncodeTiledFn>(fn);
            }
            st.err = static_cast<unsigned *>(p);
            st.sm_count = sms;
            st.status = SGEMM_OK;
        }
        st.ready = true;
    }
    *out = &st;
    return st.status;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Byte range [lo, hi) touched by a rows x cols matrix with row stride ld.
void span(const void *p, int64_t rows, int64_t cols, int64_t ld, uintptr_t *lo, uintptr_t *hi) {
    *lo = reinterpret_cast<uintptr_t>(p);
    *hi = *lo + (uintptr_t)(((rows - 1) * ld + cols) * (int64_t)sizeof(float));
}

bool overlaps(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) {
    return a0 < b1 && b0 < a1;
}

constexpr int64_t kMaxElems = int64_t(1) << 40;   // keeps every offset far from int64 overflow

// Checks shared by every entry point; on success *kernel is the choice
// before any forcing or tensor-core preference.
int check_args(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
               const float *B, int64_t ldb, float beta, const float *C, int64_t ldc,
               bool *uses_ab) {
    (void)beta;
    if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_BAD_DIM;
    *uses_ab = false;
    if (M == 0 || N == 0) return SGEMM_OK;
    if (C == nullptr) return SGEMM_ERR_NULL_PTR;
    if (ldc < N) return SGEMM_ERR_BAD_LD;
    if (M > kMaxElems / ldc) return SGEMM_ERR_BAD_DIM;
    *uses_ab = (alpha != 0.0f) && (K > 0);
    if (!*uses_ab) return SGEMM_OK;
    if (A == nullptr || B == nullptr) return SGEMM_ERR_NULL_PTR;
    if (lda < K || ldb < N) return SGEMM_ERR_BAD_LD;
    if (M > kMaxElems / lda || K > kMaxElems / ldb) return SGEMM_ERR_BAD_DIM;
    uintptr_t c0, c1, a0, a1, b0, b1;
    span(C, M, N, ldc, &c0, &c1);
    span(A, M, K, lda, &a0, &a1);
    span(B, K, N, ldb, &b0, &b1);
    if (overlaps(c0, c1, a0, a1) || overlaps(c0, c1, b0, b1)) return SGEMM_ERR_ALIAS;
    return SGEMM_OK;
}

// The TMA FFMA kernel reads B in place and A through its transposed copy
// (which the transpose kernel writes from any alignment and lda).
bool tma_ok(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
            int64_t ldb) {
    (void)A;
    (void)lda;
    const int64_t lim = int64_t(1) << 31;
    return aligned16(B) && ldb % 4 == 0 && M < lim && N < lim && K < lim &&
           M <= ffma_tma_max_m() && (K + 31) / 32 <= 65535;
}

bool kernel_can_run(int id, int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                    const float *B, int64_t ldb) {
    switch (id) {
        case SGEMM_KERNEL_FFMA_TMA: return tma_ok(M, N, K, A, lda, B, ldb);
        case SGEMM_KERNEL_FFMA_GENERIC: return (M + 63) / 64 <= 65535;
        case SGEMM_KERNEL_DECODE: return M <= 16 && (N + 127) / 128 <= 65535;
        case SGEMM_KERNEL_TF32X3:
        case SGEMM_KERNEL_TF32:
        case SGEMM_KERNEL_BF16: return tf32x3_can_run(M, N, K);
        default: return false;
    }
}

int choose(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
           const float *B, int64_t ldb, float beta, const float *C, int64_t ldc, int mode) {
    if (mode != SGEMM_MODE_FP32 && mode != SGEMM_MODE_3XTF32 && mode != SGEMM_MODE_TF32 &&
        mode != SGEMM_MODE_BF16)
        return SGEMM_ERR_BAD_ARG;
    bool uses_ab = false;
    const int rc = check_args(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, &uses_ab);
    if (rc != SGEMM_OK) return rc;
    if (M == 0 || N == 0) return SGEMM_KERNEL_NONE;
    if (!uses_ab) return SGEMM_KERNEL_SCALE_C;
    const int forced = g_force.load();
    if (forced != SGEMM_KERNEL_AUTO && kernel_can_run(forced, M, N, K, A, lda, B, ldb))
        return forced;
    // The tensor-core tile is 128 rows tall; skinny products stay on the
    // (FP32-exact) decode kernel.
    if (mode != SGEMM_MODE_FP32 && M > 16) {
        const int tc = mode == SGEMM_MODE_3XTF32 ? SGEMM_KERNEL_TF32X3
                       : mode == SGEMM_MODE_TF32 ? SGEMM_KERNEL_TF32
                                                 : SGEMM_KERNEL_BF16;
        if (kernel_can_run(tc, M, N, K, A, lda, B, ldb)) return tc;
    }
    if (M <= 16 && kernel_can_run(SGEMM_KERNEL_DECODE, M, N, K, A, lda, B, ldb))
        return SGEMM_KERNEL_DECODE;
    // Tiny products (at most 2^21 multiply-adds, such as 128^3) are bound by
    // launch overhead ("GPU 基础原理", section 3): the plain-load kernel does
    // them in one launch where the TMA path needs the transpose as well
    // (measured on GB300 in a replayed graph: 128^3 9.3 against 12.5 us per
    // call; equal at 256^3).
    if (M <= 1024 && N <= 1024 && K <= 1024 && M * N * K <= (int64_t(1) << 21) &&
        kernel_can_run(SGEMM_KERNEL_FFMA_GENERIC, M, N, K, A, lda, B, ldb))
        return SGEMM_KERNEL_FFMA_GENERIC;
    if (tma_ok(M, N, K, A, lda, B, ldb)) return SGEMM_KERNEL_FFMA_TMA;
    if (kernel_can_run(SGEMM_KERNEL_FFMA_GENERIC, M, N, K, A, lda, B, ldb))
        return SGEMM_KERNEL_FFMA_GENERIC;
    return SGEMM_ERR_BAD_DIM;
}

// The fused epilogue's own arguments: a known activation, and a bias (N
// floats) that does not overlap C.
int check_epilogue(int64_t M, int64_t N, const float *C, int64_t ldc, const float *bias, int act) {
    if (act < SGEMM_ACT_NONE || act > SGEMM_ACT_SILU) return SGEMM_ERR_BAD_ARG;
    if (bias == nullptr || M == 0 || N == 0) return SGEMM_OK;
    uintptr_t c0, c1, v0, v1;
    span(C, M, N, ldc, &c0, &c1);
    span(bias, 1, N, N, &v0, &v1);
    return overlaps(c0, c1, v0, v1) ? SGEMM_ERR_ALIAS : SGEMM_OK;
}

int run(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda, const float *B,
        int64_t ldb, float beta, float *C, int64_t ldc, void *stream, int mode,
        const float *bias = nullptr, int act = SGEMM_ACT_NONE) {
    const int kid = choose(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, mode);
    if (kid < 0) return kid;
    const int erc = check_epilogue(M, N, C, ldc, bias, act);
    if (erc != SGEMM_OK) return erc;
    if (kid == SGEMM_KERNEL_NONE) return SGEMM_OK;
    DeviceState *st = nullptr;
    const int ds = device_state(&st);
    if (ds != SGEMM_OK) return ds;

    GemmArgs g;
    g.M = M; g.N = N; g.K = K;
    g.alpha = alpha; g.beta = beta;
    g.A = A; g.lda = lda; g.B = B; g.ldb = ldb; g.C = C; g.ldc = ldc;
    g.stream = static_cast<cudaStream_t>(stream);
    g.err = st->err;
    g.wait_ns = (uint64_t)g_wait_ns.load();
    g.sm_count = st->sm_count;
    g.encode = g_encode;
    g.bias = bias;
    g.act = act;

    cudaError_t e = cudaSuccess;
    switch (kid) {
        case SGEMM_KERNEL_SCALE_C: e = launch_scale_c(g); break;
        case SGEMM_KERNEL_FFMA_GENERIC: e = launch_ffma_generic(g); break;
        case SGEMM_KERNEL_DECODE: e = launch_decode(g); break;
        case SGEMM_KERNEL_FFMA_TMA: {
            float *ws = nullptr;
            const int64_t nf = ffma_tma_workspace_floats(g, INT64_MAX);
            const int rc = workspace((size_t)nf * sizeof(float), g.stream, &ws);
            if (rc != SGEMM_OK) return rc;
            e = launch_ffma_tma(g, ws, nf);
            break;
        }
        case SGEMM_KERNEL_TF32X3:
        case SGEMM_KERNEL_TF32:
        case SGEMM_KERNEL_BF16: {
            const int terms = kid == SGEMM_KERNEL_TF32X3 ? 3 : kid == SGEMM_KERNEL_TF32 ? 1 : 0;
            float *ws = nullptr;
            const int rc =
                workspace(tf32_workspace_floats(M, N, K, terms) * sizeof(float), g.stream, &ws);
            if (rc != SGEMM_OK) return rc;
            e = launch_tf32(g, ws, terms);
            break;
        }
        default: return SGEMM_ERR_BAD_ARG;
    }
    return e == cudaSuccess ? SGEMM_OK : SGEMM_ERR_CUDA;
}

}  // namespace

namespace sgemm_gb300 {
bool encode_tma_2d(EncodeTiledFn enc, CUtensorMap *map, const float *base, int64_t inner,
                   int64_t rows, int64_t ld, uint32_t box_inner, uint32_t box_rows,
                   CUtensorMapSwizzle swz) {
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * sizeof(float)};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
bool encode_tma_2d_bf16(EncodeTiledFn enc, CUtensorMap *map, const void *base, int64_t inner,
                        int64_t rows, int64_t ld, uint32_t box_inner, uint32_t box_rows,
                        CUtensorMapSwizzle swz) {
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace sgemm_gb300

namespace {

// One thread waits on a barrier that nothing completes, with the library's
// bounded wait, and records the time-out.
__global__ void selftest_wait_kernel(unsigned *err, uint64_t wait_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        mbar_fence_init();
        if (!mbar_wait(smem_u32(&bar), 0, wait_ns)) record_error(err, kErrWaitTimeout);
    }
}

}  // namespace

namespace sgemm_gb300 {
cudaError_t launch_selftest_wait(unsigned *err, uint64_t wait_ns, cudaStream_t stream) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>(err, wait_ns);
    return cudaGetLastError();
}

int fill_device_args(GemmArgs &g) {
    DeviceState *st = nullptr;
    const int ds = device_state(&st);
    if (ds != SGEMM_OK) return ds;
    g.err = st->err;
    g.wait_ns = (uint64_t)g_wait_ns.load();
    g.sm_count = st->sm_count;
    g.encode = g_encode;
    return SGEMM_OK;
}
}  // namespace sgemm_gb300

extern "C" {

int sgemm(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
          const float *B, int64_t ldb, float beta, float *C, int64_t ldc, void *stream) {
    return run(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, SGEMM_MODE_FP32);
}

int sgemm_3xtf32(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
                 const float *B, int64_t ldb, float beta, float *C, int64_t ldc, void *stream) {
    return run(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, SGEMM_MODE_3XTF32);
}

int sgemm_tf32(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
               const float *B, int64_t ldb, float beta, float *C, int64_t ldc, void *stream) {
    return run(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, SGEMM_MODE_TF32);
}

int sgemm_bf16(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
               const float *B, int64_t ldb, float beta, float *C, int64_t ldc, void *stream) {
    return run(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, SGEMM_MODE_BF16);
}

int sgemm_fused(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
                const float *B, int64_t ldb, float beta, float *C, int64_t ldc, const float *bias,
                int activation, int mode, void *stream) {
    return run(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, mode, bias, activation);
}

int sgemm_status(void *stream) {
    DeviceState *st = nullptr;
    const int ds = device_state(&st);
    if (ds != SGEMM_OK) return ds;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SGEMM_ERR_CUDA;
    unsigned word = 0;
    if (cudaMemcpy(&word, st->err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SGEMM_ERR_CUDA;
    if (word != 0) {
        const unsigned zero = 0;
        if (cudaMemcpy(st->err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return SGEMM_ERR_CUDA;
        return SGEMM_ERR_TIMEOUT;
    }
    return SGEMM_OK;
}

const char *sgemm_status_string(int status) {
    switch (status) {
        case SGEMM_OK: return "success";
        case SGEMM_ERR_BAD_DIM: return "invalid dimension (negative, or too large to index)";
        case SGEMM_ERR_BAD_LD: return "leading dimension smaller than the row length";
        case SGEMM_ERR_NULL_PTR: return "a required pointer is NULL";
        case SGEMM_ERR_ALIAS: return "C overlaps A or B";
        case SGEMM_ERR_CUDA: return "a CUDA runtime or driver call failed";
        case SGEMM_ERR_DEVICE: return "the current device is not an sm_103 GPU";
        case SGEMM_ERR_TIMEOUT: return "a device-side bounded wait ran out";
        case SGEMM_ERR_BAD_ARG: return "invalid argument";
        case SGEMM_ERR_CAPTURE:
            return "the stream is being captured and the call needs a larger workspace; "
                   "run one call of this shape eagerly on the stream first";
        case SGEMM_ERR_TOO_LARGE:
            return "problem needs more than the fixed scratch of sgemm_noalloc "
                   "(K * round_up(M, 4) floats > 16777216)";
        default: return "unknown status";
    }
}

int sgemm_select_kernel(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
                        const float *B, int64_t ldb, float beta, const float *C, int64_t ldc,
                        int mode) {
    return choose(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, mode);
}

int sgemm_force_kernel(int id) {
    if (id != SGEMM_KERNEL_AUTO && id != SGEMM_KERNEL_FFMA_TMA && id != SGEMM_KERNEL_FFMA_GENERIC &&
        id != SGEMM_KERNEL_DECODE && id != SGEMM_KERNEL_TF32X3 && id != SGEMM_KERNEL_TF32 &&
        id != SGEMM_KERNEL_BF16)
        return SGEMM_ERR_BAD_ARG;
    return g_force.exchange(id);
}

int64_t sgemm_set_wait_limit(int64_t ns) {
    if (ns < 1) ns = 2000000000LL;
    return g_wait_ns.exchange(ns);
}

int sgemm_selftest_wait(int64_t ns, void *stream) {
    DeviceState *st = nullptr;
    const int ds = device_state(&st);
    if (ds != SGEMM_OK) return ds;
    if (ns < 1) ns = 1;
    return launch_selftest_wait(st->err, (uint64_t)ns, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? SGEMM_OK
               : SGEMM_ERR_CUDA;
}

int sgemm_release_workspaces(void) {
    int rc = release_host_paths() ? SGEMM_OK : SGEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_ws_mu);
    int cur = 0;
    if (cudaGetDevice(&cur) != cudaSuccess) return SGEMM_ERR_CUDA;
    for (auto &kv : g_ws) {
        if (kv.second.first == nullptr) continue;
        cudaStream_t s = reinterpret_cast<cudaStream_t>(kv.first.second);
        if (cudaSetDevice(kv.first.first) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess || cudaFree(kv.second.first) != cudaSuccess)
            rc = SGEMM_ERR_CUDA;
    }
    g_ws.clear();
    if (cudaSetDevice(cur) != cudaSuccess) rc = SGEMM_ERR_CUDA;
    return rc;
}

int sgemm_ffma_config_count(void) { return ffma_config_count(); }

int sgemm_ffma_config_info(int idx, int *bm, int *bn, int *bk, int *stages, int *threads,
                           int *ctas_per_sm) {
    if (!bm || !bn || !bk || !stages || !threads || !ctas_per_sm) return SGEMM_ERR_BAD_ARG;
    return ffma_config_info(idx, bm, bn, bk, stages, threads, ctas_per_sm) ? SGEMM_OK
                                                                          : SGEMM_ERR_BAD_ARG;
}

int sgemm_ffma_config_for(int64_t M, int64_t N, int64_t K) { return ffma_config_for(M, N, K); }

int sgemm_ffma_force_config(int idx) {
    const int prev = ffma_force_config(idx);
    return prev == -2 ? SGEMM_ERR_BAD_ARG : prev;
}

int sgemm_ffma_force_tail_sum(int mode) {
    const int prev = ffma_force_tail_sum(mode);
    return prev == -2 ? SGEMM_ERR_BAD_ARG : prev;
}

int sgemm_ffma_tail_plan(int64_t M, int64_t N, int64_t K, int64_t *units, int *span, int *tail_sum) {
    if (!units || !span || !tail_sum) return SGEMM_ERR_BAD_ARG;
    if (M < 1 || N < 1 || K < 1 || M > ffma_tma_max_m() || N > INT32_MAX || K > INT32_MAX)
        return SGEMM_ERR_BAD_DIM;
    GemmArgs g{};
    const int rc = fill_device_args(g);
    if (rc != SGEMM_OK) return rc;
    g.M = M;
    g.N = N;
    g.K = K;
    ffma_tma_plan_info(g, units, span, tail_sum);
    return SGEMM_OK;
}

int sgemm_kernel_timing(int enable) {
    const int prev = kernel_timing(enable);
    return prev == -2 ? SGEMM_ERR_BAD_ARG : prev;
}

int sgemm_kernel_timing_result(double *total_ms, int64_t *launches) {
    if (!total_ms || !launches) return SGEMM_ERR_BAD_ARG;
    return kernel_timing_result(total_ms, launches) ? SGEMM_OK : SGEMM_ERR_CUDA;
}

int sgemm_version(void) { return 100; }

}  // extern "C"
