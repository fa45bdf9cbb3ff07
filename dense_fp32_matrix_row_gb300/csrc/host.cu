// host.cu -- sgemm_host: the product for operands that live in host memory.
//
// The copies to and from the device are overlapped with the compute, one
// row panel of A and C at a time (see include/sgemm_gb300.h):
//
//   copy stream   B, A_0 (C_0), A_1 (C_1), ...       (host -> device)
//   `stream`           C_0 = alpha*A_0@B + beta*C_0, C_1 = ..., ...
//   return stream                            C_0, C_1, ... (device -> host)
//
// Two device slots hold consecutive panels, so the copy of panel p+1 and the
// copy back of panel p-1 run while panel p is computed.  Events order the
// three streams; the call forks from and joins back into `stream`, so it is
// ordered like any other work on that stream.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "sgemm_gb300.h"

using namespace sgemm_gb300;

namespace {

constexpr int kSlots = 2;
#ifndef HOST_B_PARTS
#define HOST_B_PARTS 4
#endif
constexpr int kBParts = HOST_B_PARTS;   // most K-ranges B arrives in while the first panel computes
constexpr size_t kAlign = 256;   // bytes; every device sub-buffer starts on this boundary

struct HostPath {
    std::mutex mu;                 // one enqueue at a time per (device, stream)
    bool ready = false;
    cudaStream_t up = nullptr;     // host -> device copies
    cudaStream_t down = nullptr;   // device -> host copies
    cudaEvent_t fork = nullptr, join = nullptr;
    cudaEvent_t loaded[kSlots] = {}, computed[kSlots] = {}, stored[kSlots] = {};
    cudaEvent_t bpart[kBParts] = {};   // rows of B up to K-range j are on the device
    void *buf = nullptr;           // device buffer: B, then kSlots x (A panel, C panel)
    size_t bytes = 0;
};

std::mutex g_mu;
std::map<std::pair<int, uintptr_t>, HostPath> g_paths;   // nodes never move
std::atomic<int> g_panels{0};                               // 0: the library's choice

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int create(HostPath &h) {
    if (h.ready) return SGEMM_OK;
    bool ok = cudaStreamCreateWithFlags(&h.up, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&h.down, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&h.fork, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&h.join, cudaEventDisableTiming) == cudaSuccess;
    for (int s = 0; ok && s < kSlots; ++s)
        ok = cudaEventCreateWithFlags(&h.loaded[s], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&h.computed[s], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&h.stored[s], cudaEventDisableTiming) == cudaSuccess;
    for (int j = 0; ok && j < kBParts; ++j)
        ok = cudaEventCreateWithFlags(&h.bpart[j], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        (void)cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    h.ready = true;
    return SGEMM_OK;
}

void destroy(HostPath &h) {
    if (h.buf != nullptr) (void)cudaFree(h.buf);
    if (h.up != nullptr) (void)cudaStreamDestroy(h.up);
    if (h.down != nullptr) (void)cudaStreamDestroy(h.down);
    for (cudaEvent_t e : {h.fork, h.join})
        if (e != nullptr) (void)cudaEventDestroy(e);
    for (int s = 0; s < kSlots; ++s)
        for (cudaEvent_t e : {h.loaded[s], h.computed[s], h.stored[s]})
            if (e != nullptr) (void)cudaEventDestroy(e);
    for (int j = 0; j < kBParts; ++j)
        if (h.bpart[j] != nullptr) (void)cudaEventDestroy(h.bpart[j]);
    h.buf = nullptr;
    h.bytes = 0;
    h.ready = false;
    h.up = h.down = nullptr;
    h.fork = h.join = nullptr;
    for (int s = 0; s < kSlots; ++s) h.loaded[s] = h.computed[s] = h.stored[s] = nullptr;
    for (int j = 0; j < kBParts; ++j) h.bpart[j] = nullptr;
}

// K-ranges the first panel is computed in, so that the copy of B (which the
// first panel needs in full) overlaps the first panel's products: B goes up
// range by range after A_0 and C_0, and range j is multiplied as soon as it
// has arrived (C_0 = alpha*A_0[:, range 0]@B[range 0] + beta*C_0, then
// C_0 += alpha*A_0[:, range j]@B[range j]).  Only with several panels and a
// deep K; one range otherwise.
int b_parts(int64_t M, int64_t rows, int64_t K, bool uses_ab) {
    if (!uses_ab || rows >= M) return 1;
    if (K >= 2048) return kBParts;
    if (K >= 1024) return std::min(kBParts, 2);
    return 1;
}

// Rows per panel.  Each panel adds a fixed cost (its own kernel ramp, tail
// and transposition of A; measured on GB300 about 10 us per 1024 of K), and
// the first panel's copy up and the last panel's copy down are not hidden
// behind any compute.  With t_row the copy time of one row (A and C up at
// about 209 GB/s, C down at about 192 GB/s) the count that balances the two,
// M * t_row / P against P * t_panel, is sqrt(M * t_row / t_panel), at most 8.
// Measured at 4092^3 (ms per call by panel count): 2: 2.94, 3: 2.90,
// 4: 2.84, 5: 2.77, 6: 2.79, 8: 2.78.  Skinny products run as one panel.
int64_t panel_rows(int64_t M, int64_t N, int64_t K, bool uses_ab) {
    const int forced = g_panels.load();
    int64_t P;
    if (forced > 0) {
        P = forced;
    } else if (!uses_ab || M <= 256) {
        P = 1;
    } else {
        const double t_row_us = (double)(K + N) * 4.0 / 209e3 + (double)N * 4.0 / 192e3;
        const double t_panel_us = 10.0 * (double)K / 1024.0;
        P = std::min<int64_t>(8, std::max<int64_t>(1, std::llround(std::sqrt((double)M * t_row_us / t_panel_us))));
    }
    P = std::max<int64_t>(1, std::min<int64_t>(P, M));
    int64_t rows = (M + P - 1) / P;
    if (P > 1) rows = (int64_t)round_up((size_t)rows, 128);
    return std::min(rows, M);
}

// rows x cols floats between two row-strided buffers.  Equal strides take
// one linear copy of the whole span (the driver's pitched copies run slower),
// which also moves the gap columns; callers use it only where that is
// harmless (the destination's gaps are the library's own buffer).
bool copy_rows(void *dst, int64_t dld, const void *src, int64_t sld, int64_t cols, int64_t rows,
               cudaStream_t s) {
    if (rows <= 0 || cols <= 0) return true;
    if (dld == sld)
        return cudaMemcpyAsync(dst, src, ((size_t)(rows - 1) * sld + cols) * sizeof(float),
                               cudaMemcpyDefault, s) == cudaSuccess;
    return cudaMemcpy2DAsync(dst, (size_t)dld * sizeof(float), src, (size_t)sld * sizeof(float),
                             (size_t)cols * sizeof(float), (size_t)rows, cudaMemcpyDefault,
                             s) == cudaSuccess;
}

// Leading dimension of the device copy of a host operand read with leading
// dimension `ld`: the same (so one linear copy moves it) when the gaps are
// small and, where the kernels want it, ld % 4 == 0; otherwise the row
// length rounded up to 4.
int64_t device_ld(int64_t ld, int64_t cols, bool want_mult4) {
    const bool keep = ld <= cols + 64 && (!want_mult4 || ld % 4 == 0);
    return keep ? std::max<int64_t>(ld, 1) : (int64_t)round_up((size_t)std::max<int64_t>(cols, 1), 4);
}

}  // namespace

namespace sgemm_gb300 {
// Frees the device buffers, streams and events of every host path (called by
// sgemm_release_workspaces).  Returns false if a CUDA call failed.
bool release_host_paths() {
    std::lock_guard<std::mutex> lock(g_mu);
    int cur = 0;
    if (cudaGetDevice(&cur) != cudaSuccess) return false;
    bool ok = true;
    for (auto &kv : g_paths) {
        HostPath &h = kv.second;
        std::lock_guard<std::mutex> plock(h.mu);
        if (!h.ready) continue;
        if (cudaSetDevice(kv.first.first) != cudaSuccess ||
            cudaStreamSynchronize(h.up) != cudaSuccess ||
            cudaStreamSynchronize(h.down) != cudaSuccess ||
            cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(kv.first.second)) != cudaSuccess)
            ok = false;
        destroy(h);
    }
    g_paths.clear();
    if (cudaSetDevice(cur) != cudaSuccess) ok = false;
    return ok;
}
}  // namespace sgemm_gb300

extern "C" {

int sgemm_host(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
               const float *B, int64_t ldb, float beta, float *C, int64_t ldc, int mode,
               void *stream) {
    // Argument checks on the host pointers (sizes, leading dimensions, NULL,
    // overlap of C with A or B, the mode); nothing is touched yet.
    const int kid = sgemm_select_kernel(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, mode);
    if (kid < 0) return kid;
    if (kid == SGEMM_KERNEL_NONE) return SGEMM_OK;
    // Not capturable (and the device set-up below may synchronise).
    cudaStream_t S = static_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(S, &cs) != cudaSuccess) {
        (void)cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    if (cs != cudaStreamCaptureStatusNone) return SGEMM_ERR_CAPTURE;
    GemmArgs probe{};
    int rc = fill_device_args(probe);   // the current device must be an sm_103 GPU
    if (rc != SGEMM_OK) return rc;
    const bool uses_ab = kid != SGEMM_KERNEL_SCALE_C;
    const bool reads_c = beta != 0.0f;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_ERR_CUDA;
    HostPath *hp = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        hp = &g_paths[{dev, reinterpret_cast<uintptr_t>(S)}];
    }
    HostPath &h = *hp;
    std::lock_guard<std::mutex> plock(h.mu);
    rc = create(h);
    if (rc != SGEMM_OK) return rc;

    // Device layout: B (K x ldb_d), then per slot an A panel (rows x lda_d)
    // and a C panel (rows x ldc_d).  B's leading dimension is a multiple of 4
    // so B qualifies for the TMA-staged kernels.  C keeps the host's only
    // when the host rows are contiguous: the copy back must not write the
    // caller's gap columns.
    const int64_t rows = panel_rows(M, N, K, uses_ab);
    const int64_t lda_d = uses_ab ? device_ld(lda, K, false) : 1;
    const int64_t ldb_d = uses_ab ? device_ld(ldb, N, true) : 1;
    const int64_t ldc_d = ldc == N ? N : (int64_t)round_up((size_t)N, 4);
    const size_t b_bytes = uses_ab ? round_up((size_t)K * ldb_d * sizeof(float), kAlign) : 0;
    const size_t a_bytes = uses_ab ? round_up((size_t)rows * lda_d * sizeof(float), kAlign) : 0;
    const size_t c_bytes = round_up((size_t)rows * ldc_d * sizeof(float), kAlign);
    const size_t need = b_bytes + kSlots * (a_bytes + c_bytes);
    if (h.bytes < need) {
        // Stream-ordered on `stream`: every earlier call joined back into it,
        // and this call's other streams start from the fork event below.
        const size_t nb = round_up(std::max(need, h.bytes + h.bytes / 2), size_t(2) << 20);
        if (h.buf != nullptr && cudaFreeAsync(h.buf, S) != cudaSuccess) return SGEMM_ERR_CUDA;
        h.buf = nullptr;
        h.bytes = 0;
        if (cudaMallocAsync(&h.buf, nb, S) != cudaSuccess) {
            (void)cudaGetLastError();
            h.buf = nullptr;
            return SGEMM_ERR_CUDA;
        }
        h.bytes = nb;
    }
    unsigned char *base = static_cast<unsigned char *>(h.buf);
    float *dB = reinterpret_cast<float *>(base);
    float *dA[kSlots], *dC[kSlots];
    for (int s = 0; s < kSlots; ++s) {
        dA[s] = reinterpret_cast<float *>(base + b_bytes + s * (a_bytes + c_bytes));
        dC[s] = reinterpret_cast<float *>(base + b_bytes + s * (a_bytes + c_bytes) + a_bytes);
    }

    const int nb = b_parts(M, rows, K, uses_ab);
    const int64_t kc = (K + nb - 1) / nb;   // rows of B per K-range
    bool ok = cudaEventRecord(h.fork, S) == cudaSuccess &&
              cudaStreamWaitEvent(h.up, h.fork, 0) == cudaSuccess &&
              cudaStreamWaitEvent(h.down, h.fork, 0) == cudaSuccess;
    if (ok && uses_ab && nb == 1) ok = copy_rows(dB, ldb_d, B, ldb, N, K, h.up);
    rc = ok ? SGEMM_OK : SGEMM_ERR_CUDA;
    for (int64_t r0 = 0, p = 0; rc == SGEMM_OK && r0 < M; r0 += rows, ++p) {
        const int s = (int)(p % kSlots);
        const int64_t mp = std::min(rows, M - r0);
        // the slot is free once the panel that used it last went back to the host
        if (p >= kSlots) ok = cudaStreamWaitEvent(h.up, h.stored[s], 0) == cudaSuccess;
        if (ok && uses_ab) ok = copy_rows(dA[s], lda_d, A + r0 * lda, lda, K, mp, h.up);
        if (ok && reads_c) ok = copy_rows(dC[s], ldc_d, C + r0 * ldc, ldc, N, mp, h.up);
        ok = ok && cudaEventRecord(h.loaded[s], h.up) == cudaSuccess;
        if (p == 0 && nb > 1) {   // B follows A_0 and C_0, one K-range at a time
            for (int j = 0; ok && j < nb; ++j) {
                const int64_t k0 = j * kc, kn = std::min(kc, K - k0);
                ok = copy_rows(dB + k0 * ldb_d, ldb_d, B + k0 * ldb, ldb, N, kn, h.up) &&
                     cudaEventRecord(h.bpart[j], h.up) == cudaSuccess;
            }
        }
        ok = ok && cudaStreamWaitEvent(S, h.loaded[s], 0) == cudaSuccess;
        if (!ok) {
            rc = SGEMM_ERR_CUDA;
            break;
        }
        if (p == 0 && nb > 1) {
            for (int j = 0; rc == SGEMM_OK && j < nb; ++j) {
                const int64_t k0 = j * kc, kn = std::min(kc, K - k0);
                if (cudaStreamWaitEvent(S, h.bpart[j], 0) != cudaSuccess) {
                    rc = SGEMM_ERR_CUDA;
                    break;
                }
                rc = sgemm_fused(mp, N, kn, alpha, dA[s] + k0, lda_d, dB + k0 * ldb_d, ldb_d,
                                 j == 0 ? beta : 1.0f, dC[s], ldc_d, nullptr, SGEMM_ACT_NONE,
                                 mode, stream);
            }
        } else {
            rc = sgemm_fused(mp, N, K, alpha, uses_ab ? dA[s] : nullptr, lda_d,
                             uses_ab ? dB : nullptr, ldb_d, beta, dC[s], ldc_d, nullptr,
                             SGEMM_ACT_NONE, mode, stream);
        }
        if (rc != SGEMM_OK) break;
        ok = cudaEventRecord(h.computed[s], S) == cudaSuccess &&
             cudaStreamWaitEvent(h.down, h.computed[s], 0) == cudaSuccess &&
             copy_rows(C + r0 * ldc, ldc, dC[s], ldc_d, N, mp, h.down) &&
             cudaEventRecord(h.stored[s], h.down) == cudaSuccess;
        if (!ok) rc = SGEMM_ERR_CUDA;
    }
    // Join: `stream` waits for everything enqueued on both copy streams,
    // whatever happened above (after an error some copies up may not have
    // been waited for yet), so that later work on `stream` -- a buffer
    // release or regrowth included -- is ordered after them.
    const bool joined = cudaEventRecord(h.join, h.up) == cudaSuccess &&
                        cudaStreamWaitEvent(S, h.join, 0) == cudaSuccess &&
                        cudaEventRecord(h.join, h.down) == cudaSuccess &&
                        cudaStreamWaitEvent(S, h.join, 0) == cudaSuccess;
    if (rc == SGEMM_OK && !joined) rc = SGEMM_ERR_CUDA;
    if (rc == SGEMM_ERR_CUDA) (void)cudaGetLastError();
    return rc;
}

int sgemm_host_set_panels(int panels) {
    if (panels < 0) return SGEMM_ERR_BAD_ARG;
    return g_panels.exchange(panels);
}

int64_t sgemm_host_panel_rows(int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_BAD_DIM;
    if (M == 0) return 0;
    return panel_rows(M, N, K, K > 0);
}

}  // extern "C"
