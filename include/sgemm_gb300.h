/*
 * sgemm_gb300.h -- C ABI of the GB300 (sm_103a) single-precision GEMM library.
 *
 * The operation is the general matrix multiply of the page "GPU GEMM 优化完全拆解
 * （一）：从朴素 Kernel 到共享内存分块", section "什么是 GEMM":
 *
 *     C <- alpha * A @ B + beta * C
 *
 * with A an M x K matrix, B K x N and C M x N, all row-major: element (i, j)
 * of a matrix with leading dimension ld is at ptr[i * ld + j] (the indexing of
 * the naive kernel on "CUDA 矩阵乘法优化：从朴素 Kernel 到接近 cuBLAS", section
 * "1. Kernel 1", generalised from ld = row length to any ld >= row length).
 *
 * Conventions shared by every entry point below
 * -----------------------------------------------
 * Memory      All matrix pointers are DEVICE pointers on the current CUDA
 *             device.  The caller owns every buffer; the library never frees
 *             or keeps a caller pointer past the call.  A and B are read-only.
 *             The FFMA path (M > 16) stages A through a transposed copy in a
 *             library workspace: K x round_up(M, 4) floats per (device,
 *             stream), grown on first need with cudaMallocAsync on `stream`
 *             and kept for later calls (sgemm_release_workspaces frees it).
 * Stream      `stream` is a cudaStream_t (NULL = the legacy default stream).
 *             Every call is asynchronous with respect to the host: work is
 *             enqueued on `stream` and the call returns without waiting.
 * Sizes       M, N, K >= 0.  lda >= K, ldb >= N, ldc >= N whenever that
 *             matrix is non-empty and read or written.
 * Quick paths M == 0 or N == 0: nothing is done.  K == 0 or alpha == 0:
 *             C <- beta * C and A, B are not read.  beta == 0: C is written
 *             without being read, so NaN or Inf already in C does not reach
 *             the result (the BLAS convention; the pages always read C).
 * Aliasing    C must not overlap A or B (checked on the address ranges the
 *             call would touch).
 * Alignment   Any float-aligned pointer and any ld are accepted.  When B is
 *             16-byte aligned with ldb % 4 == 0 the TMA-staged kernel runs
 *             (A and C may have any alignment); otherwise a slower kernel with
 *             plain loads does.
 * Accuracy    sgemm: FP32 FFMA arithmetic, each output a sum of K fp32
 *             products accumulated in fp32 (order differs from a serial
 *             loop).  sgemm_3xtf32: tensor-core TF32 products with the
 *             operands split into high and low TF32 parts, FP32 accumulation.
 *             Both are held to max|C - C_ref| / (K * max|A| * max|B|) <= 1e-6
 *             against an fp64 reference; small-integer inputs are exact.
 * Errors      Return values are SGEMM_* status codes (0 = success).
 *             Argument errors are detected on the host before anything is
 *             enqueued, and nothing is written.  Errors inside a kernel
 *             (a bounded wait that ran out) are recorded in a per-device
 *             word and reported by sgemm_status().
 * Threads     Entry points may be called from several host threads at once.
 */
#ifndef SGEMM_GB300_H
#define SGEMM_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define SGEMM_OK              0
#define SGEMM_ERR_BAD_DIM    -1   /* M, N or K negative, or a size too large to index */
#define SGEMM_ERR_BAD_LD     -2   /* lda < K, ldb < N or ldc < N for a matrix in use */
#define SGEMM_ERR_NULL_PTR   -3   /* a pointer the call needs is NULL */
#define SGEMM_ERR_ALIAS      -4   /* C overlaps A or B */
#define SGEMM_ERR_CUDA       -5   /* a CUDA runtime or driver call failed */
#define SGEMM_ERR_DEVICE     -6   /* the current device is not an sm_103 GPU */
#define SGEMM_ERR_TIMEOUT    -7   /* a device-side bounded wait ran out (from sgemm_status) */
#define SGEMM_ERR_BAD_ARG    -8   /* any other invalid argument */
#define SGEMM_ERR_TOO_LARGE  -9   /* beyond sgemm_noalloc's fixed scratch */
#define SGEMM_ERR_CAPTURE   -10   /* the stream is being captured and the call would allocate */

/* Kernel identifiers, for sgemm_select_kernel and sgemm_force_kernel. */
#define SGEMM_KERNEL_AUTO          0   /* library's choice (sgemm_force_kernel only) */
#define SGEMM_KERNEL_NONE          1   /* quick return, nothing launched */
#define SGEMM_KERNEL_SCALE_C       2   /* C <- beta*C only (K == 0 or alpha == 0) */
#define SGEMM_KERNEL_FFMA_TMA      3   /* TMA-staged, warp-tiled FFMA kernel */
#define SGEMM_KERNEL_FFMA_GENERIC  4   /* plain-load tiled FFMA kernel, any alignment */
#define SGEMM_KERNEL_DECODE        5   /* split-K streaming kernel for M <= 16 */
#define SGEMM_KERNEL_TF32X3        6   /* 3xTF32 tensor-core kernel (sgemm_3xtf32) */
#define SGEMM_KERNEL_TF32          7   /* 1xTF32 tensor-core kernel (sgemm_tf32) */
#define SGEMM_KERNEL_BF16          8   /* BF16 tensor-core kernel (sgemm_bf16) */

/* Activations of sgemm_fused's epilogue. */
#define SGEMM_ACT_NONE   0   /* identity */
#define SGEMM_ACT_RELU   1   /* x < 0 ? 0 : x (NaN stays NaN) */
#define SGEMM_ACT_GELU   2   /* x/2 * (1 + tanh(sqrt(2/pi) * (x + 0.044715 x^3))) */
#define SGEMM_ACT_SILU   3   /* x / (1 + exp(-x)) */

/* Arithmetic of a call, for sgemm_select_kernel's and sgemm_fused's `mode`. */
#define SGEMM_MODE_FP32    0   /* sgemm() */
#define SGEMM_MODE_3XTF32  1   /* sgemm_3xtf32() */
#define SGEMM_MODE_TF32    2   /* sgemm_tf32() */
#define SGEMM_MODE_BF16    3   /* sgemm_bf16() */

/*
 * sgemm -- C <- alpha * A @ B + beta * C in FP32 (FFMA) arithmetic.
 *
 *   M, N, K   matrix sizes (A: M x K, B: K x N, C: M x N), each >= 0
 *   alpha     scale of the product
 *   A, lda    device pointer to A and its row stride in elements
 *   B, ldb    device pointer to B and its row stride in elements
 *   beta      scale of the incoming C
 *   C, ldc    device pointer to C (read when beta != 0, always written) and
 *             its row stride in elements
 *   stream    cudaStream_t to enqueue on
 *
 * Shapes with M <= 16 run the split-K streaming kernel (the decode regime of
 * "GPU GEMM 优化完全拆解（一）", section "LLM 推理本质上是 GEMM 的串联"); the rest
 * run the tiled FFMA kernel (products of at most 2^21 multiply-adds, such as
 * 128^3, the plain-load tiled kernel in a single launch).  The tiles left
 * after the last full wave of resident blocks -- all tiles, when they do not
 * fill one wave -- may be divided by work: equal runs of K iterations whose
 * partial tiles are summed in a fixed order (the split-K reduction of "CUDA
 * 矩阵乘法优化：从朴素 Kernel 到接近 cuBLAS", section "10", applied to the tail
 * only).  The result is deterministic: the same inputs give the same bits on
 * every call on the same GPU model.
 * Stream order: the decode kernel, and the FFMA kernel behind its transpose,
 * are launched as programmatic dependents of the work before them on
 * `stream`: their blocks may start their set-up while that work finishes,
 * and wait for it to complete before touching A, B or C.  The decode kernel
 * lets the next such launch start once its blocks are past their K loop.
 * CUDA graphs: calls can be captured on `stream` (and the graph replayed)
 * once a call of the same shape has run eagerly on the same stream and
 * device: that call sets up the device and sizes the stream's workspace.  A
 * captured call never allocates: one that would need a larger workspace
 * returns SGEMM_ERR_CAPTURE with nothing enqueued.
 * Returns SGEMM_OK, or an argument/launch error code (nothing enqueued).
 */
int sgemm(int64_t M, int64_t N, int64_t K, float alpha,
          const float *A, int64_t lda, const float *B, int64_t ldb,
          float beta, float *C, int64_t ldc, void *stream);

/*
 * sgemm_3xtf32 -- the same operation on the tcgen05 tensor cores.
 *
 * Each operand x is split into hi = tf32(x) and lo = tf32(x - hi); the
 * kernel accumulates hi*hi + hi*lo + lo*hi in FP32 tensor memory, which keeps
 * single-precision accuracy (the 3xTF32 error-compensated split of Ootomo and
 * Yokota, 2022).  Arguments, conventions and errors are those of sgemm().
 * The operands are split into a workspace first (A as [M][K] hi/lo
 * arrays, B transposed to [N][K] hi/lo arrays: 2*(M+N)*round_up(K,4)
 * floats, grown like sgemm()'s workspace), so any alignment and ld are
 * accepted.  Skinny products (M <= 16) run sgemm()'s decode kernel.
 * Infinite inputs give NaN on this path (hi - inf is not finite).
 */
int sgemm_3xtf32(int64_t M, int64_t N, int64_t K, float alpha,
                 const float *A, int64_t lda, const float *B, int64_t ldb,
                 float beta, float *C, int64_t ldc, void *stream);

/*
 * sgemm_tf32 -- reduced-precision product on the tcgen05 tensor cores
 * (opt-in; TF32 is named on "CUDA 矩阵乘法优化：从朴素 Kernel 到接近 cuBLAS",
 * results-table note).
 *
 * Accuracy contract: A and B are first rounded to TF32 (FP32's sign and
 * exponent, 10 stored mantissa bits; round to nearest, ties away from zero),
 * and the result is the FP32-accumulated product of the rounded operands,
 * C = alpha * round(A) @ round(B) + beta * C.  Against that definition the
 * result meets sgemm()'s FP32 accuracy; against the unrounded product its
 * error is that of the input rounding, up to 2^-11 relative per operand
 * (about 1e-5 of K*max|A|*max|B| for random data at K = 4096).  Operands
 * that are already TF32 values (small integers, for instance) give the same
 * result as sgemm_3xtf32().  C is not rounded.
 * The operands are rounded into a workspace first (A as [M][K], B
 * transposed to [N][K]: (M+N)*round_up(K,4) floats, grown like sgemm()'s),
 * so any alignment and ld are accepted.  Skinny products (M <= 16) run
 * sgemm()'s FP32 decode kernel, which is more accurate than the contract.
 * Arguments, conventions and errors are those of sgemm().
 */
int sgemm_tf32(int64_t M, int64_t N, int64_t K, float alpha,
               const float *A, int64_t lda, const float *B, int64_t ldb,
               float beta, float *C, int64_t ldc, void *stream);

/*
 * sgemm_bf16 -- reduced-precision product on the BF16 tensor cores (opt-in).
 *
 * Accuracy contract: A and B are first rounded to BF16 (FP32's sign and
 * exponent, 7 stored mantissa bits; round to nearest, ties to even), and the
 * result is the FP32-accumulated product of the rounded operands,
 * C = alpha * round(A) @ round(B) + beta * C; against that definition it
 * meets sgemm()'s FP32 accuracy.  Against the unrounded product the error is
 * that of the input rounding, up to 2^-8 relative per operand.  Operands
 * that are already BF16 values (small integers, for instance) give the exact
 * FP32 product.  C is not rounded.
 * The operands are rounded into a workspace first (A as [M][K], B transposed
 * to [N][K], 16-bit: (M+N)*round_up(K,8)/2 floats), so any alignment and ld
 * are accepted.  Skinny products (M <= 16) run sgemm()'s FP32 decode kernel.
 * Arguments, conventions and errors are those of sgemm().
 */
int sgemm_bf16(int64_t M, int64_t N, int64_t K, float alpha,
               const float *A, int64_t lda, const float *B, int64_t ldb,
               float beta, float *C, int64_t ldc, void *stream);

/*
 * sgemm_fused -- sgemm() with the epilogue extended by a bias and an
 * activation, applied to each output before it is stored:
 *
 *     C = act(alpha * A @ B + beta * C + bias[j])      (j: the column)
 *
 * The pages fuse elementwise work into the producing kernel ("GPU 基础原理",
 * section "4.1 算子融合", with relu(x + 1) as the example) and feed GEMMs into
 * the transformer FFN
 * ("GPU GEMM 优化完全拆解（一）", section "LLM 推理本质上是 GEMM 的串联") but choose
 * no activation; these are the ones of such FFN blocks.
 *   bias        device pointer to N floats (one per column), or NULL for none;
 *               must not overlap C (SGEMM_ERR_ALIAS)
 *   activation  SGEMM_ACT_*; anything else is SGEMM_ERR_BAD_ARG
 *   mode        SGEMM_MODE_*: the arithmetic of sgemm(), sgemm_3xtf32(),
 *               sgemm_tf32() or sgemm_bf16(), with the same kernels and
 *               accuracy contracts
 * alpha*acc + beta*C + bias is formed in FP32 and the activation applied in
 * FP32 with CUDA's tanhf / expf.  When K == 0 or alpha == 0 the result is
 * act(beta * C + bias), A and B unread.  Other arguments, conventions and
 * errors are those of sgemm().
 */
int sgemm_fused(int64_t M, int64_t N, int64_t K, float alpha,
                const float *A, int64_t lda, const float *B, int64_t ldb,
                float beta, float *C, int64_t ldc, const float *bias, int activation,
                int mode, void *stream);

/*
 * sgemm_status -- wait for `stream`, then report and clear the current
 * device's kernel error word.  Returns SGEMM_OK, SGEMM_ERR_TIMEOUT when a
 * kernel's bounded wait ran out since the last call (that kernel skipped its
 * stores and exited; C is unspecified), or SGEMM_ERR_CUDA.
 */
int sgemm_status(void *stream);

/* Human-readable text for a status code; never NULL, static storage. */
const char *sgemm_status_string(int status);

/*
 * sgemm_select_kernel -- which SGEMM_KERNEL_* sgemm() would run for these
 * arguments (host-only, launches nothing, needs no GPU).  Returns a negative
 * status code for arguments sgemm() would reject.  `mode` is one of
 * SGEMM_MODE_*: the choice of sgemm(), sgemm_3xtf32(), sgemm_tf32() or
 * sgemm_bf16(); SGEMM_ERR_BAD_ARG for any other value.
 */
int sgemm_select_kernel(int64_t M, int64_t N, int64_t K, float alpha,
                        const float *A, int64_t lda, const float *B, int64_t ldb,
                        float beta, const float *C, int64_t ldc, int mode);

/*
 * sgemm_force_kernel -- test hook: make later calls (all host threads) run
 * kernel `id` whenever that kernel can take the arguments, instead of the
 * library's choice.  SGEMM_KERNEL_AUTO restores the default.  Returns the
 * previous setting, or SGEMM_ERR_BAD_ARG for an unknown id.
 */
int sgemm_force_kernel(int id);

/*
 * sgemm_set_wait_limit -- nanoseconds a device-side wait (a kernel waiting
 * for its own copies or warps) may last before the kernel gives up, records
 * SGEMM_ERR_TIMEOUT and exits (default 2e9 = 2 s; values < 1 restore it).
 * Applies to launches made after the call.  Returns the previous limit.
 */
int64_t sgemm_set_wait_limit(int64_t ns);

/*
 * sgemm_selftest_wait -- launch one block on `stream` that waits, with the
 * bounded-wait routine every kernel uses, on a barrier nothing completes,
 * giving up after `ns` nanoseconds.  The next sgemm_status() must then report
 * SGEMM_ERR_TIMEOUT while the context stays usable.  Returns the launch status.
 */
int sgemm_selftest_wait(int64_t ns, void *stream);

/*
 * sgemm_host -- the product of sgemm_fused(..., bias = NULL, SGEMM_ACT_NONE,
 * mode, stream) for operands that live in HOST memory.
 *
 * The pages overlap loading with computing between global and shared memory
 * ("GPU GEMM 优化完全拆解（一）", section "分块的思想：把 K 循环切成一段段":
 * double buffering and asynchronous copies hide the loads behind the
 * arithmetic) and queue work asynchronously from the host ("GPU 基础原理",
 * section "3. 第三种区间：开销").  This entry point applies the same overlap one
 * level up, between host and device memory: A and C (C only when
 * beta != 0) go to the device in row panels on a copy stream; each panel is
 * multiplied on `stream` as soon as it has arrived, and its rows of C go
 * back to the host on a second copy stream while the next panel is
 * multiplied.  Two device slots hold consecutive panels.  B travels first
 * (one panel) or, with several panels and K >= 1024, after A_0 and C_0 in 2
 * or 4 ranges of K, the first panel being multiplied range by range as B
 * arrives (C_0 = alpha*A_0 B_0 + beta*C_0, then C_0 += alpha*A_0 B_j): the
 * result then differs from a single call by the rounding of those partial
 * sums, within the FP32 accuracy of sgemm().
 *   A, B, C     HOST pointers (device pointers also work: the copies use
 *               cudaMemcpyDefault), row-major with lda, ldb, ldc as in
 *               sgemm().  Page-locked (pinned) host memory lets the copies
 *               run asynchronously and overlap; pageable memory works, but
 *               the driver then stages every copy and the call returns only
 *               once the copies back have finished.
 *   mode        SGEMM_MODE_*: the arithmetic and kernels of sgemm(),
 *               sgemm_3xtf32(), sgemm_tf32() or sgemm_bf16() (each panel is
 *               one call of that entry point, so results match it up to the
 *               kernel choice for the panel's row count).
 *   stream      the call is ordered after earlier work on `stream` and
 *               completes before later work on it: C holds the result once
 *               the stream is synchronised (cudaStreamSynchronize, or
 *               sgemm_status(stream)).  A, B and C must stay valid and C
 *               untouched until then.
 * Memory: the library keeps one device buffer per (device, stream) holding
 * B and two panels of A and C (grown with cudaMallocAsync on `stream`; freed
 * by sgemm_release_workspaces), plus two copy streams and a few events.
 * Panel rows: a multiple of 128; the count (at most 8) balances the copies
 * that no compute hides (the first panel's up, the last panel's down) against
 * a fixed cost per panel (sgemm_host_panel_rows reports it; sgemm_host_set_panels overrides the
 * panel count, 0 restores the library's choice and the previous setting is
 * returned).  Products with M <= 256 or without an A@B term run as one panel.
 * Errors: those of sgemm(); SGEMM_ERR_CAPTURE while `stream` is being
 * captured (the call is not capturable).  An error after some work was
 * enqueued still leaves `stream` ordered after that work.
 */
int sgemm_host(int64_t M, int64_t N, int64_t K, float alpha,
               const float *A, int64_t lda, const float *B, int64_t ldb,
               float beta, float *C, int64_t ldc, int mode, void *stream);
int sgemm_host_set_panels(int panels);
int64_t sgemm_host_panel_rows(int64_t M, int64_t N, int64_t K);

/*
 * sgemm_release_workspaces -- free the library's cached device workspaces
 * (the transposed copy of A that the FFMA kernel stages from; one buffer per
 * device and stream, grown with cudaMallocAsync on the call's stream) and
 * sgemm_host's device buffers, copy streams and events.
 * Waits for every stream that owns a workspace.  Call it only while no other
 * host thread is inside an sgemm call; later calls allocate again as needed.
 * Returns SGEMM_OK or SGEMM_ERR_CUDA.
 */
int sgemm_release_workspaces(void);

/*
 * sgemm_noalloc -- sgemm() for callers that must not allocate device memory.
 *
 * The reference pages have no counterpart to this entry point; it exists for
 * users of the library.  sgemm() calls cudaMallocAsync the first time a
 * stream needs a larger workspace for its transposed copy of A.  Some callers
 * cannot let any allocation happen: processes whose device memory is all
 * reserved up front by their own pool or by a host framework that forbids
 * later allocation, and latency-critical paths that cannot take an
 * allocation's cost or its possible synchronisation.  sgemm_noalloc runs the
 * same kernels, but keeps the transposed copy of A (and the partial tiles of
 * the divided tail) in a fixed array compiled into the library (a
 * file-scope __device__ array of 16,777,216 floats, 64 MiB).  It calls no
 * cudaMalloc, cudaMallocAsync, cudaFree or other allocating routine.  Where
 * the array has no room for the partial tiles beside A^T, the tail runs as
 * whole tiles, so the last bits can differ from sgemm()'s.
 *
 * Limit: shapes sgemm() runs on its FFMA tile kernel (M > 16, B 16-byte
 * aligned, ldb % 4 == 0) need K * round_up(M, 4) <= 16,777,216 floats
 * (M = K = 4096 just fits); larger ones return SGEMM_ERR_TOO_LARGE with
 * nothing enqueued.  All other shapes use no scratch and run as in sgemm().
 * A tensor-core kernel forced with sgemm_force_kernel (a test hook) needs a
 * workspace, so such a call returns SGEMM_ERR_BAD_ARG with nothing enqueued.
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current).  Make that first call
 * before any stream capture.
 * Sharing: every call on a device uses the same array, which keeps the last
 * call's contents.  Each call overwrites the part it reads before reading it,
 * so nothing has to be cleared, but calls that overlap on the GPU (on
 * different streams, or from host threads that do not order their streams)
 * race on the array: run them on one stream or serialise them.
 * The array occupies 64 MiB on each GPU where this entry point has been used,
 * until the process exits.  That holds under lazy module loading, the CUDA
 * default; with CUDA_MODULE_LOADING=EAGER the array is resident on every
 * device the process initialises, from context creation, whether or not
 * this entry point is ever called.
 * Arguments, conventions and other errors are those of sgemm().
 */
int sgemm_noalloc(int64_t M, int64_t N, int64_t K, float alpha,
                  const float *A, int64_t lda, const float *B, int64_t ldb,
                  float beta, float *C, int64_t ldc, void *stream);

/*
 * FFMA tile configurations (the autotuning of "CUDA 矩阵乘法优化：从朴素 Kernel 到
 * 接近 cuBLAS", section "8. Kernel 9: 参数自动调优", done per shape class).  The
 * library holds several compile-time tile configurations of the FFMA kernel;
 * a table written by dense_fp32_matrix_row_gb300/autotune.py from
 * measurements picks one per shape measured exactly (M, N and K) and per
 * (M, N) class otherwise.  These calls serve that script and
 * the tests; they do not change results beyond rounding order.
 *   sgemm_ffma_config_count   number of configurations (indices 0 .. n-1;
 *                             0 is the default)
 *   sgemm_ffma_config_info    tile rows BM, columns BN, depth BK, pipeline
 *                             stages, threads per CTA, CTAs per SM the
 *                             registers are sized for; 0, or SGEMM_ERR_BAD_ARG
 *                             for an unknown index or a NULL pointer
 *   sgemm_ffma_config_for     the configuration an FFMA-path call of this M, N,
 *                             K runs (host only)
 *   sgemm_ffma_force_config   make every later FFMA-path call run configuration
 *                             `idx` (-1: back to the table); returns the
 *                             previous setting, or SGEMM_ERR_BAD_ARG
 *   sgemm_ffma_force_tail_sum how later calls sum the partial tiles of a tail
 *                             divided by work: -1 the library's default (a
 *                             separate kernel over all tail tiles, launched
 *                             after the tile kernel), 0 the last unit to
 *                             reach each tile, inside the tile kernel, 1 the
 *                             separate kernel.  Both add the partials in the
 *                             same order, so results are the same bits.
 *                             Returns the previous setting, or
 *                             SGEMM_ERR_BAD_ARG for another value
 *   sgemm_ffma_tail_plan      the work list an sgemm() call of this shape runs
 *                             on the FFMA-TMA path on the current device:
 *                             *units CTAs, *span k-tiles per unit of the
 *                             divided tail (0: the tail is not divided) and
 *                             *tail_sum 1 when a separate kernel sums the
 *                             tail (the call then launches three kernels:
 *                             transpose, tiles, sum), else 0.  Host only;
 *                             SGEMM_OK, SGEMM_ERR_BAD_DIM for a dimension
 *                             < 1, SGEMM_ERR_BAD_ARG for a NULL pointer, or
 *                             SGEMM_ERR_DEVICE / SGEMM_ERR_CUDA
 */
int sgemm_ffma_config_count(void);
int sgemm_ffma_config_info(int idx, int *bm, int *bn, int *bk, int *stages, int *threads,
                           int *ctas_per_sm);
int sgemm_ffma_config_for(int64_t M, int64_t N, int64_t K);
int sgemm_ffma_force_config(int idx);
int sgemm_ffma_force_tail_sum(int mode);
int sgemm_ffma_tail_plan(int64_t M, int64_t N, int64_t K, int64_t *units, int *span, int *tail_sum);

/*
 * Kernel timing, a measurement hook (the benchmark's roofline figure uses it
 * to time the FFMA tile kernel apart from the transpose before it and the
 * tail sum after it).
 *   sgemm_kernel_timing(1)        start: every later FFMA-path call brackets
 *                                 its tile kernel with two CUDA events on its
 *                                 stream (up to 4096 launches are recorded;
 *                                 later ones are not); clears earlier records
 *   sgemm_kernel_timing(0)        stop recording
 *                                 Both return the previous state (0 or 1), or
 *                                 SGEMM_ERR_BAD_ARG for another value.
 *   sgemm_kernel_timing_result    waits for the recorded events and returns
 *                                 the tile kernels' summed time in *total_ms
 *                                 and their number in *launches; SGEMM_OK,
 *                                 SGEMM_ERR_BAD_ARG for a NULL pointer, or
 *                                 SGEMM_ERR_CUDA
 * The events sit between the transpose and the tile kernel on the stream, so
 * while recording the tile kernel does not start its set-up during the
 * transpose's tail; results are unchanged.  Not for use during stream
 * capture (the events would be captured).
 */
int sgemm_kernel_timing(int enable);
int sgemm_kernel_timing_result(double *total_ms, int64_t *launches);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int sgemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SGEMM_GB300_H */
