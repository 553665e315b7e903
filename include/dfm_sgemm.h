/*
 * dfm_sgemm.h -- C ABI of the GB300 (sm_103a) FP32 matrix-product library.
 *
 * The operation (all entry points that compute):
 *
 *     C[i*ldc + j] = sum_{k=0}^{K-1} A[i*lda + k] * B[k*ldb + j]
 *                    for 0 <= i < M, 0 <= j < N
 *
 * with A (M x K), B (K x N) and C (M x N) row-major fp32 with leading
 * dimensions lda, ldb, ldc in elements. Definitions followed:
 *   - "CUDA 算子优化：GEMM" (llm-tech.com.cn/posts/cuda-gemm), section
 *     "矩阵乘法": C_ij = sum_k A_ik B_kj, A M x K, B K x N, 2MNK flops.
 *   - "GEMM from naive to tiled" (arganzheng.life), section 二.1: FP32,
 *     row-major, C = A * B; section 三.1: kernels take const float*
 *     __restrict__ A, B and write float* C; section 七: shapes that are not
 *     multiples of the tile are handled by zero-filled loads and predicated
 *     stores.
 *   - hotelren.com/news/4711315 (inner vs outer product GEMM), section 4.2:
 *     the leading dimension is passed separately from the logical width.
 *
 * Semantics shared by every computing entry point:
 *   - C is overwritten (alpha = 1, beta = 0). Elements of C outside
 *     i < M, j < N (the pitch padding ldc > N) are never written. A and B
 *     are only read inside their logical extent (never in the padding).
 *   - Accuracy contract: every element satisfies
 *       |C_ij - sum_k A_ik B_kj| <= 1e-4 * sum_k |A_ik B_kj| + 1e-6
 *     and results are exact on integer-valued inputs whose partial sums stay
 *     below 2^24 in magnitude. Results are deterministic run to run for a
 *     given shape, layout, path and device.
 *   - Arithmetic: the CUDA-core paths use one fp32 fused multiply-add per
 *     product (k in an implementation order). The tensor-core path
 *     (SGEMM_PATH_TF32X3, chosen by sgemm for 16-byte-aligned operands in
 *     SGEMM_MATH_AUTO) splits each operand x = hi + lo into TF32 parts and
 *     sums A_lo B_hi + A_hi B_lo + A_hi B_hi in fp32: each product carries a
 *     relative error below about 3 * 2^-20, well inside the contract. An
 *     Inf input comes out as NaN on that path (Inf times a zero residual).
 *     sgemm_set_math_mode(SGEMM_MATH_FFMA) restricts sgemm to the CUDA-core
 *     paths.
 *   - M == 0 or N == 0: nothing is done. K == 0: C[0:M, 0:N] is set to 0.
 *   - NaN / Inf inputs propagate as IEEE fp32 arithmetic gives them.
 *
 * Memory and streams:
 *   - A, B, C are device pointers of the calling thread's current CUDA
 *     device, owned by the caller. Alignment is never an error: pointers or
 *     leading dimensions that rule out 16-byte vector / TMA access select a
 *     slower path of the same result class.
 *   - C must not overlap A or B (SGEMM_ERR_OVERLAP).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Every call is asynchronous on that stream; the library never
 *     synchronises. Errors found on the host are returned before anything is
 *     enqueued.
 *   - Workspaces. Some paths need device memory beyond A, B and C: stream-K
 *     partial tiles and tile counters, split-k pieces, row-major copies of
 *     transposed operands for the CUDA-core kernels, and 16-byte-aligned
 *     copies of misaligned operands for the tensor-core kernels (and, from
 *     2^32 multiply-adds with neither operand transposed, for the TMA-fed
 *     CUDA-core tile kernel in SGEMM_MATH_FFMA). The library
 *     keeps these in per-device workspaces, each serving one stream at a
 *     time, at most 8 per device unless stream captures hold all 8
 *     (sgemm_workspace_info reports them); they live until the process
 *     exits. A call allocates only when its stream
 *     has no workspace yet or needs a larger one: it then calls cudaMalloc,
 *     and cudaFree for the outgrown buffer after waiting on the host for
 *     that workspace's previous call, and these may synchronise the device.
 *     A call whose needs fit its stream's workspace allocates nothing and
 *     does not synchronise. With 8 workspaces in use, a ninth stream takes
 *     the least recently used one, ordered after its last call by an event
 *     wait on the device (no host synchronisation). A workspace used inside
 *     a stream capture stays with its stream for good (the graph holds its
 *     addresses). Make the first call of the largest shape on a stream
 *     outside any capture: allocation is not allowed while capturing in the
 *     global capture mode. sgemm_noalloc never allocates.
 *   - The first call on a device does one-time set-up (device query, kernel
 *     attributes, the address of the per-device status word); make that
 *     first call outside any stream capture.
 *
 * Status codes: 0 on success, a negative SGEMM_ERR_* value otherwise;
 * sgemm_status_string() names each.
 */
#ifndef DFM_SGEMM_H
#define DFM_SGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SGEMM_OK 0
#define SGEMM_ERR_INVALID_VALUE (-1)    /* negative size or ld below width  */
#define SGEMM_ERR_NULL_POINTER (-2)     /* null pointer with elements to use */
#define SGEMM_ERR_UNSUPPORTED_DEVICE (-3) /* current device is not sm_103  */
#define SGEMM_ERR_LAUNCH (-4)           /* kernel launch failed            */
#define SGEMM_ERR_WATCHDOG (-5)         /* a bounded device wait timed out  */
#define SGEMM_ERR_OVERLAP (-6)          /* C overlaps A or B               */
#define SGEMM_ERR_CUDA (-7)             /* another CUDA runtime error      */
#define SGEMM_ERR_PATH (-8)             /* forced path cannot take the call */
#define SGEMM_ERR_TOO_LARGE (-9)        /* size beyond a path's limit      */

/* Math modes (sgemm_set_math_mode). */
#define SGEMM_MATH_AUTO 0  /* fastest path within the accuracy contract     */
#define SGEMM_MATH_FFMA 1  /* CUDA-core fp32 fused multiply-add paths only   */

/* Operand forms (sgemm_ex): op(X) = X or its transpose. */
#define SGEMM_OP_N 0  /* as stored, row-major                               */
#define SGEMM_OP_T 1  /* transposed: the stored rows are op(X)'s columns    */

/* Kernel paths (sgemm_path / sgemm_plan). */
#define SGEMM_PATH_AUTO 0
#define SGEMM_PATH_TILED_TMA 1  /* TMA-fed multistage tile kernel (aligned) */
#define SGEMM_PATH_TILED_LDG 2  /* same tile core, 4-byte async loads     */
#define SGEMM_PATH_GEMV_ROW 3   /* M == 1: c = a * B, column blocks (also
                                   c = A^T b as c^T = b^T A, sgemm_ex)     */
#define SGEMM_PATH_GEMV_COL 4   /* N == 1: c = A * b, one warp per row     */
#define SGEMM_PATH_NAIVE 5      /* one thread per output (debug baseline)  */
#define SGEMM_PATH_TF32X3 6     /* tensor cores, 3 TF32 products (aligned)  */
#define SGEMM_PATH_TF32X3_PAIR 7 /* same on 2-SM pairs, 256 x 256 tiles     */
#define SGEMM_PATH_SMALL 8      /* 32 x 32 tiles, plain loads: products too
                                   small to fill the GPU (any layout)      */
#define SGEMM_PATH_COUNT 9

/*
 * sgemm: C = A * B as described above, on `stream`.
 * Arguments: M, N, K >= 0; lda >= max(1, K); ldb >= max(1, N);
 * ldc >= max(1, N). Pointers may be NULL only when the matrix has no
 * elements to read or write.
 * Errors: SGEMM_ERR_INVALID_VALUE, SGEMM_ERR_NULL_POINTER,
 * SGEMM_ERR_OVERLAP, SGEMM_ERR_UNSUPPORTED_DEVICE, SGEMM_ERR_CUDA,
 * SGEMM_ERR_LAUNCH. Watchdog timeouts are reported afterwards by
 * sgemm_watchdog_status().
 */
int sgemm(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
          const float* B, int64_t ldb, float* C, int64_t ldc, void* stream);

/*
 * sgemm_path: as sgemm, but runs the kernel path `path` (SGEMM_PATH_*)
 * instead of the one sgemm would choose. Returns SGEMM_ERR_PATH when that
 * path cannot take the arguments (e.g. TILED_TMA with an ld that is not a
 * multiple of 4, GEMV_ROW with M != 1). Meant for tests and measurement.
 */
int sgemm_path(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
               const float* B, int64_t ldb, float* C, int64_t ldc,
               void* stream, int path);

/*
 * sgemm_ex: C = alpha * op(A) * op(B) + beta * C, on `stream`.
 *   op(A) is M x K: op_a == SGEMM_OP_N, A stored M x K (row i at A + i*lda,
 *   lda >= max(1, K)); SGEMM_OP_T, A stored K x M (op(A)_ik = A[k*lda + i],
 *   lda >= max(1, M)).
 *   op(B) is K x N: op_b == SGEMM_OP_N, B stored K x N (ldb >= max(1, N));
 *   SGEMM_OP_T, B stored N x K (op(B)_kj = B[j*ldb + k], ldb >= max(1, K)).
 *   C is M x N (ldc >= max(1, N)); its pitch padding is never touched.
 * BLAS conventions: with beta == 0, C is not read (it may hold NaN); with
 * alpha == 0 or K == 0, A and B are not read (may be NULL) and C = beta * C
 * (C untouched when beta == 1). sgemm(...) is sgemm_ex(SGEMM_OP_N,
 * SGEMM_OP_N, ..., alpha = 1, ..., beta = 0, ...), with identical results.
 * The pages compute only the plain product; the operand forms and scalars
 * are the BLAS reading of the cuBLAS call they discuss ("GEMM from naive to
 * tiled", sections 二.2, 九.2). Accuracy: every element satisfies
 *   |C - C_exact| <= 1e-4 * (|alpha| * sum_k |op(A)_ik op(B)_kj|
 *                            + |beta * C_old|) + 1e-6.
 * The tensor-core kernels read transposed operands in place; the CUDA-core
 * kernels get row-major copies made in the stream's workspace (a
 * bandwidth-bound transpose, grown like the stream-K workspace). The
 * vector shapes need no copy: with M == 1, c = a * op(B) streams B as
 * stored; with N == 1, op_a == SGEMM_OP_T and contiguous c and b (ldc == 1,
 * b a row or a column with ldb == 1), c = A^T b streams A as stored as the
 * row product c^T = b^T A.
 * Errors: as sgemm, plus SGEMM_ERR_INVALID_VALUE for an unknown op.
 */
int sgemm_ex(int op_a, int op_b, int64_t M, int64_t N, int64_t K,
             float alpha, const float* A, int64_t lda, const float* B,
             int64_t ldb, float beta, float* C, int64_t ldc, void* stream);

/* sgemm_ex_path: sgemm_ex on a forced kernel path (as sgemm_path). */
int sgemm_ex_path(int op_a, int op_b, int64_t M, int64_t N, int64_t K,
                  float alpha, const float* A, int64_t lda, const float* B,
                  int64_t ldb, float beta, float* C, int64_t ldc, void* stream,
                  int path);

/*
 * sgemm_plan_ex: the kernel path sgemm_ex would take (for alpha != 0),
 * decided on the host only; as sgemm_plan.
 */
int sgemm_plan_ex(int op_a, int op_b, int64_t M, int64_t N, int64_t K,
                  int64_t lda, int64_t ldb, int64_t ldc, uint64_t a_addr,
                  uint64_t b_addr, uint64_t c_addr, int* path);

/*
 * sgemm_strided_batched: `batch` independent products
 *   C_b = alpha * op(A_b) * op(B_b) + beta * C_b,   b = 0 .. batch - 1,
 * with A_b = A + b * stride_a, B_b = B + b * stride_b, C_b = C + b * stride_c
 * (strides in floats, >= 0; a stride of 0 shares that operand between all
 * items, e.g. one weight matrix applied to a batch). Each item follows
 * sgemm_ex (same forms, scalars, accuracy and unread-operand rules). The
 * items of C must not share memory: either stacked, stride_c >= (M - 1) *
 * ldc + N, or side by side in one row pitch, stride_c >= N and
 * (batch - 1) * stride_c + N <= ldc; otherwise SGEMM_ERR_INVALID_VALUE.
 * C must not overlap any item of A or B (SGEMM_ERR_OVERLAP). batch == 0 is
 * a no-op. With 16-byte-aligned operands and strides that are multiples of
 * 4 floats, the tensor-core kernels take the whole batch in one launch
 * (one persistent schedule over the tiles of all items, so a shared
 * operand is fetched from memory once for all of them: the batched product
 * with a shared A that "如何让计算受限问题真正达到计算受限" (section 5.3,
 * fusion) gives as an example of reading data once for several
 * consumers); otherwise the items run one by one.
 */
int sgemm_strided_batched(int op_a, int op_b, int64_t M, int64_t N,
                          int64_t K, float alpha, const float* A, int64_t lda,
                          int64_t stride_a, const float* B, int64_t ldb,
                          int64_t stride_b, float beta, float* C, int64_t ldc,
                          int64_t stride_c, int64_t batch, void* stream);

/* sgemm_strided_batched_path: as above on a forced kernel path. */
int sgemm_strided_batched_path(int op_a, int op_b, int64_t M, int64_t N,
                               int64_t K, float alpha, const float* A,
                               int64_t lda, int64_t stride_a, const float* B,
                               int64_t ldb, int64_t stride_b, float beta,
                               float* C, int64_t ldc, int64_t stride_c,
                               int64_t batch, void* stream, int path);

/*
 * sgemm_set_math_mode: SGEMM_MATH_AUTO (default) or SGEMM_MATH_FFMA, for the
 * whole process, for calls that start after it returns. Returns the previous
 * mode, or SGEMM_ERR_INVALID_VALUE for an unknown mode.
 */
int sgemm_set_math_mode(int mode);

/*
 * sgemm_plan: the path sgemm would take for these arguments (in the current
 * math mode), decided on the host only (no device is touched). a_addr / b_addr / c_addr are the pointer
 * values (only their alignment is used). Writes the SGEMM_PATH_* value to
 * *path. Returns the same argument errors as sgemm (no device errors).
 */
int sgemm_plan(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
               int64_t ldc, uint64_t a_addr, uint64_t b_addr, uint64_t c_addr,
               int* path);

/*
 * sgemm_host: C = A * B for HOST matrices hA (ld lda), hB (ld ldb), hC
 * (ld ldc). The caller provides device staging buffers dA (M*K floats),
 * dB (K*N floats) and dC (M*N floats), dense (ld = K, N, N). Copies hA ->
 * dA and hB -> dB, runs the product on the staging buffers and copies
 * dC -> hC, asynchronously with respect to the host and ordered on `stream`
 * like any other work on it: it starts after the work enqueued on `stream`
 * before the call, and work enqueued on `stream` after the call starts
 * after hC has been written. hC is valid once the stream is synchronised.
 * Host buffers should be pinned (pageable memory works, without overlap).
 *
 * Large products (M >= 512 rows and M*N*K >= 2^31) are pipelined: B is
 * copied first, A in up to 4 row blocks of whole 256-row multiples on an
 * internal copy stream; each row block of C is computed on `stream` as soon
 * as its rows have landed and copied back on a second internal stream while
 * the next block computes. Each row block is computed exactly as sgemm of
 * that block, so the result meets the accuracy contract and is
 * deterministic for a given shape, but may differ in the last bits from
 * one sgemm of the whole product (the blocks can be scheduled differently).
 * The internal streams and events are per device and shared by all calls;
 * concurrent calls from several host threads are serialised while they
 * enqueue. Same errors as sgemm.
 */
int sgemm_host(int64_t M, int64_t N, int64_t K, const float* hA, int64_t lda,
               const float* hB, int64_t ldb, float* hC, int64_t ldc,
               float* dA, float* dB, float* dC, void* stream);

/*
 * sgemm_noalloc: C = A * B with the semantics, arguments and errors of
 * sgemm, for callers that must not allocate device memory at the point of
 * use -- code whose device memory is all owned by another allocator (a
 * framework's caching pool, a fixed budget), latency-critical loops that
 * cannot afford the device-wide synchronisation cudaMalloc/cudaFree imply,
 * or plug-ins in hosts that forbid allocation after start-up. sgemm() may
 * grow its stream's workspace with cudaMalloc; this entry point never calls
 * cudaMalloc, cudaFree or any allocating routine. The pages have no
 * counterpart of this entry point.
 *
 * Scratch: the stream-K partial tiles and tile counters of the TMA path live
 * in one fixed device array of 40 MiB + 512 KiB that every device which loads
 * the library holds until the process exits. Limit: a product that takes
 * the stream-K tile kernel (SGEMM_MATH_FFMA, aligned operands) may have at
 * most 16384 output tiles of 256 x 128 (e.g. M = 32768, N = 16384); a
 * larger one returns SGEMM_ERR_TOO_LARGE before any work is enqueued.
 * (The pair kernel's pieces would need 38 MiB more, so it does not use
 * the scratch.) Paths that use
 * no scratch (the tensor-core kernels, the vector kernels, the any-layout
 * tile kernel) take every size sgemm takes. The stream-K grid is capped at
 * 160 blocks; the tensor-core pair kernel runs whole tiles only (its
 * stream-K pieces would not fit) and the single-block tensor kernel does
 * not split k. Operands whose base or row stride is not 16-byte aligned
 * take the any-layout CUDA-core tile kernel (sgemm would repack them into
 * allocated memory for the tensor path, or for the TMA-fed tile kernel).
 *
 * The first call on a device fetches the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture. Every call shares the array: calls whose
 * kernels may overlap on the GPU (unordered streams) race and must be
 * ordered by the caller. Each call clears the counters it uses on `stream`
 * before its kernel runs. Results may differ from sgemm() in the last bits
 * (a different stream-K split changes the fp32 summation order); both are
 * deterministic and exact on small-integer inputs.
 */
int sgemm_noalloc(int64_t M, int64_t N, int64_t K, const float* A,
                  int64_t lda, const float* B, int64_t ldb, float* C,
                  int64_t ldc, void* stream);

/*
 * sgemm_watchdog_status: every wait inside the kernels (on an mbarrier or a
 * peer block's flag) is bounded; on timeout the kernel records the failure
 * in a per-device status word, abandons its tile and exits without trapping.
 * This call reads and clears that word for the current device. Call it after
 * synchronising the streams that ran sgemm. Returns SGEMM_OK or
 * SGEMM_ERR_WATCHDOG (then *site, if not NULL, receives the wait-site id),
 * or SGEMM_ERR_CUDA.
 */
int sgemm_watchdog_status(int* site);

/*
 * sgemm_watchdog_selftest: launches one block that waits on an mbarrier
 * nothing ever arrives at, with the same bounded-wait code the kernels use
 * and a limit of `timeout_ns` (clamped to [1e6, 2e9] ns). Synchronises the
 * stream and returns what sgemm_watchdog_status then reports (expected:
 * SGEMM_ERR_WATCHDOG). Used to test failure detection without a GPU fault.
 */
int sgemm_watchdog_selftest(void* stream, int64_t timeout_ns);

/*
 * sgemm_workspace_info: the workspaces the library holds on the current
 * device: their number (*count) and their total size in bytes
 * (*bytes). Either pointer may be NULL. Host only; returns SGEMM_OK, or
 * the set-up errors of sgemm. No counterpart on the pages (a diagnostic of
 * this library's memory use).
 */
int sgemm_workspace_info(int* count, int64_t* bytes);

/*
 * sgemm_launch_count: how many kernel launches this library has issued in
 * this process, on all devices and streams, counting each launch the CUDA
 * runtime accepted (memsets and copies are not kernels and are not
 * counted). Host only, never fails; the difference of two readings is the
 * number of the library's kernels enqueued between them. No counterpart on
 * the pages (a diagnostic of this library's work).
 */
uint64_t sgemm_launch_count(void);

/* Human-readable name of a status code (static storage). */
const char* sgemm_status_string(int status);

/* Name of an SGEMM_PATH_* value (static storage), "?" when unknown. */
const char* sgemm_path_name(int path);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int sgemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DFM_SGEMM_H */
