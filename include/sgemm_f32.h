/*
 * sgemm_f32.h -- single-precision GEMM for one NVIDIA GB300 (sm_103a), C ABI.
 *
 * Operation (all entry points that compute):
 *
 *     C = alpha * A * B + beta * C
 *
 * on row-major float32 matrices with leading dimensions, the BLAS sgemm statement with
 * op(A) = A and op(B) = B ("Lecture 4 - GPU Acceleration", CMU 11-868 notes, section 5.2
 * "Interface"), written for row-major storage the way the kernels of "SGEMM six-level
 * optimisation: evolution of the core code" index it (section 2, kernel K1: element (x, i)
 * of A at A[x * K + i], generalised here to A[x * lda + i]).
 *
 * Layout
 *   A is M x K, element (i, k) at A[i * lda + k], lda >= max(1, K).
 *   B is K x N, element (k, j) at B[k * ldb + j], ldb >= max(1, N).
 *   C is M x N, element (i, j) at C[i * ldc + j], ldc >= max(1, N).
 *   A leading dimension is the distance in elements between the starts of two consecutive
 *   rows, so a sub-matrix is passed as a pointer to its first element plus the parent's
 *   ld, with no copy (same lecture, section 5.3). Elements outside the M x N view of C are
 *   never written; elements outside the views of A and B are never read.
 *   No alignment is required. 16-byte aligned B and C with ld a multiple of 4 take the
 *   128-bit load / store paths; anything else takes 32-bit paths with the same results.
 *
 * Memory and ownership
 *   A, B and C are device pointers owned by the caller (any memory the GPU can address with
 *   a plain load: cudaMalloc, cudaMallocAsync, managed). The library keeps no pointer after
 *   the call returns. C must not overlap A or B.
 *   sgemm_f32 may allocate a workspace with a stream-ordered allocation on `stream` and
 *   free it on the same stream before returning. It holds, at its front, the copies that
 *   pre-pass kernels make before the GEMM kernel runs, and behind them split-K partial
 *   tiles (at most 64 MiB):
 *     - A^T, a K x ceil4(M) copy of A (4 * K * ceil4(M) bytes), for the plans that read A
 *       k-major: the automatic plan of every large aligned problem (268 MB at 8192^3,
 *       67 MB at 4096^3);
 *     - aligned copies of A and B (ld rounded up to a multiple of 4) when lda or ldb is not
 *       a multiple of 4 or a pointer is not 16-byte aligned;
 *   the pre-pass copies together are at most 2 GiB. The workspace comes from a memory pool
 *   the library creates per device. The pool keeps freed memory for reuse, so a repeated
 *   call does not map memory again; it holds the largest workspace a call has needed (more
 *   when calls on several streams overlap) until sgemm_f32_release_workspace() returns it
 *   or the process exits. sgemm_f32_workspace_size() reports the size a call needs;
 *   sgemm_f32_ws() takes a caller-provided workspace instead, and with
 *   sgemm_f32_workspace_size_min() bytes it needs no A^T copy: it then holds split-K
 *   partial tiles only (and aligned copies of operands TMA cannot address).
 *
 * Asynchrony
 *   Every compute call enqueues its kernels on `stream` (0 = the legacy default stream) and
 *   returns without waiting. Results are visible after the stream is synchronised.
 *   The GEMM kernels are launched with programmatic dependent launch. Their CTAs may be
 *   scheduled while the previous kernel on `stream` finishes. Each one waits for that
 *   kernel to complete (and its writes to be visible) before it reads or writes global
 *   memory, so stream order is the same as for plain launches, under stream capture too.
 *
 * Scalars and special cases (BLAS reference conventions)
 *   alpha and beta are host floats passed by value.
 *   M == 0 or N == 0: nothing is done, returns 0.
 *   alpha == 0 or K == 0: A and B are not read; C = beta * C (C = 0 when beta == 0).
 *   beta == 0: C is not read before it is written, so NaN or garbage in C does not
 *   propagate.
 *   NaN and Inf in A or B propagate by IEEE rules.
 *
 * Arithmetic
 *   FP32 fused multiply-add on the CUDA cores (round to nearest even), FP32 accumulation.
 *   The order of the k-sum differs from a sequential loop (per-thread k-sequential inside a
 *   tile; split-K partial sums added in a fixed slice order). Results are deterministic:
 *   the same call on the same device gives bitwise the same C.
 *
 * Return value (BLAS xerbla style: the first illegal argument, counted from 1)
 *    0   success
 *   -1   M < 0          -2   N < 0          -3   K < 0
 *   -5   A == NULL while A must be read
 *   -6   lda < max(1, K)
 *   -7   B == NULL while B must be read
 *   -8   ldb < max(1, N)
 *   -10  C == NULL while M > 0 and N > 0
 *   -11  ldc < max(1, N)
 *   -13  (sgemm_f32_ws only) workspace too small or NULL while one is needed
 *   -15  (sgemm_f32_noalloc only) the problem needs more split-K scratch than the
 *        library's fixed array holds
 *   >0   a cudaError_t from a launch or a stream-ordered allocation
 *   Nothing is launched when an argument is illegal. The library never aborts or traps.
 */
#ifndef SGEMM_F32_H_
#define SGEMM_F32_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Forward declaration compatible with cuda_runtime_api.h. */
typedef struct CUstream_st *cudaStream_t;

/* C = alpha * A * B + beta * C (row-major, FP32 FFMA path). See the file comment. */
int sgemm_f32(int M, int N, int K, float alpha, const float *A, int lda, const float *B,
              int ldb, float beta, float *C, int ldc, cudaStream_t stream);

/* C = alpha * op(A) * op(B) + beta * C, row-major, with BLAS transpose flags ("Lecture 4 -
 * GPU Acceleration", section 5.2: op(X) is X or X^T). transa / transb: 0 = as stored,
 * 1 = transposed. C is M x N (ldc >= max(1, N)); op(A) is M x K and op(B) is K x N:
 *   transa = 0: A stored M x K, lda >= max(1, K);  transa = 1: A stored K x M, lda >= max(1, M)
 *   transb = 0: B stored K x N, ldb >= max(1, N);  transb = 1: B stored N x K, ldb >= max(1, K)
 * (all row-major). Same memory, asynchrony and special cases as sgemm_f32. Returns 0, or
 * -i for the first illegal argument in this signature's order (transa = 1, transb = 2,
 * M = 3, ..., ldc = 13), or a cudaError_t. */
int sgemm_f32_ex(int transa, int transb, int M, int N, int K, float alpha, const float *A,
                 int lda, const float *B, int ldb, float beta, float *C, int ldc,
                 cudaStream_t stream);

/* Column-major interface with the BLAS sgemm argument list (as cuBLAS takes it, with the
 * scalars by value): C (m x n, ldc >= max(1, m)) = alpha * op(A) * op(B) + beta * C, where
 * A is m x k (transa = 0, lda >= max(1, m)) or k x m (transa = 1, lda >= max(1, k)) and B
 * is k x n (transb = 0, ldb >= max(1, k)) or n x k (transb = 1, ldb >= max(1, n)), all
 * column-major. Computed as the row-major product C^T = op(B)^T op(A)^T (the swap trick
 * of the same lecture, section 5.4). Returns 0, -i for the first illegal argument in this
 * signature's order, or a cudaError_t. */
int sgemm_f32_colmajor(int transa, int transb, int m, int n, int k, float alpha,
                       const float *A, int lda, const float *B, int ldb, float beta, float *C,
                       int ldc, cudaStream_t stream);

/* y = alpha * op(A) * x + beta * y, the matrix-vector sibling of sgemm named with it in
 * "Lecture 4 - GPU Acceleration", section 5.2 (cublasSgemv), for a row-major A (M x N,
 * lda >= max(1, N)). trans = 0: y has M elements and x has N; trans = 1: op(A) = A^T, y has
 * N elements and x has M. incx, incy: nonzero element strides (negative strides walk the
 * vector backwards, as in BLAS). FP32 FMA accumulation in a fixed order (deterministic).
 * alpha == 0 or an empty x: y = beta * y (y = 0 when beta == 0; x and A not read). Device
 * pointers, asynchronous on `stream`; the transposed case takes a small workspace from the
 * library's pool. Returns 0, -i for the first illegal argument (trans = 1, ..., incy = 11),
 * or a cudaError_t. */
int sgemv_f32(int trans, int M, int N, float alpha, const float *A, int lda, const float *x,
              int incx, float beta, float *y, int incy, cudaStream_t stream);

/* *result = sum_i x_i * y_i (cublasSdot, same lecture section), n elements with nonzero
 * strides incx, incy; `result` is a device pointer written on `stream` (0 for n == 0). FP32
 * FMA partial sums per block, added in a fixed order in a second launch (deterministic).
 * Returns 0, -i for the first illegal argument (n = 1, ..., result = 6), or a
 * cudaError_t. */
int sdot_f32(int n, const float *x, int incx, const float *y, int incy, float *result,
             cudaStream_t stream);

/* Bytes of workspace that sgemm_f32 would allocate for this problem on the current device
 * (0 when the chosen plan needs none): the pre-pass copies (A^T for the k-major plans,
 * aligned operand copies) and the split-K partial tiles, for beta != 0 (a beta = 0 call
 * may plan differently: sgemm_f32_plan reports its plan). Pointers are assumed 16-byte
 * aligned. Host-side query (the first call sets up the device). Returns the same negative
 * codes as sgemm_f32 for illegal shapes or leading dimensions, else 0 or a cudaError_t. */
int sgemm_f32_workspace_size(int M, int N, int K, int lda, int ldb, int ldc,
                             size_t *bytes);

/* The smallest workspace with which sgemm_f32_ws runs this problem: the same plan without
 * its A^T copy, i.e. only the split-K partial tiles (and aligned copies of operands that
 * TMA cannot address). Given a workspace of at least this size but smaller than
 * sgemm_f32_workspace_size, sgemm_f32_ws runs the twin configuration, which transposes A
 * in shared memory: the same tiles, K slices and k order, so the result is bitwise the
 * same, with one launch fewer and no A^T copy. (At 8192^3 on GB300: 21 MiB instead of
 * 290 MB, at 70.7 against 74.7 TFLOP/s.) Equal to sgemm_f32_workspace_size for plans
 * without an A^T copy. Same conventions and return codes as sgemm_f32_workspace_size. */
int sgemm_f32_workspace_size_min(int M, int N, int K, int lda, int ldb, int ldc,
                                 size_t *bytes);

/* Same as sgemm_f32, but any split-K workspace comes from the caller: `workspace` is a
 * device buffer of `workspace_bytes` bytes, 16-byte aligned, not read before it is written
 * and not used after the call's kernels finish. The call allocates nothing. */
int sgemm_f32_ws(int M, int N, int K, float alpha, const float *A, int lda, const float *B,
                 int ldb, float beta, float *C, int ldc, void *workspace,
                 size_t workspace_bytes, cudaStream_t stream);

/* Launch plan chosen for a problem, for tests and tuning. Host-only: no CUDA call is made
 * when num_sms > 0 (the SM count to plan for); num_sms == 0 asks the current device.
 * A and B are assumed 16-byte aligned (they decide whether the TMA-fed kernel applies).
 * alpha and beta matter only through their special values (alpha == 0, beta == 0, 1).
 * Outputs (any may be NULL):
 *   variant  tile configuration index (0 .. sgemm_f32_num_variants() - 1), -1 when no
 *            GEMM kernel runs (empty problem or beta-scale only)
 *   split      K slices of each split tile (1 = no split-K)
 *   main_tiles tiles computed whole; the remaining tiles are split into `split` K slices.
 *              These are finished by a second, reducing kernel from the workspace. When
 *              every tile is split (main_tiles == 0) into at most 8 slices and the slices
 *              fit as thread-block clusters, they are instead added inside the cluster
 *              through distributed shared memory (no second kernel, no workspace)
 *   launches   kernels enqueued by one sgemm_f32 call (pre-pass copies included)
 *   ws_bytes   workspace bytes: pre-pass copies (A^T for the k-major configurations,
 *              aligned copies of operands TMA cannot address) and split-K partial tiles
 * Returns the same negative codes as sgemm_f32 for illegal arguments, else 0. */
int sgemm_f32_plan(int M, int N, int K, int lda, int ldb, int ldc, float alpha, float beta,
                   int num_sms, int *variant, int *split, int *main_tiles, int *launches,
                   size_t *ws_bytes);

/* Tile configurations compiled into the library, for tests and tuning. */
int sgemm_f32_num_variants(void);

/* The cluster capacity the planner uses for configuration `variant` on the current device:
 * *ctas = how many of its CTAs the device holds at once in thread-block clusters of
 * `cluster` CTAs (the driver's cudaOccupancyMaxActiveClusters times the cluster size;
 * clusters sit inside one GPC, so this can be below SMs x CTAs per SM). A split of every
 * tile into `cluster` K slices is finished inside the cluster only when these CTAs fit in
 * as few waves as unclustered ones. Configurations whose shared memory cannot hold a
 * partial tile, and cluster sizes below 2, give 0; the cluster thin kernels (43, 44) give
 * their capacity for clusters of 1, 2, 4 and 8 (0 for other sizes).
 * Returns 0, -1 (variant out of range), -2 (cluster not in 1 .. 8), -3 (ctas NULL), or a
 * cudaError_t of the device set-up. */
int sgemm_f32_cluster_capacity(int variant, int cluster, int *ctas);

/* Describe variant v: CTA tile BM x BN x BK, threads per CTA, per-thread TM x TN
 * accumulator tile, pipeline stages. Returns 0; 1 for a configuration that keeps its index
 * in the table but is not compiled into this build (the outputs are still filled; forcing
 * it returns -14); or -1 if v is out of range. */
int sgemm_f32_variant_info(int v, int *BM, int *BN, int *BK, int *threads, int *TM,
                           int *TN, int *stages);

/* sgemm_f32 with the plan forced, for tests and tuning sweeps; results satisfy the same
 * contract as sgemm_f32. `variant` in [0, sgemm_f32_num_variants()) pins the tile
 * configuration (-1: automatic). `split` >= 1 splits every tile into that many K slices
 * (1: no split-K; 2 .. 8 run as thread-block clusters where the configuration and the
 * device's cluster occupancy allow, see sgemm_f32_plan); -1 computes the full waves of
 * tiles whole and splits only the tiles of the last, partial wave (slice count chosen to
 * fill it); <= -2 does the same with -split slices; 0 is automatic. Slice counts are
 * clamped so that every slice holds at least one K tile. The cluster thin kernels take
 * `split` as their cluster size, rounded up to 1, 2, 4 or 8. A TMA-fed configuration on
 * an operand TMA cannot address (lda or ldb not a multiple of 4, or a pointer not 16-byte
 * aligned) first copies it to aligned rows in the workspace; for the cluster thin kernels
 * that copy is made of the small operand only (thin-M: A, thin-N: B). Returns -14 for an
 * out-of-range variant, for a configuration that cannot run the problem (a TMA-fed one on
 * transposed operands, see sgemm_f32_ex_forced; a TMA-fed thin one whose streamed operand
 * TMA cannot address), and for the K-paired configurations when A is not 16-byte aligned
 * with lda a multiple of 4. */
int sgemm_f32_forced(int M, int N, int K, float alpha, const float *A, int lda,
                     const float *B, int ldb, float beta, float *C, int ldc, int variant,
                     int split, cudaStream_t stream);

/* Benchmarking switch: when the environment variable SGEMM_F32_FORCE is "v" or "v:s" at the
 * first call in the process, every automatic plan (sgemm_f32, sgemm_f32_ex, sgemm_f32_ws,
 * sgemm_f32_noalloc, sgemm_f32_host, sgemm_f32_plan) is the one sgemm_f32_forced would make
 * with variant v and split s, for the problems that configuration can run; the others keep
 * their automatic plan. It takes precedence over plans recorded by sgemm_f32_autotune. */

/* sgemm_f32_ex with the plan forced (variant and split as in sgemm_f32_forced). Returns
 * -14 also when the forced configuration has no path for these transpose flags or this
 * alignment:
 *   - the TMA-fed configurations need transb = 0, and transa = 0, except the k-major ones
 *     (35, 36, 39, 40), which also take transa = 1 with A_st 16-byte aligned and lda a
 *     multiple of 4 (A_st is then read directly);
 *   - the K-paired ones need transa = 0 and A 16-byte aligned with lda a multiple of 4;
 *   - the copy-fed ones carry transposed-operand paths only in configurations 2, 3, 4, 16. */
int sgemm_f32_ex_forced(int transa, int transb, int M, int N, int K, float alpha,
                        const float *A, int lda, const float *B, int ldb, float beta, float *C,
                        int ldc, int variant, int split, cudaStream_t stream);

/* Size of the fixed device scratch array used by sgemm_f32_noalloc, and its error code. */
#define SGEMM_F32_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20) /* 32 MiB per device */
#define SGEMM_F32_ERR_SCRATCH_TOO_SMALL (-15)

/* C = alpha * A * B + beta * C exactly like sgemm_f32 (same plan, same kernels, bitwise the
 * same result), for callers that are not allowed to allocate device memory. The source
 * pages have no counterpart of this entry point; it exists for how the library is used.
 *
 * Who needs it: code running inside a host framework that owns all device memory and does
 * not let libraries allocate (for example a plugin of an inference runtime whose memory is
 * planned up front), and real-time or certified loops that forbid allocation after start-up.
 * For them cudaMalloc and cudaMallocAsync are off limits: an allocation can block or
 * synchronise, can fail under memory pressure at any point, and bypasses the caller's own
 * accounting of device memory.
 *
 * How: the split-K workspace that sgemm_f32 takes from cudaMallocAsync comes instead from a
 * fixed array of SGEMM_F32_NOALLOC_SCRATCH_BYTES in device global memory owned by the
 * library; every GPU that loads the library holds that array until the process exits. The
 * call makes no cudaMalloc, cudaMallocAsync, cudaFree or other allocating call. The caller
 * still passes A, B and C, as for sgemm_f32.
 *
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current. Make that first call on a device before
 * any stream capture on it; a lookup that fails is returned as its cudaError_t and tried
 * again by the next call. Like any first library call on a device, the first call also
 * creates the library's per-device memory pool, empty; this entry point takes nothing from
 * it.
 *
 * Sharing: all calls in the process share the one array of a device, which keeps whatever
 * the last call left in it. Calls ordered on the GPU (the same stream, or streams ordered by
 * events) are safe. Calls that can overlap on the GPU (unordered streams, for example from
 * several host threads) race on the array and give wrong results. Nothing in the array has
 * to start at zero: a call writes every workspace element before it reads it.
 *
 * Workspace: when the plan reads a transposed copy of A (the k-major TMA-fed
 * configurations) and that copy does not fit, the call runs the twin configuration that
 * transposes A in shared memory instead. The tiles, slices and k order are the same, so
 * the result is still bitwise sgemm_f32's. sgemm_f32_ws does the same with a caller
 * workspace that is too small for the copy.
 *
 * Errors: as sgemm_f32, plus SGEMM_F32_ERR_SCRATCH_TOO_SMALL when the rest of the plan's
 * workspace does not fit the array (sgemm_f32_workspace_size() reports the full need
 * beforehand): split-K partial tiles, plus, when lda or ldb is not a multiple of 4 or A or
 * B is not 16-byte aligned, the aligned copies of those operands that the plan makes
 * (large unaligned problems therefore exceed it). Nothing is launched in that case. */
int sgemm_f32_noalloc(int M, int N, int K, float alpha, const float *A, int lda,
                      const float *B, int ldb, float beta, float *C, int ldc,
                      cudaStream_t stream);

/* C = alpha * A * B + beta * C on the tensor cores (tcgen05, kind::tf32) with the 3xTF32
 * split: every FP32 input x is split into x_hi = tf32(x) and x_lo = tf32(x - x_hi) and
 * A * B is accumulated in FP32 as A_hi B_hi + A_hi B_lo + A_lo B_hi. The dropped terms are
 * about 2^-21 of each |a b|, so the result meets the same FP32 error bound as sgemm_f32
 * (1e-4 * sum_k |a_ik b_kj| + |beta c_ij| elementwise) while running on the tensor cores.
 * Same arguments, layout, special cases and return codes as sgemm_f32. The split operands
 * live in a workspace of sgemm_f32_3xtf32_workspace_size() bytes that the call takes from
 * the library's stream-ordered pool and frees on `stream`. Reported separately from the
 * FFMA path. NaN and Inf inputs are not handled like sgemm_f32 (x - x_hi is NaN for an
 * infinite x). */
int sgemm_f32_3xtf32(int M, int N, int K, float alpha, const float *A, int lda,
                     const float *B, int ldb, float beta, float *C, int ldc,
                     cudaStream_t stream);

/* Workspace bytes sgemm_f32_3xtf32 uses for an M x N x K problem (host-only query;
 * negative codes as sgemm_f32 for negative sizes). */
int sgemm_f32_3xtf32_workspace_size(int M, int N, int K, size_t *bytes);

/* Reads and clears the tensor-core path's device status word (synchronising copy on the
 * legacy stream): 0 = fine; 1, 2, 3 = a bounded wait of the producer, MMA or epilogue
 * threads gave up (the kernel then skipped work and the result is not valid). */
int sgemm_f32_3xtf32_status(int *status);

/* Returns to the system the device memory that the library's pool on the current device
 * keeps for reuse: workspaces freed by earlier calls of every entry point (sgemm_f32 and
 * its variants, the host-buffer, 3xTF32, SGEMV / SDOT and autotune calls). Memory that a
 * call still uses is kept, and so is memory whose stream-ordered free has not yet run on
 * the GPU: synchronise the streams that ran library calls first to release everything.
 * Later calls allocate again as needed. *released_bytes (may be NULL) = bytes returned.
 * The first library call on a device creates its (empty) pool, so a first call here does.
 * Returns 0 or a cudaError_t. */
int sgemm_f32_release_workspace(size_t *released_bytes);

/* Reads and clears the device status word of the TMA-fed FFMA kernel (synchronising copy
 * on the legacy stream): 0 = fine; 1 or 2 = a bounded mbarrier wait gave up (a consumer
 * waiting for data, or the producer waiting for a free stage), in which case the kernel
 * stopped computing and the result of that call is not valid. Every mbarrier wait in the
 * library's kernels gives up after about one second of the GPU's global timer. */
int sgemm_f32_status(int *status);

/* Failure-path self-test of that bounded wait: one warp waits, with the kernels' own wait,
 * for a phase of an mbarrier that nothing ever completes. The wait must give up after
 * about one second and the kernel must end normally. Outputs: *timed_out = 1 if the wait
 * gave up (0 would mean it saw a phase complete), *seconds = the kernel's duration (CUDA
 * events). Synchronous (own stream); the context stays usable afterwards. Returns 0 or a
 * cudaError_t. */
int sgemm_f32_wait_selftest(int *timed_out, float *seconds);

/* FP32 pipe probe: the measured counterpart of the derived FP32 peak (SMs x 128 FP32 lanes
 * x 2 FLOP x SM clock) that the GEMM kernels are held against. One kernel of SMs x 8 CTAs
 * of 256 threads; each thread advances 8 independent register pairs `iters` times by
 * packed FP32 multiply-adds (fma.rn.f32x2, the GEMM inner loop's instruction) whose
 * multiplicands are pairs holding one value twice, with no memory traffic but one store
 * that never happens. (With two different values in each multiplicand pair the pipe
 * sustains about 12% less on GB300.) It runs once untimed, then `reps` times, each timed
 * with CUDA events; synchronous, on a stream of its own.
 *   iters          iterations per thread, 1 .. 2^24 (2^17 takes about 16 ms on GB300)
 *   reps           timed launches, 1 .. 100
 *   tflops         out: 4 x 8 x iters x threads FLOP / the median launch time, in TFLOP/s
 *   ms_per_launch  out (may be NULL): that median time
 * Returns 0, -1 (iters), -2 (reps), -3 (tflops NULL), or a cudaError_t. */
int sgemm_f32_fma_probe(int iters, int reps, double *tflops, float *ms_per_launch);

/* C = alpha * A * B + beta * C with A, B and C in HOST memory (row-major, the ld rules of
 * sgemm_f32). The product runs on the GPU in row blocks of about 2048 rows: B is copied to
 * the device once, and the copies of a block's A and C rows in and of its C rows out run on
 * two library-owned copy streams that overlap the GEMMs of the neighbouring blocks, which
 * run on `stream`. With two or more blocks, K >= 1024 and B of 32 MB or more, the first
 * block is computed in K chunks (256, then each twice the one before) as B and its A rows
 * arrive: each chunk's alpha * A B is added into the block, and beta * C (copied in behind
 * the chunks) is added last, so the GEMMs start after the first small chunk. That block's
 * result is rounded to FP32 once per chunk and is not bitwise the single-call result (it
 * meets the same error bound). With two or more blocks, the last block, if 1024 rows or
 * more, is computed in two calls, its last 3/8 (rounded up to 128 rows) apart, and the
 * first part's rows go back while the second part computes. Device buffers come from the
 * library's workspace pool (B, two A-block and C-block buffers, and for that head with
 * beta != 0 one more C-block buffer) and are released in stream order.
 * Host memory should be page-locked (cudaHostAlloc / cudaHostRegister) for the copies to
 * overlap; pageable memory works, with copies that do not overlap.
 * Asynchronous on `stream`: C on the host is final once `stream` has been synchronised;
 * A, B and C must stay valid until then. Returns the sgemm_f32 codes. */
int sgemm_f32_host(int M, int N, int K, float alpha, const float *A, int lda, const float *B,
                   int ldb, float beta, float *C, int ldc, cudaStream_t stream);

/* ---- Measured plan selection ("GPU GEMM 优化完全拆解（二）", autotuning section: sweep the
 * legal tile parameters and keep the fastest set, which differs from GPU to GPU). ----
 *
 * sgemm_f32_autotune times, on `stream` and the caller's operands, every compiled tile
 * configuration that can run op(A) op(B) for these transpose flags, shape, leading
 * dimensions and alignments. Each is timed with several split-K layouts: the model's own
 * choice, no split, every tile split 2, 3, 4, 6 or 8 ways, and whole waves plus a last
 * wave split the automatic number of ways or 2, 3, 4, 6 or 8 (the thin kernels: the
 * model's choice, no split, a split last wave and, for the cluster thin kernels, clusters
 * of 2, 4 and 8). Layouts that come out the same are timed once. Each candidate runs once to
 * warm up, then `reps` times (3 if reps <= 0), timed with CUDA events. Layouts the cost
 * model rates at more than 4x its best are skipped. The fastest candidate is recorded in
 * a per-process table. From then on sgemm_f32, sgemm_f32_ex, sgemm_f32_ws,
 * sgemm_f32_noalloc and sgemm_f32_plan use it instead of the model for the same shape,
 * transpose flags, alignment class (TMA-able or not), beta != 0 and SM count.
 * Arguments are those of sgemm_f32_ex. C is only read: the timed calls write a scratch
 * copy taken from the library's workspace pool. The call synchronises `stream`.
 * Outputs (any may be NULL): the chosen variant (as in sgemm_f32_forced), the split
 * argument that reproduces its layout, and its mean time in ms. An empty problem,
 * alpha == 0 or K == 0 records nothing and returns 0 with *variant = -1.
 * Returns 0, the sgemm_f32_ex codes for illegal arguments, or a cudaError_t. A recorded
 * plan may need more workspace than the model's choice. sgemm_f32_ws and
 * sgemm_f32_noalloc then return -13 / -15 for that shape, as they do for any plan that
 * does not fit. */
int sgemm_f32_autotune(int transa, int transb, int M, int N, int K, float alpha,
                       const float *A, int lda, const float *B, int ldb, float beta,
                       const float *C, int ldc, int reps, cudaStream_t stream, int *variant,
                       int *split, float *ms);

/* Number of recorded plans; forget them all (returns 0). */
int sgemm_f32_tune_count(void);
int sgemm_f32_tune_clear(void);

/* Write the recorded plans to a text file: two comment lines, then one line per plan,
 * "sms M N K flags variant split ms". Returns the number of plans written, -1 for a NULL
 * path, -2 if the file cannot be written. */
int sgemm_f32_tune_save(const char *path);

/* Add the plans of a file written by sgemm_f32_tune_save (a plan for the same key
 * replaces the recorded one). Lines whose fields are out of range are skipped. Returns
 * the number of plans loaded, -1 for a NULL path, -2 if the file cannot be read, or -3 if
 * any line was skipped (the valid ones are still loaded). */
int sgemm_f32_tune_load(const char *path);

/* Library version string, e.g. "sgemm_f32 0.1.0 sm_103a". */
const char *sgemm_f32_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SGEMM_F32_H_ */
