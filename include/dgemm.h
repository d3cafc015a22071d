/*
 * dgemm.h -- C ABI of the GB300 (sm_103a) dense GEMM library.
 *
 * Every entry point computes the plain row-major matrix product
 *
 *     C[i*ldc + j] = sum_{k=0}^{K-1} A[i*lda + k] * B[k*ldb + j],  0 <= i < M, 0 <= j < N
 *
 * as defined in "第八课：GPU 如何完成矩阵乘法" (Lesson 8: how a GPU does matrix
 * multiplication), section 一 (C = A x B with A in R^{M x K}, B in R^{K x N},
 * C_{i,j} = sum_k A_{i,k} B_{k,j}); the same formula opens "SGEMM 优化旅程",
 * Level 1, and section 4.1 of "4. 矩阵乘法（GEMM）优化".  The pages use the
 * compact row-major addressing A[row*K + k], B[k*N + col], C[row*N + col]
 * (Lesson 8 section 四, section 二十八); these entry points take BLAS-style
 * leading dimensions lda >= K, ldb >= N, ldc >= N, counted in elements.
 *
 * Semantics shared by all entry points
 *   - C is OVERWRITTEN inside its M x N region (no alpha/beta: the pages store
 *     the finished sum, C[row*N + col] = sum).  Elements of C outside that
 *     region (the ldc - N gap at the end of each row) are never written.
 *   - K == 0: the empty sum; the M x N region of C is set to zero.
 *   - M == 0 or N == 0: nothing to do; DGEMM_OK with no launch (the pointers
 *     are not looked at).
 *   - Sizes are int, as in the pages' kernel signatures; all offsets are
 *     computed in 64-bit.
 *
 * Pointers and ownership
 *   - A, B and C are DEVICE pointers (cudaMalloc'd or managed memory) on the
 *     current CUDA device, owned by the caller.  Host pointers are rejected
 *     with DGEMM_ERR_INVALID_POINTER before anything is launched.
 *   - Only natural element alignment is required (4 bytes for fp32, 2 for
 *     bf16).  Any pointer or leading dimension, aligned to 16 bytes or not, is
 *     accepted; the library chooses the load path itself.
 *   - C must not overlap the bytes A or B span: DGEMM_ERR_ALIAS.
 *
 * Execution
 *   - Asynchronous on `stream` (0 = the legacy default stream): the call
 *     validates, enqueues and returns.  Work on the same stream is ordered.
 *   - A launch failure, or a sticky error left by earlier work, is returned as
 *     DGEMM_ERR_CUDA; dgemm_last_cuda_error() gives the CUDA message.
 *   - Deterministic: the same inputs give bitwise identical C on every call
 *     (no floating-point atomics; K-split partial tiles are added in a fixed
 *     order).
 *   - Thread-safe and re-entrant; the only mutable library state is a
 *     per-thread error string and a per-device watchdog word (see
 *     dgemm_watchdog_status).
 *   - Some paths use temporary device memory (re-pitched operands, the FP32
 *     SIMT path's K-split partials, the lo parts of 3xTF32 operands, 8-bit
 *     transposes): stream-ordered allocations on `stream`, freed on `stream`
 *     at the end of the call, from a memory pool the library creates per
 *     device.  Back-to-back calls reuse the pool's memory; at the next
 *     stream, event or device synchronisation the pool returns what it holds
 *     beyond 32 MiB to the system, so no more than 32 MiB stays reserved
 *     between calls.  DGEMM_POOL_KEEP_BYTES (read once, when the pool is
 *     created) sets another bound, e.g. 0 to keep nothing.
 */
#ifndef DGEMM_H
#define DGEMM_H

#include <cuda_runtime_api.h>   /* cudaStream_t */

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  Every entry point returns one; only DGEMM_OK means the work
 * was enqueued. */
typedef enum {
    DGEMM_OK = 0,
    DGEMM_ERR_INVALID_VALUE = 1,   /* negative size, leading dimension too small */
    DGEMM_ERR_NULL_POINTER = 2,    /* NULL A, B or C with work to do            */
    DGEMM_ERR_ALIAS = 3,           /* C overlaps A or B                          */
    DGEMM_ERR_UNSUPPORTED = 4,     /* unknown mode                               */
    DGEMM_ERR_CUDA = 5,            /* CUDA runtime/driver error (see below)      */
    DGEMM_ERR_ARCH = 6,            /* current device is not compute capability 10.3 */
    DGEMM_ERR_MISALIGNED = 7,      /* pointer not aligned to its element size    */
    DGEMM_ERR_INVALID_POINTER = 8, /* A, B or C is not device-accessible memory  */
    DGEMM_ERR_WATCHDOG = 9,        /* a kernel gave up a bounded wait (see dgemm_watchdog_status) */
    DGEMM_ERR_SCRATCH_LIMIT = 10   /* gemm_f32_tc_noalloc: operands need more than its fixed scratch */
} dgemm_status_t;

/* Operand operations of dgemm_gemm_ex: op(X) = X or its transpose. */
typedef enum {
    DGEMM_OP_N = 0,  /* as stored */
    DGEMM_OP_T = 1   /* transposed */
} dgemm_op_t;

/* Arithmetic paths of dgemm_gemm_ex (element type of A and B in brackets). */
typedef enum {
    DGEMM_PATH_SIMT = 0,    /* FP32 FFMA on the CUDA cores       [fp32] */
    DGEMM_PATH_TF32 = 1,    /* tcgen05, TF32 operands            [fp32] */
    DGEMM_PATH_3XTF32 = 2,  /* tcgen05, split-precision 3xTF32   [fp32] */
    DGEMM_PATH_BF16 = 3,    /* tcgen05, BF16 operands            [bf16] */
    DGEMM_PATH_FP16 = 4,    /* tcgen05, FP16 operands            [fp16] */
    DGEMM_PATH_F8_E4M3 = 5, /* tcgen05, FP8 E4M3 operands        [fp8]  */
    DGEMM_PATH_F8_E5M2 = 6  /* tcgen05, FP8 E5M2 operands        [fp8]  */
} dgemm_path_t;

/* 8-bit float formats of gemm_f8_tc. */
typedef enum {
    DGEMM_F8_E4M3 = 0,  /* 1 sign, 4 exponent (bias 7), 3 mantissa bits; no infinities, max 448 */
    DGEMM_F8_E5M2 = 1   /* 1 sign, 5 exponent (bias 15), 2 mantissa bits; IEEE-style, max 57344 */
} dgemm_f8_format_t;

/* Tensor-core precision modes of gemm_f32_tc. */
typedef enum {
    DGEMM_TC_TF32 = 0,   /* operands read at TF32 precision (10-bit mantissa), FP32 accumulate */
    DGEMM_TC_3XTF32 = 1  /* split precision: a = a_hi + a_lo, three TF32 products, FP32-grade result */
} dgemm_tc_mode_t;

/*
 * gemm_f32_simt -- FP32 inputs, FP32 fused multiply-add on the CUDA cores.
 *
 * The register-blocked, shared-memory tiled form of the product: "SGEMM 优化旅程"
 * Levels 2-5 (shared-memory tiles, padding against bank conflicts, double
 * buffering, 8x8 register blocking per thread of a 128x128x8 block tile) and
 * Lesson 8 sections 九-十九 (tile decomposition C_tile = sum_t A_tile,t B_tile,t,
 * register accumulation, multi-level tiling, boundary zero-fill and masked
 * stores of section 二十六).
 * A: M x K fp32, row-major, leading dimension lda >= max(1, K).
 * B: K x N fp32, row-major, leading dimension ldb >= max(1, N).
 * C: M x N fp32, row-major, leading dimension ldc >= max(1, N); overwritten.
 * Accuracy: |C - C_exact| <= 1e-5 * (|A| x |B|) elementwise; exact when every
 * product and partial sum is an integer below 2^24.
 */
int gemm_f32_simt(int M, int N, int K,
                  const float *A, int lda,
                  const float *B, int ldb,
                  float *C, int ldc,
                  cudaStream_t stream);

/*
 * gemm_f32_tc -- FP32 inputs on the 5th-generation tensor cores (tcgen05).
 *
 * The tensor-core form of the product: "SGEMM 优化旅程" Level 6 and Lesson 8
 * sections 二十一-二十三 (the tensor core computes a small D = A x B + C per
 * instruction, and must be fed tiles through shared memory).  Operands are
 * staged by TMA into swizzled shared memory, accumulated in tensor memory.
 * mode = DGEMM_TC_TF32:   each operand is read at TF32 precision; accuracy
 *                         |C - C_exact| <= 2e-3 * (|A| x |B|).
 * mode = DGEMM_TC_3XTF32: each operand is split a ~ hi + lo (hi = a with the
 *                         low 13 mantissa bits cleared, lo = a - hi rounded
 *                         to TF32) and C = A_hi B_hi + A_hi B_lo + A_lo B_hi;
 *                         accuracy <= 1e-5 * (|A| x |B|).  Infinities and
 *                         NaNs propagate as in IEEE arithmetic, except that
 *                         an infinite entry meeting a finite one whose lo is
 *                         exactly 0 adds inf * 0 = NaN to that entry of C.
 *                         Large problems (those the CTA-pair kernel takes)
 *                         first write lo(A) and lo(B) to scratch the size of
 *                         A and B, one extra kernel; if that scratch cannot
 *                         be allocated, the single-CTA kernel splits the
 *                         staged tiles in shared memory instead (same result,
 *                         slower).
 * Argument layout as gemm_f32_simt.  Unknown mode: DGEMM_ERR_UNSUPPORTED.
 */
int gemm_f32_tc(int mode, int M, int N, int K,
                const float *A, int lda,
                const float *B, int ldb,
                float *C, int ldc,
                cudaStream_t stream);

/*
 * gemm_bf16_tc -- BF16 inputs, FP32 accumulate, FP32 output, on tcgen05.
 *
 * Lesson 8 section 二十二 lists BF16 among the tensor-core input types; this is
 * the BF16-in / FP32-accumulate form of gemm_f32_tc.
 * A: M x K bfloat16 (raw 16-bit patterns), row-major, lda >= max(1, K).
 * B: K x N bfloat16, row-major, ldb >= max(1, N).
 * C: M x N fp32, row-major, ldc >= max(1, N); overwritten.
 * Accuracy: |C - C_exact| <= 8e-3 * (|A| x |B|), C_exact the exact product of
 * the bf16 values.
 */
int gemm_bf16_tc(int M, int N, int K,
                 const unsigned short *A, int lda,
                 const unsigned short *B, int ldb,
                 float *C, int ldc,
                 cudaStream_t stream);

/*
 * gemm_f32_tc_noalloc -- gemm_f32_tc for callers that cannot allocate.
 *
 * The pages have no counterpart of this entry point; it exists for callers
 * that must not allocate device memory during the call: code that runs with
 * every byte of device memory reserved up front (a serving process that has
 * partitioned HBM among its models, where a new allocation can fail), code
 * called from inside an allocator or memory-manager callback (which must not
 * re-enter the allocator), and latency-critical loops that must not risk an
 * allocation failing or growing a memory pool in the middle of a run.
 *
 * Same arguments, semantics, accuracy and status codes as gemm_f32_tc.  The
 * difference is where the re-pitch scratch lives: gemm_f32_tc takes it from
 * the library's stream-ordered memory pool when A or B rows do not start on
 * 16-byte boundaries; this
 * entry point uses instead a fixed 16 MiB array (DGEMM_NOALLOC_SCRATCH_BYTES)
 * that the library holds in device memory on every GPU that loads it, until
 * the process exits.  It calls no cudaMalloc, cudaFree or other allocating
 * routine.
 *   - Limit: the re-pitched copies of A and/or B (rows rounded up to 16 bytes,
 *     each copy rounded up to 256 bytes) must fit in 16 MiB; otherwise the
 *     call returns DGEMM_ERR_SCRATCH_LIMIT and launches nothing.  Operands
 *     that need no re-pitch use no scratch, at any size.
 *   - 3xTF32 writes the lo parts of A and B into the rest of the array when
 *     they fit there; larger problems run on the single-CTA kernel, which
 *     needs no scratch for the split.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current.  Under CUDA's lazy
 *     module loading (the default) that lookup is also what loads the array
 *     into device memory, so the first call on each device must come before
 *     the caller reserves all device memory, and before any stream capture
 *     begins on the device.  The address is kept for the life of the process:
 *     do not use the library across cudaDeviceReset.
 *   - Results are bitwise those of gemm_f32_tc in TF32 mode, and in 3xTF32
 *     mode whenever the lo parts fit in the array (or the problem is small
 *     enough for the single-CTA kernel anyway); larger 3xTF32 problems run
 *     on a different kernel and agree with gemm_f32_tc only within the
 *     3xTF32 tolerance.
 *   - Every call on a device shares the one array, and it keeps the last
 *     call's contents.  Each call overwrites all the scratch it reads before
 *     reading it, so nothing needs clearing; but two calls whose work
 *     overlaps on the GPU (different streams, no ordering between them) race
 *     on the array and may corrupt each other's results.  Order such calls
 *     on one stream or with events.
 */
int gemm_f32_tc_noalloc(int mode, int M, int N, int K,
                        const float *A, int lda,
                        const float *B, int ldb,
                        float *C, int ldc,
                        cudaStream_t stream);

/* Size in bytes of the fixed scratch array gemm_f32_tc_noalloc uses. */
#define DGEMM_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * gemm_f16_tc -- FP16 inputs, FP32 accumulate, FP32 output, on tcgen05.
 *
 * The tensor-core input type of "SGEMM 优化旅程" Level 6 (half operands with
 * a float accumulator, there through WMMA fragments) and the first entry of
 * Lesson 8 section 二十二's list of tensor-core formats; the same kernels as
 * gemm_bf16_tc with IEEE binary16 operands.
 * A: M x K float16 (raw 16-bit patterns), row-major, lda >= max(1, K).
 * B: K x N float16, row-major, ldb >= max(1, N).
 * C: M x N fp32, row-major, ldc >= max(1, N); overwritten.
 * The fp16 inputs are exact, so only the FP32 accumulation rounds: at most
 * K/16 rounded additions of the accumulator, |C - C_exact| <= 2e-4 *
 * (|A| x |B|) for K <= 16384.
 */
int gemm_f16_tc(int M, int N, int K,
                const unsigned short *A, int lda,
                const unsigned short *B, int ldb,
                float *C, int ldc,
                cudaStream_t stream);

/*
 * gemm_f8_tc -- FP8 inputs (E4M3 or E5M2), FP32 accumulate, FP32 output, on
 * tcgen05 (kind::f8f6f4).
 *
 * Lesson 8 section 二十二 lists FP8 among the tensor cores' input formats;
 * the pages give it no scaling convention, so the 8-bit values are the
 * operands as given (scale 1; a caller with scaled data multiplies C by the
 * product of its scales).  `format` (dgemm_f8_format_t) applies to A and B.
 * A: M x K bytes, row-major, lda >= max(1, K).
 * B: K x N bytes, row-major, ldb >= max(1, N).
 * C: M x N fp32, row-major, ldc >= max(1, N); overwritten.
 * The tensor cores read 8-bit operands K-major only, so B (K x N, N
 * contiguous) is transposed into stream-ordered scratch (N x K) before the
 * GEMM: one extra kernel moving 2 x |B| bytes.  With B already stored N x K
 * (dgemm_gemm_ex, op_b = DGEMM_OP_T) nothing is moved.
 * The 8-bit inputs are exact and so are their products in fp32, so only the
 * FP32 accumulation rounds (once per MMA instruction, K/32 times):
 * |C - C_exact| <= 2e-4 * (|A| x |B|) for K <= 16384 (measured: 1e-7).
 * Unknown format: DGEMM_ERR_UNSUPPORTED.
 */
int gemm_f8_tc(int format, int M, int N, int K,
               const unsigned char *A, int lda,
               const unsigned char *B, int ldb,
               float *C, int ldc,
               cudaStream_t stream);

/*
 * dgemm_gemm_ex -- C = op(A) x op(B) on any path, with transposed operands.
 *
 * Lesson 8 section 二十八 ("矩阵布局为什么重要") describes row- and column-major
 * storage and the transpose flags that GEMM interfaces carry for them.  Here
 * every matrix is stored row-major; a transposed operand is simply stored
 * with its other dimension contiguous (a column-major op(X) is a row-major
 * X^T):
 *   op_a = DGEMM_OP_N: A is M x K, lda >= max(1, K);  op(A) = A
 *   op_a = DGEMM_OP_T: A is K x M, lda >= max(1, M);  op(A) = A^T
 *   op_b = DGEMM_OP_N: B is K x N, ldb >= max(1, N);  op(B) = B
 *   op_b = DGEMM_OP_T: B is N x K, ldb >= max(1, K);  op(B) = B^T
 * C is M x N fp32, row-major, ldc >= max(1, N); C[i][j] = sum_k op(A)[i][k]
 * op(B)[k][j].  `path` (dgemm_path_t) selects the arithmetic and the element
 * type of A and B; accuracy, semantics and status codes are those of the
 * corresponding entry point above (gemm_f32_simt, gemm_f32_tc, gemm_bf16_tc,
 * gemm_f16_tc, gemm_f8_tc), which equal dgemm_gemm_ex with op_a = op_b =
 * DGEMM_OP_N.  The FP8 paths read op(A) as M x K and op(B) as N x K natively
 * (op_a = N, op_b = T); other layouts are transposed into scratch first.
 * Unknown path or op: DGEMM_ERR_UNSUPPORTED.
 */
int dgemm_gemm_ex(int path, int op_a, int op_b, int M, int N, int K,
                  const void *A, int lda,
                  const void *B, int ldb,
                  float *C, int ldc,
                  cudaStream_t stream);

/* Static English text for a status code (never NULL). */
const char *dgemm_status_string(int status);

/* The CUDA error text behind the calling thread's last DGEMM_ERR_CUDA
 * ("" if none).  The pointer stays valid until the thread's next call. */
const char *dgemm_last_cuda_error(void);

/*
 * dgemm_watchdog_status -- synchronise `stream`, then read and clear the
 * current device's watchdog word.  The tensor-core kernels bound every wait
 * on a shared-memory barrier; a wait that runs out (a hardware or library
 * fault, never expected in normal use) makes the kernel record where it gave
 * up, drain its copies, free its tensor memory and return, leaving C
 * incomplete.  Returns DGEMM_OK when no kernel gave up since the last read,
 * DGEMM_ERR_WATCHDOG when one did (*where, if not NULL, gets the recorded
 * site code), DGEMM_ERR_CUDA on a CUDA error.  With the environment variable
 * DGEMM_TC_TEST_STALL=1 the first CTA of each tensor-core launch waits on a
 * barrier that nothing arrives at, so that this path can be tested: the call
 * returns after a few seconds with C incomplete and the status set.
 */
int dgemm_watchdog_status(cudaStream_t stream, int *where);

/* Library version as an integer, major*10000 + minor*100 + patch. */
int dgemm_version(void);

/* Number of kernels this library has launched in this process, on any
 * device or stream (a diagnostic for counting launches around a region). */
unsigned long long dgemm_kernel_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* DGEMM_H */
