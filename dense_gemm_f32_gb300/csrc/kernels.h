// kernels.h -- internal launchers behind the C ABI (not exported).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace dg {

// FP32 FFMA GEMM.  ab_vec: A and B rows start on 16-byte boundaries (base
// pointers 16-byte aligned, lda % 4 == 0, ldb % 4 == 0).  c_vec: same for C.
// When the output tiles leave a last wave at most half full, those tiles
// are split along K (partials in stream-ordered scratch, summed in a fixed
// order by the last part to finish).
// a_t: A is stored K x M (op(A) = A^T); b_t: B is stored N x K (op(B) = B^T).
cudaError_t launch_simt(bool a_t, bool b_t, int M, int N, int K, const float *A, int64_t lda,
                        const float *B, int64_t ldb, float *C, int64_t ldc, bool ab_vec,
                        bool c_vec, int num_sms, cudaStream_t stream);

// One operand layout each (unit u = 2 * a_t + b_t, one translation unit each).
#define DG_DECLARE_SIMT_UNIT(u)                                                            \
  cudaError_t launch_simt_unit_##u(int M, int N, int K, const float *A, int64_t lda,       \
                                   const float *B, int64_t ldb, float *C, int64_t ldc,     \
                                   bool ab_vec, bool c_vec, int num_sms, cudaStream_t stream);
DG_DECLARE_SIMT_UNIT(0)
DG_DECLARE_SIMT_UNIT(1)
DG_DECLARE_SIMT_UNIT(2)
DG_DECLARE_SIMT_UNIT(3)
#undef DG_DECLARE_SIMT_UNIT

// C[i*ldc + j] = 0 for i < M, j < N (the empty sum, K == 0).
cudaError_t launch_zero_fill(float *C, int M, int N, int64_t ldc, int num_sms,
                             cudaStream_t stream);

// Element type of a tensor-core GEMM's operands.
enum class TcKind { kTF32 = 0, k3xTF32 = 1, kBF16 = 2, kF16 = 3, kE4M3 = 4, kE5M2 = 5 };

// tcgen05 GEMM, C = op(A) op(B).  a_t: A is stored K x M (op(A) = A^T), else
// M x K; b_t: B is stored N x K (op(B) = B^T), else K x N; all row-major with
// leading dimensions in elements.  A and B must satisfy the TMA rules
// (16-byte aligned base, leading dimension * element size a multiple of 16
// bytes).  C fp32 row-major.
// Problems with few tiles split them along K across thread-block clusters;
// nothing is allocated.
// 3xTF32 on the CTA-pair kernel reads the lo parts of A and B from A_lo and
// B_lo (launch_split_lo, same leading dimensions); with A_lo or B_lo null
// it runs on the single-CTA kernel, which splits in shared memory.
cudaError_t launch_tc(TcKind kind, bool a_t, bool b_t, int M, int N, int K, const void *A,
                      int64_t lda, const void *B, int64_t ldb, float *C, int64_t ldc, bool c_vec,
                      int num_sms, cudaStream_t stream, const void *A_lo = nullptr,
                      const void *B_lo = nullptr);

// One operand layout each (unit u = 2 * a_t + b_t, one translation unit each);
// `watchdog` is the device address of the watchdog word.
#define DG_DECLARE_TC_UNIT(u)                                                                 \
  cudaError_t launch_tc_unit_##u(TcKind kind, int M, int N, int K, const void *A, int64_t lda, \
                                 const void *B, int64_t ldb, float *C, int64_t ldc, bool c_vec, \
                                 int num_sms, int *watchdog, cudaStream_t stream,              \
                                 const void *A_lo, const void *B_lo);
DG_DECLARE_TC_UNIT(0)
DG_DECLARE_TC_UNIT(1)
DG_DECLARE_TC_UNIT(2)
DG_DECLARE_TC_UNIT(3)
#undef DG_DECLARE_TC_UNIT

// Staging of operands TMA cannot read as they are, up to two jobs (A and B)
// in one launch.  A re-pitch copies a rows x cols matrix of elem_bytes-sized
// elements (4, 2 or 1) from (src, lds) to (dst, ldd), the padding columns up
// to ldd zeroed: operands whose rows do not start on 16-byte boundaries (dst
// 16-byte aligned, ldd * elem_bytes a multiple of 16).  A transpose (8-bit
// elements only) writes dst = src^T, cols x rows with ldd >= rows: 8-bit
// operands into the K-major layout the tensor cores read (A as M x K, B as
// N x K).  Leading dimensions are in elements; jobs with no rows or columns
// are skipped.
struct StageJob {
  const void *src;
  int64_t lds;
  void *dst;
  int64_t ldd;
  int rows, cols;  // of the source
  bool transpose;
};
cudaError_t launch_stage(const StageJob *jobs, int njobs, int elem_bytes, int num_sms,
                         cudaStream_t stream);

// 3xTF32 split pre-pass: A_lo = lo(A) (a_rows x a_cols, leading dimension
// lda) and B_lo = lo(B) likewise, lo(x) = x - trunc_tf32(x) rounded to TF32
// (0 for infinities and NaNs), in one launch.  All four bases 16-byte aligned,
// lda and ldb multiples of 4.
cudaError_t launch_split_lo(const float *A, int64_t lda, float *A_lo, int a_rows, int a_cols,
                            const float *B, int64_t ldb, float *B_lo, int b_rows, int b_cols,
                            int num_sms, cudaStream_t stream);

// Whether a tensor-core GEMM of M x N runs on the CTA-pair kernel (256 x 256
// tiles) rather than the single-CTA kernel: once there are enough pair tiles
// to occupy at least a quarter of the SMs, since it has half as many tiles.
// DGEMM_TC_PAIR=0 / =1 forces one of them (read on every call, for tests and
// tuning).
bool tc_use_pair(int M, int N, int num_sms);

// Stream-ordered scratch from the library's memory pool on the current device
// (freed scratch is reused by later allocations; at a synchronisation the pool
// keeps at most its release threshold, 32 MiB by default, reserved).
cudaError_t scratch_alloc(void **ptr, size_t bytes, cudaStream_t stream);
cudaError_t scratch_free(void *ptr, cudaStream_t stream);

// Count one successful kernel launch (dgemm_kernel_launches).
void count_launch();

// Device address of the current device's watchdog word (0, or the site code
// of the first bounded wait that gave up in any kernel of the library);
// nullptr if it cannot be looked up.
int *watchdog_address();

// Read and clear the device's watchdog word after synchronising `stream`.
cudaError_t read_watchdog(cudaStream_t stream, int *code);

}  // namespace dg
