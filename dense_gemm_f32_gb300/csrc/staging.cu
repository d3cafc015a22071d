// staging.cu -- re-pitching of operands the tensor-memory accelerator cannot
// address, and the transpose of 8-bit operands into the K-major layout the
// tensor cores read them in, and the split pre-pass of 3xTF32.
//
// TMA reads a matrix only if its base is 16-byte aligned and its row pitch is
// a multiple of 16 bytes ("第八课：GPU 如何完成矩阵乘法" section 二十二 lists
// data alignment among the conditions for the tensor cores to be used).  An
// operand whose rows miss that (e.g. an odd leading dimension) is copied once
// into scratch with its pitch rounded up to 16 bytes and the padding columns
// zeroed, and the GEMM reads the copy.
#include <cstdint>
#include <cuda_runtime.h>

#include "kernels.h"
#include "launch.cuh"
#include "tf32_split.cuh"

namespace dg {
namespace {

// One operand of a re-pitch launch.
struct RepitchOp {
  const uint8_t *src;
  uint8_t *dst;
  int64_t lds_bytes, ldd_bytes, row_bytes;
  int rows;
};

__global__ void repitch_kernel(RepitchOp op0, RepitchOp op1, int es) {
  // One 16-byte destination chunk per thread-iteration (dst rows are
  // 16-byte aligned, ldd_bytes a multiple of 16): 16 / es element loads from
  // the unaligned source row, one 128-bit store; columns past the row are
  // zeroed.  Rows run along y, chunks along x, so there is no division per
  // element; the operand is grid z (chosen field by field: indexing a
  // parameter array with blockIdx.z would copy the parameters to local memory
  // in every thread).
  pdl_launch_dependents();
  pdl_wait();
  const bool second = blockIdx.z != 0;
  const uint8_t *__restrict__ src = second ? op1.src : op0.src;
  uint8_t *__restrict__ dst = second ? op1.dst : op0.dst;
  const int64_t lds_bytes = second ? op1.lds_bytes : op0.lds_bytes;
  const int64_t ldd_bytes = second ? op1.ldd_bytes : op0.ldd_bytes;
  const int64_t row_bytes = second ? op1.row_bytes : op0.row_bytes;
  const int rows = second ? op1.rows : op0.rows;
  const int64_t chunks = ldd_bytes / 16;
  for (int r = blockIdx.y; r < rows; r += gridDim.y) {
    const uint8_t *srow = src + (int64_t)r * lds_bytes;
    uint4 *drow = reinterpret_cast<uint4 *>(dst + (int64_t)r * ldd_bytes);
    for (int64_t ch = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; ch < chunks;
         ch += (int64_t)gridDim.x * blockDim.x) {
      const int64_t c0 = ch * 16;
      uint32_t w[4];
      if (es == 1) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t v = 0;
#pragma unroll
          for (int b = 0; b < 4; ++b)
            if (c0 + 4 * k + b < row_bytes) v |= (uint32_t)srow[c0 + 4 * k + b] << (8 * b);
          w[k] = v;
        }
      } else if (es == 4) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          w[k] = c0 + 4 * k < row_bytes ? *reinterpret_cast<const uint32_t *>(srow + c0 + 4 * k)
                                        : 0u;
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t lo = c0 + 4 * k < row_bytes
                                  ? *reinterpret_cast<const uint16_t *>(srow + c0 + 4 * k) : 0u;
          const uint32_t hi = c0 + 4 * k + 2 < row_bytes
                                  ? *reinterpret_cast<const uint16_t *>(srow + c0 + 4 * k + 2) : 0u;
          w[k] = lo | (hi << 16);
        }
      }
      drow[ch] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// dst = src^T for a rows x cols matrix of bytes: dst[c][r] = src[r][c].
// 64 x 64-byte tiles, 256 threads.  Interior tiles whose rows are 4-byte
// aligned move 32-bit words: each thread loads four words of one 4 x 4-byte
// block through shared memory and transposes it in registers with byte
// permutes; sixteen threads cover 64 contiguous bytes of an output row.
// Edge tiles and unaligned operands go byte by byte.
constexpr int kT = 64;
__global__ void __launch_bounds__(256)
    transpose8_kernel(const uint8_t *__restrict__ src, int64_t lds, uint8_t *__restrict__ dst,
                      int64_t ldd, int rows, int cols, int words_ok) {
  __shared__ uint32_t tile[kT][kT / 4 + 1];
  pdl_launch_dependents();
  pdl_wait();
  const int tid = threadIdx.x;
  const int tiles_c = (cols + kT - 1) / kT;
  const int64_t ntiles = (int64_t)((rows + kT - 1) / kT) * tiles_c;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int r0 = (int)(t / tiles_c) * kT, c0 = (int)(t % tiles_c) * kT;
    const bool full = words_ok && r0 + kT <= rows && c0 + kT <= cols;
    if (full) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int r = tid / 16 + 16 * k, w = tid % 16;
        tile[r][w] = *reinterpret_cast<const uint32_t *>(src + (int64_t)(r0 + r) * lds + c0 + 4 * w);
      }
      __syncthreads();
      const int cb = tid / 16, rb = tid % 16;  // 4-column block, 4-row block
      const uint32_t x0 = tile[4 * rb][cb], x1 = tile[4 * rb + 1][cb];
      const uint32_t x2 = tile[4 * rb + 2][cb], x3 = tile[4 * rb + 3][cb];
      const uint32_t t0 = __byte_perm(x0, x1, 0x5140), t1 = __byte_perm(x2, x3, 0x5140);
      const uint32_t t2 = __byte_perm(x0, x1, 0x7362), t3 = __byte_perm(x2, x3, 0x7362);
      const uint32_t o[4] = {__byte_perm(t0, t1, 0x5410), __byte_perm(t0, t1, 0x7632),
                             __byte_perm(t2, t3, 0x5410), __byte_perm(t2, t3, 0x7632)};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint32_t *>(dst + (int64_t)(c0 + 4 * cb + j) * ldd + r0 + 4 * rb) = o[j];
      __syncthreads();
    } else {
      for (int e = tid; e < kT * kT; e += blockDim.x) {
        const int i = e / kT, j = e % kT;  // output row c0 + i, output column r0 + j
        if (c0 + i < cols && r0 + j < rows)
          dst[(int64_t)(c0 + i) * ldd + r0 + j] = src[(int64_t)(r0 + j) * lds + c0 + i];
      }
    }
  }
}

// lo part of the 3xTF32 split of one operand: L[r][c] = split_lo(X[r][c])
// for r < rows, c < cols, with the same leading dimension (a multiple of 4,
// both bases 16-byte aligned: the operand already meets the TMA rules).
struct SplitOperand {
  const uint32_t *x;
  uint32_t *lo;
  int64_t ld;
  int rows, cols;
};

// Blocks [0, blocks_a) split operand a, the rest operand b.  Within an
// operand: rows along blockIdx (grid-stride), 16-byte chunks of a row along
// the threads; the chunk at the end of a row that is not whole goes element by
// element (the row may end there in memory).
__global__ void split_lo_kernel(SplitOperand a, SplitOperand b, int blocks_a) {
  pdl_launch_dependents();
  pdl_wait();
  const bool first = (int)blockIdx.x < blocks_a;
  const SplitOperand op = first ? a : b;
  const int nblocks = first ? blocks_a : (int)gridDim.x - blocks_a;
  const int bid = first ? (int)blockIdx.x : (int)blockIdx.x - blocks_a;
  const int chunks = (op.cols + 3) / 4;
  const int whole = op.cols / 4;
  for (int r = bid; r < op.rows; r += nblocks) {
    const uint32_t *xr = op.x + (int64_t)r * op.ld;
    uint32_t *lr = op.lo + (int64_t)r * op.ld;
    for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
      if (c < whole) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(xr) + c);
        reinterpret_cast<uint4 *>(lr)[c] = make_uint4(split_lo_tf32(v.x), split_lo_tf32(v.y),
                                                      split_lo_tf32(v.z), split_lo_tf32(v.w));
      } else {
        for (int j = 4 * c; j < op.cols; ++j) lr[j] = split_lo_tf32(__ldg(xr + j));
      }
    }
  }
}

}  // namespace

cudaError_t launch_transpose8(const void *src, int64_t lds, void *dst, int64_t ldd, int rows,
                              int cols, int num_sms, cudaStream_t stream) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  const int64_t ntiles = (int64_t)((rows + kT - 1) / kT) * ((cols + kT - 1) / kT);
  int64_t grid = (int64_t)num_sms * 8;
  if (grid > ntiles) grid = ntiles;
  const bool words_ok = reinterpret_cast<uintptr_t>(src) % 4 == 0 && lds % 4 == 0 &&
                        reinterpret_cast<uintptr_t>(dst) % 4 == 0 && ldd % 4 == 0;
  const cudaError_t e = launch_kernel(transpose8_kernel, dim3((unsigned)grid), dim3(256), 0, stream, 1,
                                      static_cast<const uint8_t *>(src), lds,
                                      static_cast<uint8_t *>(dst), ldd, rows, cols,
                                      words_ok ? 1 : 0);
  if (e == cudaSuccess) count_launch();
  return e;
}

cudaError_t launch_repitch(const RepitchJob *jobs, int njobs, int elem_bytes, int num_sms,
                           cudaStream_t stream) {
  RepitchOp ops[2] = {};
  int n = 0, max_rows = 0;
  int64_t max_chunks = 0;
  for (int j = 0; j < njobs && j < 2; ++j) {
    if (jobs[j].rows <= 0) continue;
    RepitchOp &o = ops[n++];
    o.src = static_cast<const uint8_t *>(jobs[j].src);
    o.dst = static_cast<uint8_t *>(jobs[j].dst);
    o.lds_bytes = jobs[j].lds * elem_bytes;
    o.ldd_bytes = jobs[j].ldd * elem_bytes;
    o.row_bytes = (int64_t)jobs[j].cols * elem_bytes;
    o.rows = jobs[j].rows;
    const int64_t chunks = o.ldd_bytes / 16;
    max_chunks = chunks > max_chunks ? chunks : max_chunks;
    max_rows = o.rows > max_rows ? o.rows : max_rows;
  }
  if (n == 0) return cudaSuccess;
  const int bx = (int)((max_chunks + 255) / 256 < 8 ? (max_chunks + 255) / 256 : 8);
  int64_t by = (int64_t)num_sms * 16 / (bx * n);
  if (by > max_rows) by = max_rows;
  if (by > 65535) by = 65535;
  if (by < 1) by = 1;
  const cudaError_t e = launch_kernel(repitch_kernel, dim3((unsigned)bx, (unsigned)by, (unsigned)n),
                                      dim3(256), 0, stream, 1, ops[0], ops[1], elem_bytes);
  if (e == cudaSuccess) count_launch();
  return e;
}

cudaError_t launch_split_lo(const float *A, int64_t lda, float *A_lo, int a_rows, int a_cols,
                            const float *B, int64_t ldb, float *B_lo, int b_rows, int b_cols,
                            int num_sms, cudaStream_t stream) {
  if ((a_rows <= 0 || a_cols <= 0) && (b_rows <= 0 || b_cols <= 0)) return cudaSuccess;
  const SplitOperand a = {reinterpret_cast<const uint32_t *>(A), reinterpret_cast<uint32_t *>(A_lo),
                          lda, a_cols > 0 ? a_rows : 0, a_cols};
  const SplitOperand b = {reinterpret_cast<const uint32_t *>(B), reinterpret_cast<uint32_t *>(B_lo),
                          ldb, b_cols > 0 ? b_rows : 0, b_cols};
  // blocks in proportion to the bytes of each operand, 8 per SM in all
  const double ea = (double)a.rows * a_cols, eb = (double)b.rows * b_cols;
  const int total = num_sms * 8;
  int ba = (int)(total * ea / (ea + eb) + 0.5);
  if (ba < 1 && a.rows > 0) ba = 1;
  if (ba > a.rows) ba = a.rows;
  int bb = total - ba;
  if (bb < 1 && b.rows > 0) bb = 1;
  if (bb > b.rows) bb = b.rows;
  const cudaError_t e = launch_kernel(split_lo_kernel, dim3((unsigned)(ba + bb)), dim3(256), 0,
                                      stream, 1, a, b, ba);
  if (e == cudaSuccess) count_launch();
  return e;
}

}  // namespace dg
