// staging.cu -- re-pitching of operands the tensor-memory accelerator cannot
// address.
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

namespace dg {
namespace {

__global__ void repitch_kernel(const uint8_t *__restrict__ src, int64_t lds_bytes,
                               uint8_t *__restrict__ dst, int64_t ldd_bytes, int rows,
                               int64_t row_bytes, int es) {
  // One 16-byte destination chunk per thread-iteration (dst rows are
  // 16-byte aligned, ldd_bytes a multiple of 16): 16 / es element loads from
  // the unaligned source row, one 128-bit store; columns past the row are
  // zeroed.  Rows run along y, chunks along x, so there is no division per
  // element.
  const int64_t chunks = ldd_bytes / 16;
  for (int r = blockIdx.y; r < rows; r += gridDim.y) {
    const uint8_t *srow = src + (int64_t)r * lds_bytes;
    uint4 *drow = reinterpret_cast<uint4 *>(dst + (int64_t)r * ldd_bytes);
    for (int64_t ch = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; ch < chunks;
         ch += (int64_t)gridDim.x * blockDim.x) {
      const int64_t c0 = ch * 16;
      uint32_t w[4];
      if (es == 4) {
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

}  // namespace

cudaError_t launch_repitch(const void *src, int64_t lds, void *dst, int64_t ldd, int rows,
                           int cols, int elem_bytes, int num_sms, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const int64_t chunks = ldd * elem_bytes / 16;
  const int bx = (int)((chunks + 255) / 256 < 8 ? (chunks + 255) / 256 : 8);
  int64_t by = (int64_t)num_sms * 16 / bx;
  if (by > rows) by = rows;
  if (by > 65535) by = 65535;
  if (by < 1) by = 1;
  repitch_kernel<<<dim3((unsigned)bx, (unsigned)by), 256, 0, stream>>>(
      static_cast<const uint8_t *>(src), lds * elem_bytes, static_cast<uint8_t *>(dst),
      ldd * elem_bytes, rows, (int64_t)cols * elem_bytes, elem_bytes);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

}  // namespace dg
