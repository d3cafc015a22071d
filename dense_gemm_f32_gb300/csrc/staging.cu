// staging.cu -- re-pitching of operands the tensor-memory accelerator cannot
// address, and the transpose of 8-bit operands into the K-major layout the
// tensor cores read them in, and the split pre-pass of 3xTF32.
//
// TMA reads a matrix only if its base is 16-byte aligned and its row pitch is
// a multiple of 16 bytes ("第八课：GPU 如何完成矩阵乘法" section 二十二 lists
// data alignment among the conditions for the tensor cores to be used).  An
// operand whose rows miss that (e.g. an odd leading dimension) is copied once
// into scratch with its pitch rounded up to 16 bytes and the padding columns
// zeroed, and the GEMM reads the copy.  Whatever a call needs for its two
// operands (a re-pitch, a transpose, one of each) goes out in one launch.
#include <cstdint>
#include <cuda_runtime.h>

#include "kernels.h"
#include "launch.cuh"
#include "tf32_split.cuh"

namespace dg {
namespace {

// One job of a staging launch, in bytes.
struct StageOp {
  const uint8_t *src;
  uint8_t *dst;
  int64_t lds, ldd;   // leading dimensions (bytes)
  int64_t row_bytes;  // bytes of a source row
  int rows, cols;     // source rows; source columns (bytes)
  int transpose;      // 1: byte transpose, 0: re-pitch
  int aux;            // transpose: 32-bit words allowed; re-pitch: log2(threads per row)
};

// Bytes off .. off + 15 of the 32 bytes x then y (little-endian words).  off
// is a multiple of the element size ES: 4-byte elements need only a choice of
// words, narrower ones a funnel shift as well.
template <int ES>
__device__ __forceinline__ uint4 bytes_at(uint4 x, uint4 y, int off) {
  const uint32_t w[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
  const int s = off >> 2;
  uint32_t a[5];
#pragma unroll
  for (int j = 0; j < 5; ++j) a[j] = s == 0 ? w[j] : s == 1 ? w[j + 1] : s == 2 ? w[j + 2] : w[j + 3];
  if constexpr (ES == 4) {
    return make_uint4(a[0], a[1], a[2], a[3]);
  } else {
    const int sh = 8 * (off & 3);
    return make_uint4(__funnelshift_r(a[0], a[1], sh), __funnelshift_r(a[1], a[2], sh),
                      __funnelshift_r(a[2], a[3], sh), __funnelshift_r(a[3], a[4], sh));
  }
}

// Row bytes [pos, pos + 16) (pos a multiple of 16), zero past the row's end,
// by element-sized loads of the elements inside the row, all issued before any
// is combined.
template <int ES>
__device__ __forceinline__ uint4 row_chunk(const uint8_t *__restrict__ srow, int64_t pos,
                                           int64_t row_bytes) {
  uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int k = 0; k < 16; k += ES) {
    if (pos + k < row_bytes) {
      uint32_t e;
      if constexpr (ES == 4)
        e = *reinterpret_cast<const uint32_t *>(srow + pos + k);
      else if constexpr (ES == 2)
        e = *reinterpret_cast<const uint16_t *>(srow + pos + k);
      else
        e = srow[pos + k];
      w[k >> 2] |= e << (8 * (k & 3));
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Re-pitch of ES-byte elements: destination row r is the source row's bytes
// followed by zeros up to ldd (the destination 16-byte aligned, ldd a
// multiple of 16).  A 16-byte destination chunk whose source bytes straddle
// two aligned 16-byte blocks lying wholly inside the row is made from two
// 128-bit loads; the chunks at the row's two ends load their own elements, so
// no byte outside the row is read.  Either way a chunk costs one memory round
// trip.  A block's 1 << aux threads share a row, so that short rows fill the
// block with several rows instead of leaving threads idle.
template <int ES>
__device__ __forceinline__ void repitch_rows(const StageOp &op, int bid, int nblocks) {
  const int lg = op.aux;
  const int cx = 1 << lg;
  const int lane = (int)threadIdx.x & (cx - 1);
  const int rpb = (int)blockDim.x >> lg;  // rows per block
  const int chunks = (int)(op.ldd / 16);
  const int64_t row_bytes = op.row_bytes;
  for (int64_t r = (int64_t)bid * rpb + ((int)threadIdx.x >> lg); r < op.rows;
       r += (int64_t)nblocks * rpb) {
    const uint8_t *srow = op.src + r * op.lds;
    const int off = (int)(reinterpret_cast<uintptr_t>(srow) & 15);
    // Aligned block b covers row bytes [16 b - off, 16 b - off + 16), and
    // chunk ch (row bytes [16 ch, 16 ch + 16)) is bytes off .. off + 15 of
    // blocks ch and ch + 1 (block ch alone if off = 0).  Those blocks lie
    // wholly inside the row for ch in [ch_lo, ch_hi).
    const uint4 *blocks = reinterpret_cast<const uint4 *>(srow - off);
    const int ch_lo = off != 0;
    const int64_t hi = (row_bytes + off - (off != 0 ? 16 : 0)) / 16;
    const int ch_hi = hi < 0 ? 0 : hi > chunks ? chunks : (int)hi;
    uint4 *drow = reinterpret_cast<uint4 *>(op.dst + r * op.ldd);
    for (int ch = lane; ch < chunks; ch += cx) {
      uint4 v;
      if (ch >= ch_lo && ch < ch_hi) {
        const uint4 x = __ldg(blocks + ch);
        const uint4 y = off != 0 ? __ldg(blocks + ch + 1) : x;
        v = bytes_at<ES>(x, y, off);
      } else {
        v = row_chunk<ES>(srow, 16 * (int64_t)ch, row_bytes);
      }
      drow[ch] = v;
    }
  }
}

// Byte transpose: dst[c][r] = src[r][c] for the rows x cols source, over
// 64 x 64-byte tiles (256 threads).  Interior tiles whose rows are 4-byte
// aligned move 32-bit words: each thread loads four words of one 4 x 4-byte
// block through shared memory and transposes it in registers with byte
// permutes; sixteen threads cover 64 contiguous bytes of an output row.
// Edge tiles and unaligned operands go byte by byte, each thread's sixteen
// loads issued together (a tile then costs one memory round trip, not one
// per byte a thread moves).
constexpr int kT = 64;
constexpr int kTileBytes = kT * (kT / 4 + 1) * 4;  // dynamic shared memory of a transposing launch
__device__ __forceinline__ void transpose_tiles(const StageOp &op, int bid, int nblocks,
                                                uint32_t (*tile)[kT / 4 + 1]) {
  const int tid = threadIdx.x;
  const int rows = op.rows, cols = op.cols;
  const uint8_t *__restrict__ src = op.src;
  uint8_t *__restrict__ dst = op.dst;
  const int tiles_c = (cols + kT - 1) / kT;
  const int64_t ntiles = (int64_t)((rows + kT - 1) / kT) * tiles_c;
  for (int64_t t = bid; t < ntiles; t += nblocks) {
    const int r0 = (int)(t / tiles_c) * kT, c0 = (int)(t % tiles_c) * kT;
    const bool full = op.aux && r0 + kT <= rows && c0 + kT <= cols;
    if (full) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int r = tid / 16 + 16 * k, w = tid % 16;
        tile[r][w] = *reinterpret_cast<const uint32_t *>(src + (int64_t)(r0 + r) * op.lds + c0 + 4 * w);
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
        *reinterpret_cast<uint32_t *>(dst + (int64_t)(c0 + 4 * cb + j) * op.ldd + r0 + 4 * rb) = o[j];
      __syncthreads();
    } else {  // 16 bytes a thread, every load in flight before the first store
      constexpr int kPer = kT * kT / 256;
      uint32_t v[kPer / 4] = {};  // byte k of the thread in byte k % 4 of word k / 4
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int i = tid / kT + (256 / kT) * k, j = tid % kT;  // output row c0 + i, column r0 + j
        if (c0 + i < cols && r0 + j < rows)
          v[k / 4] |= (uint32_t)src[(int64_t)(r0 + j) * op.lds + c0 + i] << (8 * (k % 4));
      }
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int i = tid / kT + (256 / kT) * k, j = tid % kT;
        if (c0 + i < cols && r0 + j < rows)
          dst[(int64_t)(c0 + i) * op.ldd + r0 + j] = (uint8_t)(v[k / 4] >> (8 * (k % 4)));
      }
    }
  }
}

// Up to two staging jobs in one launch, of ES-byte elements (transposes for
// ES = 1 only): blocks [0, blocks0) take job 0, the rest job 1 (the job
// chosen field by field: indexing a parameter array by block would copy the
// parameters to local memory in every thread).  A job's role is uniform over
// a block, so the transpose's block barriers are safe.  Shared memory is
// dynamic and given only to launches with a transpose, so that re-pitch
// blocks leave room for the GEMM's CTAs, which are launched beside them
// (programmatic dependent launch) and wait for them to finish.
template <int ES>
__global__ void __launch_bounds__(256, 8) stage_kernel(StageOp j0, StageOp j1, int blocks0) {
  pdl_launch_dependents();
  pdl_wait();
  const bool first = (int)blockIdx.x < blocks0;
  const StageOp op = first ? j0 : j1;
  const int bid = first ? (int)blockIdx.x : (int)blockIdx.x - blocks0;
  const int nblocks = first ? blocks0 : (int)gridDim.x - blocks0;
  if constexpr (ES == 1) {
    if (op.transpose) {
      extern __shared__ uint32_t stage_smem[];
      transpose_tiles(op, bid, nblocks, reinterpret_cast<uint32_t(*)[kT / 4 + 1]>(stage_smem));
      return;
    }
  }
  repitch_rows<ES>(op, bid, nblocks);
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

cudaError_t launch_stage(const StageJob *jobs, int njobs, int elem_bytes, int num_sms,
                         cudaStream_t stream) {
  StageOp ops[2] = {};
  int blocks[2] = {0, 0};
  int n = 0;
  for (int j = 0; j < njobs && j < 2; ++j) {
    if (jobs[j].transpose && elem_bytes != 1) return cudaErrorInvalidValue;  // 8-bit only
    if (jobs[j].rows > 0 && jobs[j].cols > 0) ++n;
  }
  for (int j = 0, k = 0; j < njobs && j < 2; ++j) {
    const StageJob &jb = jobs[j];
    if (jb.rows <= 0 || jb.cols <= 0) continue;
    StageOp &o = ops[k];
    o.src = static_cast<const uint8_t *>(jb.src);
    o.dst = static_cast<uint8_t *>(jb.dst);
    o.lds = jb.lds * elem_bytes;
    o.ldd = jb.ldd * elem_bytes;
    o.row_bytes = (int64_t)jb.cols * elem_bytes;
    o.rows = jb.rows;
    o.cols = jb.cols * elem_bytes;
    o.transpose = jb.transpose ? 1 : 0;
    int64_t b;
    if (jb.transpose) {  // 64 x 64 tiles, up to 8 blocks per SM
      o.aux = reinterpret_cast<uintptr_t>(jb.src) % 4 == 0 && o.lds % 4 == 0 &&
              reinterpret_cast<uintptr_t>(jb.dst) % 4 == 0 && o.ldd % 4 == 0;
      b = (int64_t)((o.rows + kT - 1) / kT) * ((o.cols + kT - 1) / kT);
      if (b > (int64_t)num_sms * 8) b = (int64_t)num_sms * 8;
    } else {  // threads per row: the chunks of a row rounded up to a power of two, at most 256
      const int64_t chunks = o.ldd / 16;
      int lg = 0;
      while (lg < 8 && ((int64_t)1 << lg) < chunks) ++lg;
      o.aux = lg;
      const int rpb = 256 >> lg;
      b = (o.rows + rpb - 1) / rpb;
      if (b > (int64_t)num_sms * 16 / n) b = (int64_t)num_sms * 16 / n;
    }
    blocks[k++] = (int)(b < 1 ? 1 : b);
  }
  if (n == 0) return cudaSuccess;
  const size_t smem = ops[0].transpose || ops[1].transpose ? kTileBytes : 0;
  void (*kern)(StageOp, StageOp, int) =
      elem_bytes == 4 ? stage_kernel<4> : elem_bytes == 2 ? stage_kernel<2> : stage_kernel<1>;
  const cudaError_t e = launch_kernel(kern, dim3((unsigned)(blocks[0] + blocks[1])), dim3(256), smem,
                                      stream, 1, ops[0], ops[1], blocks[0]);
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
