// simt.cu -- FP32 GEMM on the CUDA cores (FFMA), register blocked.
//
// The block-tiled, register-blocked SGEMM that "SGEMM 优化旅程" builds up in
// Levels 2-5, with the sizes its Level 5 names (block tile 128 x 128 x 8,
// 256 threads, an 8 x 8 register tile per thread), and the structure of
// "第八课：GPU 如何完成矩阵乘法": C_tile = sum_t A_tile,t x B_tile,t (section 九),
// accumulation in registers with one store per element (section 十四),
// multi-level block / warp / thread tiling (section 十九), double-buffered
// shared memory (section 二十四), zero-fill and masked stores at the edges
// (section 二十六), padding against bank conflicts (section 二十七).
//
// GB300 specifics that differ from the pages' kernels:
//  * A is stored transposed (k-major) in shared memory, so that both operand
//    fragments are read with 128-bit shared loads; the transposed stores use a
//    4-float row padding, which makes them bank-conflict free.
//  * The per-warp tile is 64 x 32 with 8 x 4 lanes, so each 128-bit fragment
//    load of a warp touches one 128-byte line (one shared-memory wavefront).
//  * Global loads are 128-bit where the operand rows are 16-byte aligned
//    (template kVec); ragged edges fall back to masked scalar loads.
//  * Thread blocks walk the C tiles in groups of 8 tile rows so that panels
//    of A and B are re-read from L2 instead of HBM.
#include <cstdint>
#include <cuda_runtime.h>

#include "kernels.h"

namespace dg {
namespace {

constexpr int BM = 128, BN = 128, BK = 8;
constexpr int kThreads = 256;
constexpr int kApad = 4;          // As row = BM + 4 floats (528 B, 16-B multiple)
constexpr int kGroupM = 8;        // tile rows per raster group

// Load 4 consecutive elements X[r][c..c+3] of an R x Cn row-major matrix,
// zero outside it.  kVec: the row start is 16-byte aligned and c % 4 == 0.
template <bool kVec>
__device__ __forceinline__ float4 load4(const float *__restrict__ X, int64_t ld, int r, int c,
                                        int R, int Cn) {
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  if (r < R) {
    const float *q = X + (int64_t)r * ld + c;
    if (kVec && c + 3 < Cn) {
      v = __ldg(reinterpret_cast<const float4 *>(q));
    } else {
      if (c + 0 < Cn) v.x = __ldg(q + 0);
      if (c + 1 < Cn) v.y = __ldg(q + 1);
      if (c + 2 < Cn) v.z = __ldg(q + 2);
      if (c + 3 < Cn) v.w = __ldg(q + 3);
    }
  }
  return v;
}

template <bool kVec>
__global__ void __launch_bounds__(kThreads, 2)
    sgemm_simt_kernel(int M, int N, int K, const float *__restrict__ A, int64_t lda,
                      const float *__restrict__ B, int64_t ldb, float *__restrict__ C,
                      int64_t ldc, int c_vec) {
  __shared__ __align__(16) float As[2][BK][BM + kApad];
  __shared__ __align__(16) float Bs[2][BK][BN];

  // ---- grouped raster: tile id -> (tile row, tile col)
  const int tiles_m = (M + BM - 1) / BM;
  const int tiles_n = (N + BN - 1) / BN;
  const int tile = blockIdx.x;
  const int per_group = kGroupM * tiles_n;
  const int group = tile / per_group;
  const int first_m = group * kGroupM;
  const int gsize = min(tiles_m - first_m, kGroupM);
  const int in_group = tile - group * per_group;
  const int tm = first_m + in_group % gsize;
  const int tn = in_group / gsize;
  const int m0 = tm * BM, n0 = tn * BN;

  const int tid = threadIdx.x;
  // global -> shared load assignment: one float4 of A and one of B per thread
  const int a_row = tid >> 1, a_col = (tid & 1) * 4;     // A tile 128 x 8
  const int b_row = tid >> 5, b_col = (tid & 31) * 4;    // B tile 8 x 128

  // compute assignment: warp tile 64 x 32, lanes 8 (M) x 4 (N), thread 8 x 8
  const int warp = tid >> 5, lane = tid & 31;
  const int wm = warp >> 2, wn = warp & 3;               // 2 x 4 warps
  const int lm = lane >> 2, ln = lane & 3;
  const int row_base = wm * 64 + lm * 4;                 // rows row_base + {0..3, 32..35}
  const int col_base = wn * 32 + ln * 4;                 // cols col_base + {0..3, 16..19}

  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  const int KT = (K + BK - 1) / BK;

  float4 ra = load4<kVec>(A, lda, m0 + a_row, a_col, M, K);
  float4 rb = load4<kVec>(B, ldb, b_row, n0 + b_col, K, N);
  As[0][a_col + 0][a_row] = ra.x;
  As[0][a_col + 1][a_row] = ra.y;
  As[0][a_col + 2][a_row] = ra.z;
  As[0][a_col + 3][a_row] = ra.w;
  *reinterpret_cast<float4 *>(&Bs[0][b_row][b_col]) = rb;
  __syncthreads();

  for (int kt = 0; kt < KT; ++kt) {
    const int cur = kt & 1;
    const bool more = kt + 1 < KT;
    if (more) {
      const int k0 = (kt + 1) * BK;
      ra = load4<kVec>(A, lda, m0 + a_row, k0 + a_col, M, K);
      rb = load4<kVec>(B, ldb, k0 + b_row, n0 + b_col, K, N);
    }
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4 *>(&As[cur][kk][row_base]);
      const float4 a1 = *reinterpret_cast<const float4 *>(&As[cur][kk][row_base + 32]);
      const float4 b0 = *reinterpret_cast<const float4 *>(&Bs[cur][kk][col_base]);
      const float4 b1 = *reinterpret_cast<const float4 *>(&Bs[cur][kk][col_base + 16]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    if (more) {
      const int nxt = cur ^ 1;
      As[nxt][a_col + 0][a_row] = ra.x;
      As[nxt][a_col + 1][a_row] = ra.y;
      As[nxt][a_col + 2][a_row] = ra.z;
      As[nxt][a_col + 3][a_row] = ra.w;
      *reinterpret_cast<float4 *>(&Bs[nxt][b_row][b_col]) = rb;
    }
    __syncthreads();
  }

  // ---- epilogue: masked stores, 128-bit where C rows are 16-byte aligned
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = m0 + row_base + (i & 3) + (i >> 2) * 32;
    if (r >= M) continue;
    float *crow = C + (int64_t)r * ldc;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = n0 + col_base + h * 16;
      const float *v = &acc[i][h * 4];
      if (c_vec && c + 3 < N) {
        *reinterpret_cast<float4 *>(crow + c) = make_float4(v[0], v[1], v[2], v[3]);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (c + j < N) crow[c + j] = v[j];
      }
    }
  }
}

__global__ void zero_fill_kernel(float *__restrict__ C, int M, int N, int64_t ldc) {
  const int64_t total = (int64_t)M * N;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = e / N, c = e - r * N;
    C[r * ldc + c] = 0.f;
  }
}

}  // namespace

cudaError_t launch_simt(int M, int N, int K, const float *A, int64_t lda, const float *B,
                        int64_t ldb, float *C, int64_t ldc, bool ab_vec, bool c_vec,
                        cudaStream_t stream) {
  const int64_t tiles = (int64_t)((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  if (tiles > 0x7fffffff) return cudaErrorInvalidValue;
  dim3 grid((unsigned)tiles), block(kThreads);
  if (ab_vec)
    sgemm_simt_kernel<true><<<grid, block, 0, stream>>>(M, N, K, A, lda, B, ldb, C, ldc, c_vec);
  else
    sgemm_simt_kernel<false><<<grid, block, 0, stream>>>(M, N, K, A, lda, B, ldb, C, ldc, c_vec);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

cudaError_t launch_zero_fill(float *C, int M, int N, int64_t ldc, int num_sms,
                             cudaStream_t stream) {
  const int64_t total = (int64_t)M * N;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = (int64_t)num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  zero_fill_kernel<<<(unsigned)blocks, 256, 0, stream>>>(C, M, N, ldc);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

}  // namespace dg
