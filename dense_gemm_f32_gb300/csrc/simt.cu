// simt.cu -- FP32 GEMM on the CUDA cores (FFMA), register blocked.
//
// The block-tiled, register-blocked SGEMM that "SGEMM 优化旅程" builds up in
// Levels 2-5 (shared-memory tiles, padding against bank conflicts, double
// buffering, a register tile per thread) with the structure of
// "第八课：GPU 如何完成矩阵乘法": C_tile = sum_t A_tile,t x B_tile,t (section 九),
// accumulation in registers with one store per element (section 十四),
// multi-level block / warp / thread tiling (section 十九), copies that run
// ahead of the arithmetic (sections 二十三-二十五), zero-fill and masked
// stores at the edges (section 二十六), no bank conflicts (section 二十七).
//
// Two kernels:
//  * sgemm_ring_kernel (operands TMA can address, B stored K x N): the
//    global -> shared copies are TMA boxes into a ring of STAGES stages,
//    each with a "full" mbarrier (the copy's bytes landed) and an "empty"
//    mbarrier (every warp is done reading it).  No thread stages data in
//    registers and there is no block-wide barrier in the main loop; the lane
//    that refills a stage rotates over the warps.  A lands k-contiguous in
//    128B-swizzled rows (or k-major when stored K x M) and every thread owns
//    rows 8 apart, so one 128-bit shared load per row gives four k values
//    and the eight rows of a warp's load fall in eight different bank groups.
//  * sgemm_simt_kernel (other operands: rows that are not 16-byte aligned, B
//    stored N x K, and small problems): 128-bit global loads into registers,
//    stored to one of two shared buffers (A transposed, +4-float row pad),
//    one block-wide barrier per k-block.
// Both issue the inner product as packed fma.rn.f32x2: each row of the
// register tile does {a_i, a_i} x {b_2h, b_2h+1} + acc, every multiply-add
// rounded once in k order, so C is bitwise what scalar FFMAs give.
// Shapes were chosen by measurement on GB300 (tile shapes, stages, warp and
// lane layouts, FMA order).
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>
#include <cuda_runtime.h>

#include "kernels.h"
#include "launch.cuh"
#include "ptx.cuh"
#include "tmap.cuh"

// This file is compiled once per operand layout: DGEMM_SIMT_UNIT = 2 * AT + BT
// (AT: A stored K x M; BT: B stored N x K), so the layouts compile in
// parallel.  Unit 0 also holds the dispatch and the zero fill.
#ifndef DGEMM_SIMT_UNIT
#define DGEMM_SIMT_UNIT 0
#endif
// 1 (default): the inner product issues the packed two-wide fma.rn.f32x2,
// one instruction per two multiply-adds of a row of the register tile; 0:
// scalar fmaf.  Both round each multiply-add once, in the same order, so they
// give bitwise identical C.  The kernel is bound by instruction issue (about
// 12% of its instructions are not FFMAs), and halving the FFMA instructions
// measured 52.7 -> 59.8 TFLOP/s at 8192^3 on GB300.
#ifndef DGEMM_SIMT_FFMA2
#define DGEMM_SIMT_FFMA2 1
#endif
#define DG_SCAT2(a, b) a##b
#define DG_SCAT(a, b) DG_SCAT2(a, b)
#define DG_SIMT_UNIT_LAUNCHER DG_SCAT(launch_simt_unit_, DGEMM_SIMT_UNIT)

namespace dg {
namespace {

constexpr bool kUnitAT = (DGEMM_SIMT_UNIT >> 1) & 1;
constexpr bool kUnitBT = DGEMM_SIMT_UNIT & 1;
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

// After a kernel's main loop: the thread's TM x TN accumulators, acc[i][4h ..
// 4h + 3] at tile row row_of(i) and tile columns col_of(h) .. + 3, go to C.
//  * Whole tile: masked stores, 128-bit where C's rows are 16-byte aligned.
//  * K-split over a cluster (every tile split, cluster_parts != 0): the part
//    parks its partial tile in its own shared memory at `park` (BM rows of
//    PART_PITCH floats; the caller has made sure nothing else uses it any
//    more), then each CTA adds one slice of the tile's rows over all parts,
//    in part order, through distributed shared memory and writes it to C.
//    Every thread reaches both cluster barriers.
//  * K-split through scratch (the tiles of a partial last wave): the part
//    writes its partial tile to `work`; the last part to finish (an atomic
//    counter) sums all parts in part order, so the result does not depend on
//    which finishes last, and writes C.
template <int BM, int BN, int THREADS, int TM, int TN, int PART_PITCH, class RowOf, class ColOf>
__device__ __forceinline__ void finish_tile(const float (&acc)[TM][TN], RowOf row_of, ColOf col_of,
                                            float *park, int M, int N, float *__restrict__ C,
                                            int64_t ldc, int c_vec, int m0, int n0, bool split,
                                            int tile, int part, int split_first, int split_parts,
                                            float *__restrict__ work,
                                            unsigned int *__restrict__ counters,
                                            int cluster_parts) {
  const int tid = threadIdx.x;
  if (split && cluster_parts) {
#pragma unroll
    for (int i = 0; i < TM; ++i) {
      const int rl = row_of(i);
#pragma unroll
      for (int h = 0; h < TN / 4; ++h)
        *reinterpret_cast<float4 *>(park + rl * PART_PITCH + col_of(h)) =
            make_float4(acc[i][h * 4], acc[i][h * 4 + 1], acc[i][h * 4 + 2], acc[i][h * 4 + 3]);
    }
    __syncwarp();
    cluster_sync();  // partials written (release) and visible (acquire)
    const int rank = (int)cluster_ctarank();
    const int r0 = (BM * rank) / split_parts, r1 = (BM * (rank + 1)) / split_parts;
    constexpr int Q = BN / 4;
    const uint32_t base = smem_u32(park);
    uint32_t peer[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) peer[p] = p < split_parts ? mapa_shared(base, (uint32_t)p) : 0u;
    for (int e = tid; e < (r1 - r0) * Q; e += THREADS) {
      const int rl = r0 + e / Q, cl = 4 * (e % Q);
      const uint32_t off = (uint32_t)((rl * PART_PITCH + cl) * 4);
      float4 v[8];
#pragma unroll
      for (int p = 0; p < 8; ++p)
        if (p < split_parts) v[p] = ld_cluster_f4(peer[p] + off);
      float4 sum = v[0];  // parts added in K order
#pragma unroll
      for (int p = 1; p < 8; ++p)
        if (p < split_parts) sum.x += v[p].x, sum.y += v[p].y, sum.z += v[p].z, sum.w += v[p].w;
      const int r = m0 + rl, c = n0 + cl;
      if (r < M) {
        float *d = C + (int64_t)r * ldc + c;
        if (c_vec && c + 3 < N) {
          *reinterpret_cast<float4 *>(d) = sum;
        } else {
          if (c < N) d[0] = sum.x;
          if (c + 1 < N) d[1] = sum.y;
          if (c + 2 < N) d[2] = sum.z;
          if (c + 3 < N) d[3] = sum.w;
        }
      }
    }
    __syncwarp();
    cluster_sync();  // no CTA leaves while a peer may still read its partial
    return;
  }

  if (split) {
    const int64_t slot = (int64_t)(tile - split_first) * split_parts;
    float *mine = work + (slot + part) * (BM * BN);
#pragma unroll
    for (int i = 0; i < TM; ++i) {
      const int rl = row_of(i);
#pragma unroll
      for (int h = 0; h < TN / 4; ++h)
        *reinterpret_cast<float4 *>(mine + rl * BN + col_of(h)) =
            make_float4(acc[i][h * 4], acc[i][h * 4 + 1], acc[i][h * 4 + 2], acc[i][h * 4 + 3]);
    }
    __threadfence();
    __syncthreads();
    __shared__ int last;
    if (threadIdx.x == 0)
      last = atomicAdd(&counters[tile - split_first], 1u) == (unsigned)(split_parts - 1);
    __syncthreads();
    if (!last) return;
    __threadfence();
    // Sum the parts in part order and write C.  The accumulators are dead
    // here, so the tile is walked as a flat array of float4s (consecutive
    // threads, consecutive columns): a batch of CH float4s per thread is
    // loaded from one part at a time, all in flight together, so each part
    // costs one L2 round trip per batch.  -0 + x is x exactly, so the first
    // add copies part 0.
    const float *parts0 = work + slot * (BM * BN);
    constexpr int Q = BN / 4;                      // float4s per tile row
    constexpr int V = BM * Q / THREADS;            // float4s per thread
    constexpr int CH = V < 16 ? V : 16;
    static_assert(V % CH == 0, "whole batches");
#pragma unroll 1
    for (int c0 = 0; c0 < V; c0 += CH) {
      float4 sum[CH];
#pragma unroll
      for (int q = 0; q < CH; ++q) sum[q] = make_float4(-0.f, -0.f, -0.f, -0.f);
      for (int p = 0; p < split_parts; ++p) {
        const float4 *src = reinterpret_cast<const float4 *>(parts0 + (int64_t)p * (BM * BN));
#pragma unroll
        for (int q = 0; q < CH; ++q) {
          const float4 v = __ldcg(src + (c0 + q) * THREADS + tid);
          sum[q].x += v.x, sum[q].y += v.y, sum[q].z += v.z, sum[q].w += v.w;
        }
      }
#pragma unroll
      for (int q = 0; q < CH; ++q) {
        const int e = (c0 + q) * THREADS + tid;
        const int r = m0 + e / Q, c = n0 + (e % Q) * 4;
        if (r >= M) continue;
        float *d = C + (int64_t)r * ldc + c;
        if (c_vec && c + 3 < N) {
          *reinterpret_cast<float4 *>(d) = sum[q];
        } else {
          if (c < N) d[0] = sum[q].x;
          if (c + 1 < N) d[1] = sum[q].y;
          if (c + 2 < N) d[2] = sum[q].z;
          if (c + 3 < N) d[3] = sum[q].w;
        }
      }
    }
    if (threadIdx.x == 0) counters[tile - split_first] = 0u;
    return;
  }

#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int r = m0 + row_of(i);
    if (r >= M) continue;
    float *crow = C + (int64_t)r * ldc;
#pragma unroll
    for (int h = 0; h < TN / 4; ++h) {
      const int c = n0 + col_of(h);
      const float *w = &acc[i][h * 4];
      if (c_vec && c + 3 < N) {
        *reinterpret_cast<float4 *>(crow + c) = make_float4(w[0], w[1], w[2], w[3]);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (c + j < N) crow[c + j] = w[j];
      }
    }
  }
}

// Block tile BM x BN x BK, WM x WN warps, each warp a (BM/WM) x (BN/WN) tile
// with its 32 lanes arranged LM x LN; every thread owns TM x TN outputs made
// of 4 x 4 blocks spaced LM*4 rows and LN*4 columns apart, so that each
// 128-bit fragment load of a warp reads one contiguous line.
template <int BM_, int BN_, int BK_, int WM_, int WN_, int LM_, int MIN_BLOCKS_>
struct SimtCfg {
  static constexpr int BM = BM_, BN = BN_, BK = BK_, WM = WM_, WN = WN_;
  static constexpr int LM = LM_, LN = 32 / LM_;
  static constexpr int AROW = BM + 4;                   // floats per As row (+4 pad)
  static constexpr int BROW = BN + 4;                   // floats per Bs row (+4 pad)
  static constexpr int THREADS = WM * WN * 32;
  static constexpr int TM = BM / WM / LM, TN = BN / WN / LN;
  static constexpr int MIN_BLOCKS = MIN_BLOCKS_;
  static constexpr int A_VECS = BM * BK / 4 / THREADS;  // float4 loads of A per thread
  static constexpr int B_VECS = BK * BN / 4 / THREADS;  // float4 loads of B per thread
  static_assert(TM % 4 == 0 && TN % 4 == 0, "thread tile is made of 4x4 blocks");
  static_assert(A_VECS >= 1 && B_VECS >= 1, "every thread loads A and B");
  static_assert(BM * BK % (4 * THREADS) == 0 && BK * BN % (4 * THREADS) == 0, "even loads");
  static constexpr int SMEM_BYTES = 2 * BK * AROW * 4 + 2 * BK * BROW * 4;  // two buffers
  // Cluster K-split: a part's BM x BN partial tile parked in shared memory,
  // rows padded by 4 floats.
  static constexpr int PART_PITCH = BN + 4;
  static constexpr int PART_BYTES = BM * PART_PITCH * 4;
  static constexpr int SMEM_CLUSTER = SMEM_BYTES > PART_BYTES ? SMEM_BYTES : PART_BYTES;
};

// AT: A is stored K x M (op(A) = A^T); BT: B is stored N x K (op(B) = B^T).
// Shared memory always holds A k-major and B n-major; a transposed A lands
// there with plain 128-bit stores, a transposed B with transposing scalar
// stores (the row pads keep both conflict-free).
template <class G, bool kVec, bool AT, bool BT>
__global__ void __launch_bounds__(G::THREADS, G::MIN_BLOCKS)
    sgemm_simt_kernel(int M, int N, int K, const float *__restrict__ A, int64_t lda,
                      const float *__restrict__ B, int64_t ldb, float *__restrict__ C,
                      int64_t ldc, int c_vec, int split_first, int split_parts,
                      float *__restrict__ work, unsigned int *__restrict__ counters,
                      int cluster_parts) {
  constexpr int BM = G::BM, BN = G::BN, BK = G::BK, TM = G::TM, TN = G::TN;
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel on the stream has completed
  // A stored k-major (transposed): a 128-bit load gives 4 consecutive rows.
  extern __shared__ float4 simt_smem[];
  auto As = reinterpret_cast<float(*)[BK][G::AROW]>(simt_smem);
  auto Bs = reinterpret_cast<float(*)[BK][G::BROW]>(reinterpret_cast<float *>(simt_smem) +
                                                      2 * BK * G::AROW);

  // ---- work unit -> (tile, K range).  Blocks below split_first each own a
  // whole tile; the tiles from split_first on (the last, partial wave) are
  // each split along K into split_parts parts, one block per part.
  const int KT = (K + BK - 1) / BK;
  const bool split = split_parts > 1 && (int)blockIdx.x >= split_first;
  int tile = blockIdx.x, part = 0, kt_begin = 0, kt_end = KT;
  if (split) {
    const int u = blockIdx.x - split_first;
    tile = split_first + u / split_parts;
    part = u % split_parts;
    const int per = (KT + split_parts - 1) / split_parts;
    kt_begin = min(KT, part * per);
    kt_end = min(KT, kt_begin + per);
  }

  // ---- grouped raster: tile id -> (tile row, tile col)
  const int tiles_m = (M + BM - 1) / BM;
  const int tiles_n = (N + BN - 1) / BN;
  const int per_group = kGroupM * tiles_n;
  const int group = tile / per_group;
  const int first_m = group * kGroupM;
  const int gsize = min(tiles_m - first_m, kGroupM);
  const int in_group = tile - group * per_group;
  const int m0 = (first_m + in_group % gsize) * BM;
  const int n0 = (in_group / gsize) * BN;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int wm = warp / G::WN, wn = warp % G::WN;
  const int lm = lane / G::LN, ln = lane % G::LN;
  const int row_base = wm * (BM / G::WM) + lm * 4;   // + c * LM * 4, c < TM / 4
  const int col_base = wn * (BN / G::WN) + ln * 4;   // + c * LN * 4, c < TN / 4

#if DGEMM_SIMT_FFMA2
  // Packed accumulators: acc2[i][h] = {acc[i][2h], acc[i][2h+1]} for the
  // two-wide fma.rn.f32x2 (one instruction per two multiply-adds).
  uint64_t acc2[TM][TN / 2];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int h = 0; h < TN / 2; ++h) acc2[i][h] = 0ull;  // two +0.0f
#else
  float acc[TM][TN];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
#endif

  // global -> shared assignment, 128-bit vectors along each stored row:
  // A: BM rows x BK/4 (stored M x K) or BK rows x BM/4 (stored K x M);
  // B: BK rows x BN/4 (stored K x N) or BN rows x BK/4 (stored N x K).
  float4 ra[G::A_VECS], rb[G::B_VECS];
  auto load_tiles = [&](int k0) {
#pragma unroll
    for (int v = 0; v < G::A_VECS; ++v) {
      const int e = tid + v * G::THREADS;
      if constexpr (AT)
        ra[v] = load4<kVec>(A, lda, k0 + e / (BM / 4), m0 + (e % (BM / 4)) * 4, K, M);
      else
        ra[v] = load4<kVec>(A, lda, m0 + e / (BK / 4), k0 + (e % (BK / 4)) * 4, M, K);
    }
#pragma unroll
    for (int v = 0; v < G::B_VECS; ++v) {
      const int e = tid + v * G::THREADS;
      if constexpr (BT)
        rb[v] = load4<kVec>(B, ldb, n0 + e / (BK / 4), k0 + (e % (BK / 4)) * 4, N, K);
      else
        rb[v] = load4<kVec>(B, ldb, k0 + e / (BN / 4), n0 + (e % (BN / 4)) * 4, K, N);
    }
  };
  auto store_tiles = [&](int buf) {
#pragma unroll
    for (int v = 0; v < G::A_VECS; ++v) {
      const int e = tid + v * G::THREADS;
      if constexpr (AT) {
        *reinterpret_cast<float4 *>(&As[buf][e / (BM / 4)][(e % (BM / 4)) * 4]) = ra[v];
      } else {
        const int r = e / (BK / 4), c = (e % (BK / 4)) * 4;
        As[buf][c + 0][r] = ra[v].x;
        As[buf][c + 1][r] = ra[v].y;
        As[buf][c + 2][r] = ra[v].z;
        As[buf][c + 3][r] = ra[v].w;
      }
    }
#pragma unroll
    for (int v = 0; v < G::B_VECS; ++v) {
      const int e = tid + v * G::THREADS;
      if constexpr (BT) {
        const int r = e / (BK / 4), c = (e % (BK / 4)) * 4;
        Bs[buf][c + 0][r] = rb[v].x;
        Bs[buf][c + 1][r] = rb[v].y;
        Bs[buf][c + 2][r] = rb[v].z;
        Bs[buf][c + 3][r] = rb[v].w;
      } else {
        *reinterpret_cast<float4 *>(&Bs[buf][e / (BN / 4)][(e % (BN / 4)) * 4]) = rb[v];
      }
    }
  };

  load_tiles(kt_begin * BK);
  store_tiles(0);
  __syncthreads();

  for (int kt = kt_begin; kt < kt_end; ++kt) {
    const int cur = (kt - kt_begin) & 1;
    const bool more = kt + 1 < kt_end;
    if (more) load_tiles((kt + 1) * BK);
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[TM], b[TN];
#pragma unroll
      for (int c = 0; c < TM / 4; ++c) {
        const float4 v =
            *reinterpret_cast<const float4 *>(&As[cur][kk][row_base + c * G::LM * 4]);
        a[4 * c] = v.x, a[4 * c + 1] = v.y, a[4 * c + 2] = v.z, a[4 * c + 3] = v.w;
      }
#pragma unroll
      for (int c = 0; c < TN / 4; ++c) {
        const float4 v =
            *reinterpret_cast<const float4 *>(&Bs[cur][kk][col_base + c * G::LN * 4]);
        b[4 * c] = v.x, b[4 * c + 1] = v.y, b[4 * c + 2] = v.z, b[4 * c + 3] = v.w;
      }
#if DGEMM_SIMT_FFMA2
      // {a_i, a_i} x {b_2h, b_2h+1} + acc2[i][h]: a_i duplicated into a
      // register pair (one move per row), b pairs straight from the 128-bit
      // shared loads.
#pragma unroll
      for (int i = 0; i < TM; ++i) {
        uint64_t aa;
        asm("mov.b64 %0, {%1, %1};" : "=l"(aa) : "f"(a[i]));
#pragma unroll
        for (int h = 0; h < TN / 2; ++h) {
          uint64_t bb;
          asm("mov.b64 %0, {%1, %2};" : "=l"(bb) : "f"(b[2 * h]), "f"(b[2 * h + 1]));
          asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2[i][h]) : "l"(aa), "l"(bb));
        }
      }
#else
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
#endif
    }
    if (more) store_tiles(cur ^ 1);
    __syncthreads();
  }
#if DGEMM_SIMT_FFMA2
  float acc[TM][TN];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int h = 0; h < TN / 2; ++h)
      asm("mov.b64 {%0, %1}, %2;" : "=f"(acc[i][2 * h]), "=f"(acc[i][2 * h + 1]) : "l"(acc2[i][h]));
#endif
  finish_tile<BM, BN, G::THREADS, TM, TN, G::PART_PITCH>(
      acc, [&](int i) { return row_base + (i / 4) * G::LM * 4 + (i % 4); },
      [&](int h) { return col_base + h * G::LN * 4; }, reinterpret_cast<float *>(simt_smem), M, N,
      C, ldc, c_vec, m0, n0, split, tile, part, split_first, split_parts, work, counters,
      cluster_parts);
}

// ---------------------------------------------------------------------------
// TMA ring kernel.  Block tile BM x BN, k-block BK = 32 (one 128-byte row of
// A), WM x WN warps of 64 x (4 * TN) outputs, lanes 8 (lm) x 4 (ln), an
// 8 x TN register tile per thread:
//  * row i (i < 8) of a thread is tile row wm * 64 + lm + 8 i for A stored
//    M x K (A's shared tile [m][k] in 128B-swizzled rows: 16-byte chunk q of
//    row r sits at chunk q ^ (r & 7), so the eight rows lm + 8 i of a warp's
//    load are in eight different bank groups), or wm * 64 + 4 lm + 32 (i / 4)
//    + i % 4 for A stored K x M (shared tile [k][m], four consecutive rows
//    per 128-bit load);
//  * column block h (h < TN / 4) is tile columns wn * 4 TN + 4 ln + 16 h ..
//    + 3 of B's shared tile [k][n].
template <int BM_, int BN_, int WM_, int WN_, int TN_, int STAGES_, int MIN_BLOCKS_>
struct RingCfg {
  static constexpr int BM = BM_, BN = BN_, BK = 32, WM = WM_, WN = WN_;
  static constexpr int LM = 8, LN = 4, TM = 8, TN = TN_;
  static constexpr int THREADS = WM * WN * 32, NWARPS = WM * WN;
  static constexpr int WTM = LM * TM, WTN = LN * TN;  // warp tile
  static_assert(WM * WTM == BM && WN * WTN == BN, "the warps tile the block");
  static_assert(TN % 4 == 0, "column blocks of 4");
  static constexpr int STAGES = STAGES_, MIN_BLOCKS = MIN_BLOCKS_;
  // A stage is refilled by the warp that finishes k-block i + 1 of the CTA's
  // range, once every warp is done with k-block i (the stage's next load is
  // then STAGES - 2 k-blocks ahead of the fastest warp).
  static constexpr int LAG = 2;
  static_assert(STAGES >= 3, "at least one k-block of look-ahead");
  static constexpr int A_BYTES = BM * BK * 4, B_BYTES = BK * BN * 4;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static_assert(A_BYTES % 1024 == 0 && STAGE_BYTES % 1024 == 0, "swizzle atoms stay aligned");
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
  // Cluster K-split: the part's partial tile parked over the idle ring.
  static constexpr int PART_PITCH = BN + 4;
  static constexpr int PART_BYTES = BM * PART_PITCH * 4;
  static constexpr int DATA_BYTES = RING_BYTES > PART_BYTES ? RING_BYTES : PART_BYTES;
  // full and empty barriers, the test-stall barrier, the count of issued
  // k-blocks, the abort flag
  static constexpr int TAIL_BYTES = (2 * STAGES + 1) * 8 + 8;
  static constexpr int SMEM_BYTES = 1024 + DATA_BYTES + TAIL_BYTES;  // 1024: alignment slack
};

// Watchdog site codes of the ring kernel (distinct from the tensor-core
// kernels' codes).
enum : int {
  kSiteRingFull = 0x81,       // a warp's wait for a stage's copy
  kSiteRingEmpty = 0x82,      // a refill's wait for the warps to release a stage
  kSiteRingDrain = 0x83,      // the wait for copies still in flight after an abort
  kSiteRingTestStall = 0x84,  // DGEMM_SIMT_TEST_STALL: warp 0 of CTA 0's test wait ran out
};

template <class G, bool AT>
__global__ void __launch_bounds__(G::THREADS, G::MIN_BLOCKS)
    sgemm_ring_kernel(const __grid_constant__ CUtensorMap tmap_a,
                      const __grid_constant__ CUtensorMap tmap_b, int M, int N, int K,
                      float *__restrict__ C, int64_t ldc, int c_vec, int split_first,
                      int split_parts, float *__restrict__ work,
                      unsigned int *__restrict__ counters, int cluster_parts, int *watchdog,
                      int stall) {
  constexpr int BM = G::BM, BN = G::BN, BK = G::BK, TM = G::TM, TN = G::TN, S = G::STAGES;
  pdl_launch_dependents();
  extern __shared__ uint8_t ring_smem_raw[];
  const uint32_t raw = smem_u32(ring_smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128B swizzle atoms: 1024-byte aligned
  uint8_t *smem = ring_smem_raw + (base - raw);
  const uint32_t bars = base + G::DATA_BYTES;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
  const uint32_t stall_bar = bars + 8u * (2 * S);  // nothing ever arrives here
  int *issued = reinterpret_cast<int *>(smem + G::DATA_BYTES + 8 * (2 * S + 1));
  volatile int *abort_flag = issued + 1;

  // ---- work unit -> (tile, K range), as in sgemm_simt_kernel
  const int KT = (K + BK - 1) / BK;
  const bool split = split_parts > 1 && (int)blockIdx.x >= split_first;
  int tile = blockIdx.x, part = 0, kt_begin = 0, kt_end = KT;
  if (split) {
    const int u = blockIdx.x - split_first;
    tile = split_first + u / split_parts;
    part = u % split_parts;
    const int per = (KT + split_parts - 1) / split_parts;
    kt_begin = min(KT, part * per);
    kt_end = min(KT, kt_begin + per);
  }
  const int nkb = kt_end - kt_begin;
  const int tiles_m = (M + BM - 1) / BM;
  const int tiles_n = (N + BN - 1) / BN;
  const int per_group = kGroupM * tiles_n;
  const int group = tile / per_group;
  const int first_m = group * kGroupM;
  const int gsize = min(tiles_m - first_m, kGroupM);
  const int in_group = tile - group * per_group;
  const int m0 = (first_m + in_group % gsize) * BM;
  const int n0 = (in_group / gsize) * BN;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), G::NWARPS);
    }
    mbar_init(stall_bar, 1);
    *issued = 0;
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
  }
  __syncthreads();
  pdl_wait();  // set-up done; the previous kernel on the stream has completed

  // k-block i of this CTA's range -> stage i % S.  The copy's bytes are
  // announced before it is issued; boxes reaching past M, N or K are
  // zero-filled and still count in full.
  auto issue = [&](int i) {
    const int s = i % S;
    const int k0 = (kt_begin + i) * BK;
    const uint32_t dst = base + (uint32_t)(s * G::STAGE_BYTES);
    mbar_arrive_expect_tx(full_bar(s), (uint32_t)G::STAGE_BYTES);
    if constexpr (AT)
      tma_load_2d(dst, &tmap_a, full_bar(s), m0, k0);
    else
      tma_load_2d(dst, &tmap_a, full_bar(s), k0, m0);
    tma_load_2d(dst + G::A_BYTES, &tmap_b, full_bar(s), n0, k0);
    atomicAdd(issued, 1);
  };
  if (tid == 0)
    for (int i = 0; i < nkb && i < S; ++i) issue(i);

  const int wm = warp / G::WN, wn = warp % G::WN;
  const int lm = lane >> 2, ln = lane & 3;
  auto row_of = [&](int i) {
    return AT ? wm * G::WTM + lm * 4 + (i >> 2) * 32 + (i & 3) : wm * G::WTM + lm + 8 * i;
  };
  auto col_of = [&](int h) { return wn * G::WTN + ln * 4 + 16 * h; };
  // byte offsets within a stage
  const uint32_t a_thr = AT ? (uint32_t)((wm * G::WTM + lm * 4) * 4)
                            : (uint32_t)((wm * G::WTM + lm) * (BK * 4));
  const uint32_t b_thr = (uint32_t)(G::A_BYTES + (wn * G::WTN + ln * 4) * 4);
  auto lds4 = [&](uint32_t off) { return *reinterpret_cast<const float4 *>(smem + off); };

  uint64_t acc2[TM][TN / 2];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int h = 0; h < TN / 2; ++h) acc2[i][h] = 0ull;  // two +0.0f

  // acc[i][2h .. 2h+1] += {a_i, a_i} x {b_2h, b_2h+1}: all a_i duplicated
  // first, then the products column pair by column pair.
  auto fma_block = [&](const float (&a)[TM], const float4 (&b4)[TN / 4]) {
    uint64_t aa[TM], bb[TN / 2];
#pragma unroll
    for (int i = 0; i < TM; ++i) asm("mov.b64 %0, {%1, %1};" : "=l"(aa[i]) : "f"(a[i]));
#pragma unroll
    for (int h = 0; h < TN / 4; ++h) {
      asm("mov.b64 %0, {%1, %2};" : "=l"(bb[2 * h]) : "f"(b4[h].x), "f"(b4[h].y));
      asm("mov.b64 %0, {%1, %2};" : "=l"(bb[2 * h + 1]) : "f"(b4[h].z), "f"(b4[h].w));
    }
#pragma unroll
    for (int h = 0; h < TN / 2; ++h)
#pragma unroll
      for (int i = 0; i < TM; ++i)
        asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2[i][h]) : "l"(aa[i]), "l"(bb[h]));
  };
  auto comp = [](const float4 &v, int t) { return t == 0 ? v.x : t == 1 ? v.y : t == 2 ? v.z : v.w; };

  if (stall && blockIdx.x == 0 && warp == 0) {
    // Test hook: wait on a barrier that nothing arrives at, so that the
    // bounded wait runs out and the abort path below runs for real.
    const bool got = mbar_wait(stall_bar, 0);
    if (!__all_sync(0xffffffffu, got) && lane == 0) {
      atomicCAS(watchdog, 0, kSiteRingTestStall);
      *abort_flag = 1;
    }
  }
  for (int it = 0; it < nkb && !(stall && blockIdx.x == 0 && warp == 0); ++it) {
    const int s = it % S;
    const uint32_t ph = (uint32_t)(it / S) & 1u;
    bool got = mbar_try_wait(full_bar(s), ph) || (!*abort_flag && mbar_wait(full_bar(s), ph));
    if (!__all_sync(0xffffffffu, got)) {
      if (lane == 0 && !*abort_flag) {
        atomicCAS(watchdog, 0, kSiteRingFull);
        *abort_flag = 1;
      }
      break;
    }
    const uint32_t st = (uint32_t)(s * G::STAGE_BYTES);
    if constexpr (!AT) {
#pragma unroll
      for (int q = 0; q < BK / 4; ++q) {
        float4 a4[TM];
#pragma unroll
        for (int i = 0; i < TM; ++i)
          a4[i] = lds4(st + a_thr + i * 8 * (BK * 4) + (((uint32_t)q ^ (uint32_t)lm) << 4));
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          float4 b4[TN / 4];
#pragma unroll
          for (int h = 0; h < TN / 4; ++h) b4[h] = lds4(st + b_thr + (4 * q + t) * (BN * 4) + 64 * h);
          float a[TM];
#pragma unroll
          for (int i = 0; i < TM; ++i) a[i] = comp(a4[i], t);
          fma_block(a, b4);
        }
      }
    } else {
#pragma unroll
      for (int kk = 0; kk < BK; ++kk) {
        float4 a4[TM / 4], b4[TN / 4];
#pragma unroll
        for (int c = 0; c < TM / 4; ++c) a4[c] = lds4(st + a_thr + kk * (BM * 4) + c * 128);
#pragma unroll
        for (int h = 0; h < TN / 4; ++h) b4[h] = lds4(st + b_thr + kk * (BN * 4) + 64 * h);
        float a[TM];
#pragma unroll
        for (int i = 0; i < TM; ++i) a[i] = comp(a4[i >> 2], i & 3);
        fma_block(a, b4);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_bar(s));
    // Refill: the stage of k-block it + 1 - LAG gets k-block it + 1 - LAG + S
    // once every warp has released it; the refilling lane rotates.
    if (lane == 0 && warp == it % G::NWARPS) {
      const int done = it + 1 - G::LAG;
      if (done >= 0 && done + S < nkb) {
        const int ds = done % S;
        const uint32_t dph = (uint32_t)(done / S) & 1u;
        if (mbar_try_wait(empty_bar(ds), dph) || (!*abort_flag && mbar_wait(empty_bar(ds), dph))) {
          issue(done + S);
        } else if (!*abort_flag) {
          atomicCAS(watchdog, 0, kSiteRingEmpty);
          *abort_flag = 1;
        }
      }
    }
  }
  __syncthreads();
  if (*abort_flag) {
    // Only after an abort can copies still be in flight: at most the last S
    // issued, one per stage.  Wait (bounded) for them, so that no TMA write
    // lands after the CTA has left or while the ring is reused below.
    if (tid == 0) {
      const int n = *issued;
      for (int i = n - 1; i >= 0 && i >= n - S; --i)
        if (!mbar_wait(full_bar(i % S), (uint32_t)(i / S) & 1u)) atomicCAS(watchdog, 0, kSiteRingDrain);
    }
    __syncthreads();
  }

  float acc[TM][TN];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int h = 0; h < TN / 2; ++h)
      asm("mov.b64 {%0, %1}, %2;" : "=f"(acc[i][2 * h]), "=f"(acc[i][2 * h + 1]) : "l"(acc2[i][h]));
  finish_tile<BM, BN, G::THREADS, TM, TN, G::PART_PITCH>(
      acc, row_of, col_of, reinterpret_cast<float *>(smem), M, N, C, ldc, c_vec, m0, n0, split,
      tile, part, split_first, split_parts, work, counters, cluster_parts);
}

// Clusters of `size` CTAs of `kern` (threads, smem bytes each) that can be
// resident at once on device `dev`; 0 if none.  Cached per kernel, device
// and size.
int simt_active_clusters(const void *kern, int threads, int smem, int dev, int size) {
  static std::mutex mu;
  static std::map<std::tuple<const void *, int, int>, int> cache;
  const auto key = std::make_tuple(kern, dev, size);
  {
    std::lock_guard<std::mutex> lock(mu);
    const auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)size, 1, 1);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)size;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 0) {
    cudaGetLastError();  // not sticky; treat as "does not fit"
    n = 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = n;
  return n;
}

// The grid of one SIMT launch of `kern` (threads per CTA, min_blocks CTAs
// per SM, bm x bn tiles, KT k-blocks):
//  * whole tiles, one CTA each;
//  * when the tiles leave a last wave at most half full, that wave's tiles
//    split along K into up to 8 parts of at least 4 k-blocks, one CTA each,
//    partials through scratch (finish_tile);
//  * when every tile is split (a small problem) and the parts' clusters are
//    all resident at once, each tile's parts as one thread-block cluster,
//    partials through distributed shared memory: no scratch, no second pass
//    (a cluster that waits for a second wave doubles the time).
// launch(grid, cluster, split_first, parts, work, counters, cluster_parts)
// enqueues the kernel.
template <class Launch>
cudaError_t run_simt_grid(const void *kern, int threads, int smem_cluster, int min_blocks,
                          int64_t tiles, int KT, int bm, int bn, int num_sms, cudaStream_t stream,
                          Launch launch) {
  const int64_t slots = (int64_t)num_sms * min_blocks;
  const int64_t rem = slots > 0 ? tiles % slots : 0;
  int parts = 1;
  if (rem > 0) parts = (int)(slots / rem < 8 ? slots / rem : 8);
  while (parts > 1 && KT < 4 * parts) --parts;  // keep at least 4 k-blocks per part
  if (parts > 1 && rem == tiles) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    for (int p = parts; p >= 2; --p)
      if (tiles <= simt_active_clusters(kern, threads, smem_cluster, dev, p))
        return launch(tiles * p, p, (int64_t)0, p, static_cast<float *>(nullptr),
                      static_cast<unsigned int *>(nullptr), 1);
  }
  if (parts <= 1)
    return launch(tiles, 1, tiles, 1, static_cast<float *>(nullptr),
                  static_cast<unsigned int *>(nullptr), 0);
  const int64_t split_first = tiles - rem;
  const int64_t grid = split_first + rem * parts;
  const size_t work_bytes = (size_t)(rem * parts) * bm * bn * sizeof(float);
  void *scratch = nullptr;
  cudaError_t e = scratch_alloc(&scratch, work_bytes + (size_t)rem * sizeof(unsigned int), stream);
  if (e != cudaSuccess) return e;
  float *work = static_cast<float *>(scratch);
  unsigned int *counters =
      reinterpret_cast<unsigned int *>(static_cast<char *>(scratch) + work_bytes);
  e = cudaMemsetAsync(counters, 0, (size_t)rem * sizeof(unsigned int), stream);
  if (e == cudaSuccess) e = launch(grid, 1, split_first, parts, work, counters, 0);
  const cudaError_t e2 = scratch_free(scratch, stream);
  return e == cudaSuccess ? e2 : e;
}

// Opt `kern` in to `smem` bytes of dynamic shared memory (once per device).
template <class Kern>
cudaError_t allow_smem(Kern kern, int smem, std::atomic<bool> (&done)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev].store(true, std::memory_order_release);
  return e;
}

template <class G, bool AT, bool BT>
cudaError_t launch_simt_cfg(int M, int N, int K, const float *A, int64_t lda, const float *B,
                            int64_t ldb, float *C, int64_t ldc, bool ab_vec, bool c_vec,
                            int num_sms, cudaStream_t stream) {
  const int64_t tiles = (int64_t)((M + G::BM - 1) / G::BM) * ((N + G::BN - 1) / G::BN);
  if (tiles > 0x3fffffff) return cudaErrorInvalidValue;
  auto kern = ab_vec ? sgemm_simt_kernel<G, true, AT, BT> : sgemm_simt_kernel<G, false, AT, BT>;
  static std::atomic<bool> done[2][64] = {};
  cudaError_t e = allow_smem(kern, G::SMEM_CLUSTER, done[ab_vec]);
  if (e != cudaSuccess) return e;
  const int KT = (K + G::BK - 1) / G::BK;
  return run_simt_grid(
      reinterpret_cast<const void *>(kern), G::THREADS, G::SMEM_CLUSTER, G::MIN_BLOCKS, tiles, KT,
      G::BM, G::BN, num_sms, stream,
      [&](int64_t grid, int cluster, int64_t split_first, int parts, float *work,
          unsigned int *counters, int cparts) {
        return launch_kernel(kern, dim3((unsigned)grid), dim3(G::THREADS),
                             cluster > 1 ? G::SMEM_CLUSTER : G::SMEM_BYTES, stream,
                             (unsigned)cluster, M, N, K, A, lda, B, ldb, C, ldc, c_vec ? 1 : 0,
                             (int)split_first, parts, work, counters, cparts);
      });
}

// DGEMM_SIMT_TEST_STALL=1 makes warp 0 of the ring kernel's first CTA wait on
// a barrier that nothing arrives at: the wait runs out after ~2 s and the
// kernel takes its abort path (watchdog site code, drained copies,
// incomplete C).  For the failure-detection test only; read at every launch.
[[maybe_unused]] int simt_test_stall() {
  const char *e = getenv("DGEMM_SIMT_TEST_STALL");
  return (e && e[0] == '1') ? 1 : 0;
}

// The TMA ring kernel for A stored M x K (AT = false) or K x M and B stored
// K x N, both with 16-byte aligned rows.
template <class G, bool AT>
cudaError_t launch_ring_cfg(int M, int N, int K, const float *A, int64_t lda, const float *B,
                            int64_t ldb, float *C, int64_t ldc, bool c_vec, int num_sms,
                            cudaStream_t stream) {
  const int64_t tiles = (int64_t)((M + G::BM - 1) / G::BM) * ((N + G::BN - 1) / G::BN);
  if (tiles > 0x3fffffff) return cudaErrorInvalidValue;
  CUtensorMap ta, tb;
  const bool ok_a =
      AT ? make_map(&ta, A, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, K, M, lda, G::BM, G::BK,
                    CU_TENSOR_MAP_SWIZZLE_NONE)
         : make_map(&ta, A, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, M, K, lda, G::BK, G::BM,
                    CU_TENSOR_MAP_SWIZZLE_128B);
  const bool ok_b = make_map(&tb, B, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, K, N, ldb, G::BN, G::BK,
                             CU_TENSOR_MAP_SWIZZLE_NONE);
  if (!ok_a || !ok_b) return cudaErrorInvalidValue;
  int *wd = watchdog_address();
  if (wd == nullptr) return cudaErrorInvalidSymbol;
  auto kern = sgemm_ring_kernel<G, AT>;
  static std::atomic<bool> done[64] = {};
  cudaError_t e = allow_smem(kern, G::SMEM_BYTES, done);
  if (e != cudaSuccess) return e;
  const int KT = (K + G::BK - 1) / G::BK;
  return run_simt_grid(
      reinterpret_cast<const void *>(kern), G::THREADS, G::SMEM_BYTES, G::MIN_BLOCKS, tiles, KT,
      G::BM, G::BN, num_sms, stream,
      [&](int64_t grid, int cluster, int64_t split_first, int parts, float *work,
          unsigned int *counters, int cparts) {
        return launch_kernel(kern, dim3((unsigned)grid), dim3(G::THREADS), G::SMEM_BYTES, stream,
                             (unsigned)cluster, ta, tb, M, N, K, C, ldc, c_vec ? 1 : 0,
                             (int)split_first, parts, work, counters, cparts, wd,
                             simt_test_stall());
      });
}

#if DGEMM_SIMT_UNIT == 0
__global__ void zero_fill_kernel(float *__restrict__ C, int M, int N, int64_t ldc) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t total = (int64_t)M * N;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = e / N, c = e - r * N;
    C[r * ldc + c] = 0.f;
  }
}
#endif

}  // namespace

// Register-staged kernel: 128 x 256 x 16 block tiles, 256 threads as 2 x 4
// warps of 64 x 64, an 8 x 16 register tile per thread, one CTA per SM.
// (DGEMM_SIMT_CFG overrides it for tuning sweeps: BM,BN,BK,WM,WN,LM,MIN_BLOCKS.)
#ifndef DGEMM_SIMT_CFG
#define DGEMM_SIMT_CFG 128, 256, 16, 2, 4, 8, 1
#endif
using SimtShipped = SimtCfg<DGEMM_SIMT_CFG>;
// Small problems: 64 x 64 x 16 block tiles, 128 threads as 2 x 2 warps of
// 32 x 32, a 4 x 8 register tile per thread, up to 4 CTAs per SM.  At 64^3
// the shipped 128 x 256 tile computes eight times the useful work on one SM.
using SimtSmall = SimtCfg<64, 64, 16, 2, 2, 8, 4>;

// The small configuration runs when the shipped tiles are fewer than an
// eighth of the SMs (the K-split cannot make up for that: 512^3 has 8 tiles)
// or when a third or more of their area would be padding (M or N well below
// a multiple of 128 or 256: 64 x 4096 x 4096 pads half of each tile).
// Measured on GB300 with the K-split on both: small ahead 1.3x at 512^3,
// 1.9x at 64 x 4096 x 4096 and 2.8x at 4096 x 64 x 4096; shipped ahead
// 1.2-1.4x at 1024^3, 1000 x 1013 x 997, 1536^3 and 256 x 8192 x 1024, and
// 1.05x at 3000 x 200 x 2000 (a quarter padding).  DGEMM_SIMT_SMALL=0 / =1
// forces one of them (read on every call, for tests and tuning).
static bool simt_use_small(int M, int N, int num_sms) {
  const char *e = getenv("DGEMM_SIMT_SMALL");
  if (e && e[0] == '0') return false;
  if (e && e[0] == '1') return true;
  const int64_t tm = (M + SimtShipped::BM - 1) / SimtShipped::BM;
  const int64_t tn = (N + SimtShipped::BN - 1) / SimtShipped::BN;
  const double padded = (double)(tm * SimtShipped::BM) * (double)(tn * SimtShipped::BN);
  return tm * tn * 8 < num_sms || padded >= 1.5 * (double)M * (double)N;
}

// TMA ring kernel: 128 x 256 tiles of 8 warps, one CTA per SM, 4 stages of
// 48 KB (RingWide), or 128 x 128 tiles of 4 warps, two CTAs per SM, 3 stages
// of 32 KB (RingSquare); 8 x 16 register tiles either way.
using RingWide = RingCfg<128, 256, 2, 4, 16, 4, 1>;
using RingSquare = RingCfg<128, 128, 2, 2, 16, 3, 2>;

// Which kernel takes operands the ring kernel can read: 1 RingWide, 2
// RingSquare, 0 the register-staged kernel.  DGEMM_SIMT_RING=0/1/2 forces
// one (read on every call, for tests and tuning).
static int simt_ring_choice() {
  const char *e = getenv("DGEMM_SIMT_RING");
  if (e && e[0] >= '0' && e[0] <= '2' && e[1] == 0) return e[0] - '0';
  return 1;
}

// This unit's operand layout.
cudaError_t DG_SIMT_UNIT_LAUNCHER(int M, int N, int K, const float *A, int64_t lda,
                                  const float *B, int64_t ldb, float *C, int64_t ldc, bool ab_vec,
                                  bool c_vec, int num_sms, cudaStream_t stream) {
  if (simt_use_small(M, N, num_sms))
    return launch_simt_cfg<SimtSmall, kUnitAT, kUnitBT>(M, N, K, A, lda, B, ldb, C, ldc, ab_vec,
                                                        c_vec, num_sms, stream);
  if constexpr (!kUnitBT) {
    // B stored K x N and both operands' rows 16-byte aligned: TMA can read them
    if (ab_vec) {
      const int ring = simt_ring_choice();
      if (ring == 1)
        return launch_ring_cfg<RingWide, kUnitAT>(M, N, K, A, lda, B, ldb, C, ldc, c_vec, num_sms,
                                                  stream);
      if (ring == 2)
        return launch_ring_cfg<RingSquare, kUnitAT>(M, N, K, A, lda, B, ldb, C, ldc, c_vec,
                                                    num_sms, stream);
    }
  }
  return launch_simt_cfg<SimtShipped, kUnitAT, kUnitBT>(M, N, K, A, lda, B, ldb, C, ldc, ab_vec,
                                                        c_vec, num_sms, stream);
}

#if DGEMM_SIMT_UNIT == 0
cudaError_t launch_simt(bool a_t, bool b_t, int M, int N, int K, const float *A, int64_t lda,
                        const float *B, int64_t ldb, float *C, int64_t ldc, bool ab_vec,
                        bool c_vec, int num_sms, cudaStream_t stream) {
  cudaError_t e;
  switch ((a_t ? 2 : 0) + (b_t ? 1 : 0)) {
    case 0:
      e = launch_simt_unit_0(M, N, K, A, lda, B, ldb, C, ldc, ab_vec, c_vec, num_sms, stream);
      break;
    case 1:
      e = launch_simt_unit_1(M, N, K, A, lda, B, ldb, C, ldc, ab_vec, c_vec, num_sms, stream);
      break;
    case 2:
      e = launch_simt_unit_2(M, N, K, A, lda, B, ldb, C, ldc, ab_vec, c_vec, num_sms, stream);
      break;
    default:
      e = launch_simt_unit_3(M, N, K, A, lda, B, ldb, C, ldc, ab_vec, c_vec, num_sms, stream);
  }
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
  const cudaError_t e =
      launch_kernel(zero_fill_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, 1, C, M, N, ldc);
  if (e == cudaSuccess) count_launch();
  return e;
}
#endif

}  // namespace dg
