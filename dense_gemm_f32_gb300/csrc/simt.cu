// simt.cu -- FP32 GEMM on the CUDA cores (FFMA), register blocked.
//
// The block-tiled, register-blocked SGEMM that "SGEMM 优化旅程" builds up in
// Levels 2-5 (shared-memory tiles, padding against bank conflicts, double
// buffering, a register tile per thread) with the structure of
// "第八课：GPU 如何完成矩阵乘法": C_tile = sum_t A_tile,t x B_tile,t (section 九),
// accumulation in registers with one store per element (section 十四),
// multi-level block / warp / thread tiling (section 十九), double-buffered
// shared memory (section 二十四), zero-fill and masked stores at the edges
// (section 二十六), padding against bank conflicts (section 二十七).
//
// Shipped shape (chosen by measurement on GB300 over tile shapes, BK, lane
// orders, unroll depths and packed fma.rn.f32x2 variants): block tile
// 128 x 256 x 16, 256 threads as 2 x 4 warps of 64 x 64, lanes 8 x 4, an
// 8 x 16 register tile per thread, one CTA per SM, the inner product in
// packed two-wide FMAs (DGEMM_SIMT_FFMA2).
// GB300 specifics that differ from the pages' kernels:
//  * A is stored transposed (k-major) in shared memory so that both operand
//    fragments are read with 128-bit shared loads; its rows carry a 4-float
//    pad that keeps the transposed stores free of bank conflicts.
//  * Every 128-bit fragment load of a warp reads one contiguous line.
//  * Global loads are 128-bit where the operand rows are 16-byte aligned
//    (template kVec); ragged edges fall back to masked scalar loads.
//  * Thread blocks walk the C tiles in groups of 8 tile rows so that panels
//    of A and B are re-read from L2 instead of HBM.
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

  if (split && cluster_parts) {
    // Every tile is split and the parts of a tile form one thread-block
    // cluster (CTA rank = part): park the partial tile in this CTA's shared
    // memory (free since the main loop's last barrier), then each CTA adds
    // one slice of the tile's rows over all parts, in part order, through
    // distributed shared memory and writes it to C.  Every thread reaches
    // both cluster barriers.
    float *park = reinterpret_cast<float *>(simt_smem);
#pragma unroll
    for (int i = 0; i < TM; ++i) {
      const int rl = row_base + (i / 4) * G::LM * 4 + (i % 4);
#pragma unroll
      for (int h = 0; h < TN / 4; ++h)
        *reinterpret_cast<float4 *>(park + rl * G::PART_PITCH + col_base + h * G::LN * 4) =
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
    for (int e = tid; e < (r1 - r0) * Q; e += G::THREADS) {
      const int rl = r0 + e / Q, cl = 4 * (e % Q);
      const uint32_t off = (uint32_t)((rl * G::PART_PITCH + cl) * 4);
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
    // Park this part's partial tile; the last part to finish sums all parts
    // in part order (so the result does not depend on which finishes last)
    // and writes C.
    const int64_t slot = (int64_t)(tile - split_first) * split_parts;
    float *mine = work + (slot + part) * (BM * BN);
#pragma unroll
    for (int i = 0; i < TM; ++i) {
      const int rl = row_base + (i / 4) * G::LM * 4 + (i % 4);
#pragma unroll
      for (int h = 0; h < TN / 4; ++h) {
        const int cl = col_base + h * G::LN * 4;
        *reinterpret_cast<float4 *>(mine + rl * BN + cl) =
            make_float4(acc[i][h * 4], acc[i][h * 4 + 1], acc[i][h * 4 + 2], acc[i][h * 4 + 3]);
      }
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
    constexpr int Q = BN / 4;                         // float4s per tile row
    constexpr int V = BM * Q / G::THREADS;            // float4s per thread
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
          const float4 v = __ldcg(src + (c0 + q) * G::THREADS + tid);
          sum[q].x += v.x, sum[q].y += v.y, sum[q].z += v.z, sum[q].w += v.w;
        }
      }
#pragma unroll
      for (int q = 0; q < CH; ++q) {
        const int e = (c0 + q) * G::THREADS + tid;
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

  // ---- epilogue: masked stores, 128-bit where C rows are 16-byte aligned
#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int r = m0 + row_base + (i / 4) * G::LM * 4 + (i % 4);
    if (r >= M) continue;
    float *crow = C + (int64_t)r * ldc;
#pragma unroll
    for (int h = 0; h < TN / 4; ++h) {
      const int c = n0 + col_base + h * G::LN * 4;
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

template <class G, bool AT, bool BT>
cudaError_t launch_simt_cfg(int M, int N, int K, const float *A, int64_t lda, const float *B,
                            int64_t ldb, float *C, int64_t ldc, bool ab_vec, bool c_vec,
                            int num_sms, cudaStream_t stream) {
  const int64_t tiles = (int64_t)((M + G::BM - 1) / G::BM) * ((N + G::BN - 1) / G::BN);
  if (tiles > 0x3fffffff) return cudaErrorInvalidValue;
  auto kern = ab_vec ? sgemm_simt_kernel<G, true, AT, BT> : sgemm_simt_kernel<G, false, AT, BT>;
  {
    // opt in to the dynamic shared memory of the cluster K-split (per device, once)
    static std::atomic<bool> done[2][64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !done[ab_vec][dev].load(std::memory_order_acquire)) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               G::SMEM_CLUSTER);
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < 64) done[ab_vec][dev].store(true, std::memory_order_release);
    }
  }
  // Tail split: when the tiles leave a last wave that is at most half full,
  // its tiles are split along K so that the wave's blocks finish sooner.
  const int64_t slots = (int64_t)num_sms * G::MIN_BLOCKS;
  const int64_t rem = tiles % slots;
  const int KT = (K + G::BK - 1) / G::BK;
  int parts = 1;
  if (rem > 0 && num_sms > 0) parts = (int)(slots / rem < 8 ? slots / rem : 8);
  while (parts > 1 && KT < 4 * parts) --parts;  // keep at least 4 k-blocks per part
  int64_t split_first = tiles, grid = tiles;
  float *work = nullptr;
  unsigned int *counters = nullptr;
  void *scratch = nullptr;
  cudaError_t e = cudaSuccess;
  int cparts = 0;  // cluster size for the all-split case, if its clusters fit at once
  if (parts > 1 && rem == tiles) {
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    for (int p = parts; p >= 2 && cparts == 0; --p)
      if (tiles <= simt_active_clusters(reinterpret_cast<const void *>(kern), G::THREADS,
                                        G::SMEM_CLUSTER, dev, p))
        cparts = p;
  }
  if (cparts > 1) {
    // Every tile is split (a small problem): the parts of a tile run as one
    // cluster and add their partials through distributed shared memory; no
    // scratch, no second pass.  Only cluster sizes whose clusters are all
    // resident at once are used: a cluster that waits for a second wave
    // doubles the time.
    parts = cparts;
    return launch_kernel(kern, dim3((unsigned)(tiles * parts)), dim3(G::THREADS), G::SMEM_CLUSTER,
                         stream, (unsigned)parts, M, N, K, A, lda, B, ldb, C, ldc, c_vec ? 1 : 0,
                         0, parts, nullptr, nullptr, 1);
  }
  if (parts > 1) {
    split_first = tiles - rem;
    grid = split_first + rem * parts;
    const size_t work_bytes = (size_t)(rem * parts) * G::BM * G::BN * sizeof(float);
    e = scratch_alloc(&scratch, work_bytes + (size_t)rem * sizeof(unsigned int), stream);
    if (e != cudaSuccess) return e;
    work = static_cast<float *>(scratch);
    counters = reinterpret_cast<unsigned int *>(static_cast<char *>(scratch) + work_bytes);
    e = cudaMemsetAsync(counters, 0, (size_t)rem * sizeof(unsigned int), stream);
  }
  if (e == cudaSuccess) {
    e = launch_kernel(kern, dim3((unsigned)grid), dim3(G::THREADS), G::SMEM_BYTES, stream, 1, M, N,
                      K, A, lda, B, ldb, C, ldc, c_vec ? 1 : 0, (int)split_first, parts, work,
                      counters, 0);
  }
  if (scratch) {
    const cudaError_t e2 = scratch_free(scratch, stream);
    if (e == cudaSuccess) e = e2;
  }
  return e;
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

// The configuration the library ships (see the variant table in the design doc).
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

// This unit's operand layout.
cudaError_t DG_SIMT_UNIT_LAUNCHER(int M, int N, int K, const float *A, int64_t lda,
                                  const float *B, int64_t ldb, float *C, int64_t ldc, bool ab_vec,
                                  bool c_vec, int num_sms, cudaStream_t stream) {
  if (simt_use_small(M, N, num_sms))
    return launch_simt_cfg<SimtSmall, kUnitAT, kUnitBT>(M, N, K, A, lda, B, ldb, C, ldc, ab_vec,
                                                        c_vec, num_sms, stream);
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
