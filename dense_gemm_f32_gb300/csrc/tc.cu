// tc.cu -- dense GEMM on the 5th-generation tensor cores (tcgen05) of sm_103a.
//
// What it computes: C = A x B, row-major, C[i][j] = sum_k A[i][k] B[k][j]
// ("第八课：GPU 如何完成矩阵乘法" section 一), by the tile decomposition
// C_tile = sum_t A_tile,t x B_tile,t of section 九, with the tensor core doing
// each tile's small matrix multiply-accumulate (section 二十一, "SGEMM 优化旅程"
// Level 6) and the data supply decoupled from the math by an asynchronous,
// multi-buffered copy pipeline (sections 二十三-二十五).
//
// Blackwell design (none of this is on the pages, which stop at WMMA):
//  * Two persistent kernels: tc_gemm_kernel, one CTA per SM walking 128 x BN
//    output tiles, and tc2_gemm_kernel, CTA pairs (clusters of 2) walking
//    256 x 256 tiles with tcgen05.mma.cta_group::2; tiles are visited in
//    groups of tile rows (L2 reuse of the A and B panels; see raster_group_m).
//  * Warp roles: TMA producer(s) (the pair kernel has one thread per
//    operand, warps 0 and 6), warp 1 issues tcgen05.mma (one thread) and owns
//    the TMEM allocation, warps 2-5 drain the accumulator (tcgen05.ld ->
//    registers -> global, or shared memory and TMA stores).  For 3xTF32 the
//    single-CTA kernel's remaining warps split each staged fp32 tile into hi
//    and lo TF32 parts; the pair kernel loads lo parts that a pre-pass wrote
//    (staging.cu: split_lo_kernel) next to the raw tiles.
//  * Operands: A (M x K, K contiguous) is K-major, B (K x N, N contiguous) is
//    MN-major (either may be stored transposed instead); they arrive by TMA
//    boxes of one 128-byte swizzle row width into 128B-swizzled shared
//    memory, the layout the MMA's shared-memory descriptors describe; an
//    MN-major operand whose extent allows it comes through a 3-D tensor map,
//    one instruction for all its column blocks.  TMA fills the out-of-range
//    part of an edge box with zeros (the pages' zero-fill of partial tiles,
//    section 二十六).
//  * Accumulators: fp32 in tensor memory, two buffers of BN columns each, so
//    the epilogue of tile i overlaps the main loop of tile i + 1.
//  * Problems with too few tiles to occupy the GPU split each tile along K
//    over a thread-block cluster of 2-8 CTAs: every CTA accumulates one K
//    range, parks its partial tile in its own shared memory, and the CTAs then
//    add the partials across the cluster (distributed shared memory) in part
//    order, each CTA writing a slice of the tile's rows to C.
//  * Every wait is bounded (ptx.cuh); on a timeout the CTA records the site in
//    the device watchdog word, drains what it issued, frees TMEM and returns.
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "kernels.h"
#include "launch.cuh"
#include "ptx.cuh"
#include "tf32_split.cuh"
#include "tmap.cuh"

// This file is compiled once per operand layout: DGEMM_TC_UNIT = 2 * AT + BT
// selects which kernels one translation unit instantiates (AT: A stored
// K x M; BT: B stored N x K), so the four layouts compile in parallel.  Unit
// 0 also holds the watchdog word and the dispatch.
#ifndef DGEMM_TC_UNIT
#define DGEMM_TC_UNIT 0
#endif
#define DG_CAT2(a, b) a##b
#define DG_CAT(a, b) DG_CAT2(a, b)
#define DG_UNIT_LAUNCHER DG_CAT(launch_tc_unit_, DGEMM_TC_UNIT)

namespace dg {

#if DGEMM_TC_UNIT == 0
// Device watchdog word: 0, or the site code of the first wait that gave up.
// Kernels of every unit receive its address as an argument.
__device__ int g_watchdog = 0;
#endif

namespace {

constexpr bool kUnitAT = (DGEMM_TC_UNIT >> 1) & 1;
// Bits of the kernels' `mn3d` argument: that MN-major operand is read through
// a 3-D tensor map, one TMA instruction per stage (else one per 128-byte
// column block; see make_map3).
constexpr int kA3d = 1, kB3d = 2;
constexpr bool kUnitBT = DGEMM_TC_UNIT & 1;

constexpr int BM = 128;

// Watchdog site codes (role * 16 + place).
enum : int {
  kSiteProducerEmpty = 0x11,
  kSiteProducerDrain = 0x12,
  kSiteMmaFull = 0x21,
  kSiteMmaAccEmpty = 0x22,
  kSiteMmaDrain = 0x23,
  kSiteEpiAccFull = 0x31,
  kSiteSplitFull = 0x41,
  kSiteTestStall = 0x24,  // DGEMM_TC_TEST_STALL: the MMA thread's test wait ran out
};

// AT: A is stored K x M (op(A) = A^T), read MN-major.  BT: B is stored N x K
// (op(B) = B^T), read K-major.  The defaults are the row-major A (K-major)
// and B (MN-major) of the plain product.
template <TcKind KIND, int BN_, bool AT_ = false, bool BT_ = false, int BUDGET_ = 196608,
          int KD_ = 1>
struct Cfg {
  static constexpr bool AT = AT_, BT = BT_;
  // 16-bit operands (BF16 or FP16, tcgen05 kind::f16) vs 32-bit (TF32 kinds)
  static constexpr bool k16 = KIND == TcKind::kBF16 || KIND == TcKind::kF16;
  // 8-bit float operands (tcgen05 kind::f8f6f4), read K-major only
  static constexpr bool k8 = KIND == TcKind::kE4M3 || KIND == TcKind::kE5M2;
  // operand format code of the instruction descriptor: F16 0, BF16 1, TF32 2
  // (kind::f8f6f4 codes: E4M3 0, E5M2 1)
  static constexpr uint32_t kFmt = KIND == TcKind::kF16    ? 0u
                                   : KIND == TcKind::kBF16 ? 1u
                                   : KIND == TcKind::kE4M3 ? 0u
                                   : KIND == TcKind::kE5M2 ? 1u
                                                           : 2u;
  static constexpr bool kSplit = KIND == TcKind::k3xTF32;
  static constexpr int BN = BN_;
  static constexpr int ES = k8 ? 1 : k16 ? 2 : 4;  // operand element bytes
  // k per stage: KD 128-byte swizzle rows (a TMA load costs a nearly fixed
  // time per box on this part, so deeper stages move more bytes per second)
  static constexpr int KD = KD_;
  static constexpr int BK = KD * 128 / ES;
  static constexpr int UMMA_K = 32 / ES;          // k per MMA instruction (32 bytes)
  static constexpr int KSTEPS = BK / UMMA_K;      // MMAs per stage (per product)
  static constexpr int BOX = 128 / ES;            // elements in one 128-byte swizzle row
  static constexpr int BOX_N = BOX;               // N columns per MN-major B box
  static constexpr int A_BYTES = BM * 128 * KD;   // 128 M x BK, either major
  static constexpr int B_BYTES = BN * 128 * KD;   // BN N x BK, either major
  // MN-major operands arrive as boxes of 128 bytes (of M or N) x BK rows;
  // K-major operands as KD boxes of 128 bytes of K x (rows), one after the
  // other (the box stride then is one such box).
  static constexpr int A_BOXES = AT ? BM / BOX : KD;
  static constexpr int A_BOX_BYTES = AT ? BK * 128 : BM * 128;
  static constexpr int B_BOXES = BT ? KD : BN / BOX;
  static constexpr int B_BOX_BYTES = BT ? BN * 128 : BK * 128;
  static constexpr int RAW_BYTES = A_BYTES + B_BYTES;               // what TMA writes
  static constexpr int STAGE_BYTES = RAW_BYTES * (kSplit ? 2 : 1);  // + lo copies
  // stages that fit the shared-memory budget: 192 KB (one CTA per SM), or
  // 96 KB for the small-problem configuration (two CTAs per SM)
  static constexpr int STAGES = BUDGET_ / STAGE_BYTES;
  static constexpr int ACC_COLS = 2 * BN;                           // two fp32 accumulators
  static constexpr int TMEM_COLS = ACC_COLS <= 32 ? 32 : ACC_COLS <= 64 ? 64
                                   : ACC_COLS <= 128 ? 128 : ACC_COLS <= 256 ? 256 : 512;
  static constexpr int kEpiWarp0 = 2, kEpiWarps = 4;
  static constexpr int kSplitWarp0 = 6, kSplitWarps = kSplit ? 4 : 0;
  static constexpr int THREADS = 32 * (2 + kEpiWarps + kSplitWarps);
  // barriers: full[S], empty[S], split[S], acc_full[2], acc_empty[2], drain
  static constexpr int NUM_BARS = 3 * STAGES + 6;  // + the test-stall barrier
  // Epilogue staging: per epilogue warp 32 rows x 16 fp32 (64-byte rows,
  // 16-byte chunks swizzled by row), so that C is written row by row.
  static constexpr int EPI_COLS = 16;
  static constexpr int EPI_WARP_BYTES = 32 * EPI_COLS * 4;
  static constexpr int EPI_BYTES = kEpiWarps * EPI_WARP_BYTES;
  static constexpr int SMEM_BYTES =
      STAGES * STAGE_BYTES + EPI_BYTES + NUM_BARS * 8 + 16 + 1024;  // +1024: align slack
  // CTAs that fit on one SM (228 KB of shared memory, 1 KB reserved per CTA;
  // 512 TMEM columns)
  static constexpr int CTAS_PER_SM =
      (2 * (SMEM_BYTES + 1024) <= 233472 && 2 * TMEM_COLS <= 512) ? 2 : 1;
  // K-split: the partial 128 x BN tile parked in the (then idle) stage area,
  // rows padded by 4 floats so that the epilogue's 16-byte row stores from 8
  // consecutive lanes fall in distinct banks.
  static constexpr int PART_PITCH = BN + 4;
  static constexpr int MAX_SPLITS = 8;  // portable cluster size

  static_assert((!AT || BM % BOX == 0) && (BT || BN % BOX == 0), "whole number of MN-major boxes");
  static_assert(KD == 1 || KD == 2, "one or two swizzle rows of K per stage");
  static_assert(BK <= 256, "an MN-major box holds at most 256 rows of K");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M = 128");
  static_assert(STAGES >= 2, "pipeline needs at least two stages");
  static_assert(ACC_COLS <= 512, "TMEM has 512 columns");
  static_assert(kSplitWarp0 == kEpiWarp0 + kEpiWarps, "split warps follow the epilogue warps");
  static_assert(BM * PART_PITCH * 4 <= STAGES * STAGE_BYTES, "partial tile fits the stage area");
  static_assert(BM * BN * 4 <= STAGES * STAGE_BYTES, "a staged C tile fits the stage area");
  static_assert(SMEM_BYTES <= 232448, "fits the 227 KB opt-in shared memory of a CTA");

  // B (MN-major) layout.  16-bit operands use the plain 128-byte swizzle
  // (16-byte chunks permuted within each 128-byte row); 32-bit MN-major
  // operands need the 128-byte swizzle with 32-byte atoms (descriptor layout
  // type 1, TMA mode SWIZZLE_128B_ATOM_32B).  Rows of a B box are contiguous
  // 128-byte lines, so the K-group stride is (group rows) x 128 B: 512 B
  // covers both a 4-row and an 8-row swizzle period for the 8-row MMA slice.
  // MN-major swizzle: 128-byte rows of 16-byte chunks for 16-bit operands,
  // 32-byte atoms for 32-bit ones (layout type 1); K-group stride 1024 / 512 B.
  static constexpr uint32_t MN_LAYOUT = k16 ? 2u : 1u;
  static constexpr uint32_t MN_SBO = k16 ? 1024u : 512u;
  static_assert(!k8 || (!AT && BT), "8-bit operands are read K-major: A as M x K, B as N x K");

  // Instruction descriptor: D fp32, A/B format, A major (bit 15: 1 = MN),
  // B major (bit 16: 1 = MN), N >> 3 at bit 17, M >> 4 at bit 24.
  static constexpr uint32_t IDESC = (1u << 4) | (kFmt << 7) | (kFmt << 10) |
                                    ((AT ? 1u : 0u) << 15) | ((BT ? 0u : 1u) << 16) |
                                    ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
};

// Shared-memory matrix descriptor of a swizzled operand tile: start address,
// leading / stride byte offsets (16-byte units), version 1, base offset 0
// (tiles are 1024-byte aligned), layout type at bits 61-63 (2 = 128-byte
// swizzle, 1 = 128-byte swizzle with 32-byte atoms).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t layout = 2u) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)layout << 61);
}

// Tile id -> (tile row, tile col): tiles are walked in groups of `group_m`
// tile rows, column by column inside a group, so that the CTAs working at the
// same time share A row panels and B column panels in L2.
// Descriptor of the k-th MMA slice (UMMA_K elements of K) of an operand tile
// at saddr: K-major tiles advance 32 bytes inside the swizzle row; MN-major
// tiles advance UMMA_K / 8 groups of 8 K-rows.  box_bytes is the distance
// between the 128-byte MN blocks of an MN-major tile.
template <class G, bool kMN>
__device__ __forceinline__ uint64_t operand_desc(uint32_t saddr, int k, uint32_t box_bytes) {
  if constexpr (kMN)
    return smem_desc(saddr + (uint32_t)(k * (G::UMMA_K / 8) * 1024), box_bytes, G::MN_SBO,
                     G::MN_LAYOUT);
  else  // K-major: 4 MMAs of 32 bytes of K per 128-byte box, boxes box_bytes apart
    return smem_desc(saddr + (uint32_t)((k >> 2) * box_bytes + (k & 3) * 32), 16, 1024);
}

__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int group_m,
                                            int &tm, int &tn) {
  const int per_group = group_m * tiles_n;
  const int group = tile / per_group;
  const int first = group * group_m;
  const int gsize = min(tiles_m - first, group_m);
  const int r = tile - group * per_group;
  tm = first + r % gsize;
  tn = r / gsize;
}

__device__ __forceinline__ void watchdog_trip(int *watchdog, int site, volatile int *abort_flag) {
  atomicCAS(watchdog, 0, site);
  *abort_flag = 1;
}

template <TcKind KIND, int BN, bool AT, bool BT, int BUDGET, int KD>
__global__ void __launch_bounds__(Cfg<KIND, BN, AT, BT, BUDGET, KD>::THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                   const __grid_constant__ CUtensorMap tmap_b, float *__restrict__ C, int M,
                   int N, int K, int64_t ldc, int c_vec, int group_m, int *watchdog,
                   int splits, int mn3d, int stall) {
  using G = Cfg<KIND, BN, AT, BT, BUDGET, KD>;
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the swizzle atoms.
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw_base);

  const uint32_t bars = base + G::STAGES * G::STAGE_BYTES + G::EPI_BYTES;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (G::STAGES + s); };
  auto split_bar = [&](int s) { return bars + 8u * (2 * G::STAGES + s); };
  auto accf_bar = [&](int b) { return bars + 8u * (3 * G::STAGES + b); };
  auto acce_bar = [&](int b) { return bars + 8u * (3 * G::STAGES + 2 + b); };
  const uint32_t drain_bar = bars + 8u * (3 * G::STAGES + 4);
  const uint32_t stall_bar = bars + 8u * (3 * G::STAGES + 5);  // nothing ever arrives here
  uint8_t *tail = smem + G::STAGES * G::STAGE_BYTES + G::EPI_BYTES + G::NUM_BARS * 8;
  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(tail);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tail + 4);

  auto a_tile = [&](int s) { return base + (uint32_t)(s * G::STAGE_BYTES); };
  auto b_tile = [&](int s) { return base + (uint32_t)(s * G::STAGE_BYTES + G::A_BYTES); };
  auto a_lo = [&](int s) { return a_tile(s) + (uint32_t)G::RAW_BYTES; };
  auto b_lo = [&](int s) { return b_tile(s) + (uint32_t)G::RAW_BYTES; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles_m = (M + BM - 1) / BM;
  const int tiles_n = (N + BN - 1) / BN;
  const int num_tiles = tiles_m * tiles_n;
  const int kblocks = (K + G::BK - 1) / G::BK;
  // Work units: each tile split along K into `splits` parts (1 = whole
  // tiles); the host picks splits so that every part has k-blocks.  With
  // splits > 1 the launch is one unit per CTA in clusters of `splits` CTAs,
  // so a cluster's CTAs hold the parts of one tile and CTA rank = part.
  const int units = num_tiles * splits;
  const int per = (kblocks + splits - 1) / splits;
  auto unit_tile = [&](int u) { return u / splits; };
  auto unit_kb0 = [&](int u) { return min(kblocks, (u % splits) * per); };
  auto unit_kb1 = [&](int u) { return min(kblocks, (u % splits) * per + per); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < G::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(split_bar(s), G::kSplitWarps > 0 ? G::kSplitWarps : 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), G::kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    mbar_init(stall_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t *>(tmem_slot)), G::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // set-up done; the previous kernel on the stream has completed

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;  // stages loaded so far (for the drain on abort)
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        int tm, tn;
        tile_coords(unit_tile(u), tiles_m, tiles_n, group_m, tm, tn);
        for (int kb = unit_kb0(u); kb < unit_kb1(u); ++kb) {
          if (!mbar_try_wait(empty_bar(stage), phase ^ 1u) &&
              (*abort_flag || !mbar_wait(empty_bar(stage), phase ^ 1u))) {
            if (!*abort_flag) watchdog_trip(watchdog, kSiteProducerEmpty, abort_flag);
            ok = false;
            break;
          }
          if (AT && (mn3d & kA3d)) {  // A stored K x M, all its column blocks at once
            tma_load_3d(a_tile(stage), &tmap_a, full_bar(stage), 0, kb * G::BK, tm * BM / G::BOX);
          } else {
#pragma unroll
            for (int j = 0; j < G::A_BOXES; ++j) {
              if constexpr (AT)  // A stored K x M: boxes of BOX columns of M x BK rows
                tma_load_2d(a_tile(stage) + j * G::A_BOX_BYTES, &tmap_a, full_bar(stage),
                            tm * BM + j * G::BOX, kb * G::BK);
              else  // A stored M x K: box j holds k-chunk j (BOX of K) x BM rows
                tma_load_2d(a_tile(stage) + j * G::A_BOX_BYTES, &tmap_a, full_bar(stage),
                            kb * G::BK + j * G::BOX, tm * BM);
            }
          }
          if (!BT && (mn3d & kB3d)) {  // B stored K x N, all its column blocks at once
            tma_load_3d(b_tile(stage), &tmap_b, full_bar(stage), 0, kb * G::BK, tn * BN / G::BOX_N);
          } else {
#pragma unroll
            for (int j = 0; j < G::B_BOXES; ++j) {
              if constexpr (BT)  // B stored N x K: box j holds k-chunk j x BN rows
                tma_load_2d(b_tile(stage) + j * G::B_BOX_BYTES, &tmap_b, full_bar(stage),
                            kb * G::BK + j * G::BOX, tn * BN);
              else
                tma_load_2d(b_tile(stage) + j * G::B_BOX_BYTES, &tmap_b, full_bar(stage),
                            tn * BN + j * G::BOX_N, kb * G::BK);
            }
          }
          // bytes announced after the copies are issued (see the pair kernel)
          mbar_arrive_expect_tx(full_bar(stage), (uint32_t)G::RAW_BYTES);
          ++issued;
          if (++stage == G::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Wait (bounded) for the copies of the last stages issued, so that no
        // TMA write lands after this CTA has left.
        int s = stage;
        uint32_t ph = phase;
        const int n = issued < G::STAGES ? issued : G::STAGES;
        for (int i = 0; i < n; ++i) {
          if (--s < 0) {
            s = G::STAGES - 1;
            ph ^= 1u;
          }
          if (!mbar_wait(full_bar(s), ph)) atomicCAS(watchdog, 0, kSiteProducerDrain);
        }
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      if (stall && blockIdx.x == 0) {
        // Test hook: wait on a barrier that nothing arrives at, so that the
        // bounded wait runs out and the abort path below runs for real.
        if (!mbar_wait(stall_bar, 0)) watchdog_trip(watchdog, kSiteTestStall, abort_flag);
        ok = false;
      }
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        if (*abort_flag || !mbar_wait(acce_bar(acc), acc_phase ^ 1u)) {
          if (!*abort_flag) watchdog_trip(watchdog, kSiteMmaAccEmpty, abort_flag);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        const int kb0 = unit_kb0(u);
        for (int kb = kb0; kb < unit_kb1(u); ++kb) {
          const uint32_t ready = G::kSplit ? split_bar(stage) : full_bar(stage);
          if (!mbar_try_wait(ready, phase) && (*abort_flag || !mbar_wait(ready, phase))) {
            if (!*abort_flag) watchdog_trip(watchdog, kSiteMmaFull, abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < G::KSTEPS; ++k) {
            const uint64_t ad = operand_desc<G, AT>(a_tile(stage), k, G::A_BOX_BYTES);
            const uint64_t bd = operand_desc<G, !BT>(b_tile(stage), k, G::B_BOX_BYTES);
            const uint32_t accum = (kb > kb0 || k > 0) ? 1u : 0u;
            if constexpr (G::kSplit) {
              const uint64_t adl = operand_desc<G, AT>(a_lo(stage), k, G::A_BOX_BYTES);
              const uint64_t bdl = operand_desc<G, !BT>(b_lo(stage), k, G::B_BOX_BYTES);
              umma_tf32(d_tmem, adl, bd, G::IDESC, accum);  // A_lo B_hi
              umma_tf32(d_tmem, ad, bdl, G::IDESC, 1u);      // A_hi B_lo
              umma_tf32(d_tmem, ad, bd, G::IDESC, 1u);       // A_hi B_hi
            } else if constexpr (G::k8) {
              umma_f8(d_tmem, ad, bd, G::IDESC, accum);
            } else if constexpr (G::k16) {
              umma_f16(d_tmem, ad, bd, G::IDESC, accum);
            } else {
              umma_tf32(d_tmem, ad, bd, G::IDESC, accum);
            }
          }
          umma_commit(empty_bar(stage));  // frees the stage once these MMAs finish
          if (++stage == G::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(accf_bar(acc));  // accumulator complete
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // Drain: wait until every MMA issued above has completed before TMEM is
      // released (on the normal path the epilogue has already seen them all).
      umma_commit(drain_bar);
      if (!mbar_wait(drain_bar, 0)) atomicCAS(watchdog, 0, kSiteMmaDrain);
    }
  } else if (warp < G::kEpiWarp0 + G::kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      int tm, tn;
      tile_coords(unit_tile(u), tiles_m, tiles_n, group_m, tm, tn);
      // every lane waits, so that each one acquires the accumulator itself
      bool ok = !*abort_flag && mbar_wait(accf_bar(acc), acc_phase);
      if (!ok && lane == 0 && !*abort_flag) watchdog_trip(watchdog, kSiteEpiAccFull, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const int trow = quarter * 32 + lane;  // this thread's accumulator row
      const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
      if (splits > 1) {
        // K-split part: park the partial tile in shared memory.  Every MMA of
        // the unit has completed (accf), so the stage area is no longer read
        // by the tensor core nor written by TMA.
        float *prow = reinterpret_cast<float *>(smem) + trow * G::PART_PITCH;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(t_row + (uint32_t)c0, r);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4 *>(prow + c0 + j) =
                make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                            __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
        }
        tc_fence_before();
        break;  // one unit per CTA
      }
      // Except for a few narrow tiles, C goes out row by row through shared
      // memory, so that every store writes whole lines: each thread writes
      // its accumulator row there (16-byte chunks, chunk q of row r at
      // q ^ (r & 7) within its group of eight, so a quarter-warp's eight
      // rows fill the 32 banks), then the warp writes C along rows: 16-byte
      // stores, four or eight lanes to a row, when C's rows start on 16-byte
      // boundaries, else one element per lane.  Columns and rows outside C
      // are skipped (warp-uniform).
      const int row0 = tm * BM + quarter * 32;  // C row of the warp's staged row 0
      const int ncols = min(BN, N - tn * BN);   // columns of this tile inside C
      if (ncols <= 64 && units <= 16) {
        // A few narrow tiles (the whole call is latency-bound): each thread
        // stores its own row straight from registers, the fewest steps.
        const int row = row0 + lane;
#pragma unroll 1
        for (int c0 = 0; row0 < M && c0 < ncols; c0 += 32) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(t_row + (uint32_t)c0, r);
          tmem_wait_ld();
          const int col = tn * BN + c0;
          float *d = C + (int64_t)row * ldc + col;
          if (row < M) {
            if (c_vec && col + 32 <= N) {
#pragma unroll
              for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4 *>(d + j) =
                    make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (col + j < N) d[j] = __uint_as_float(r[j]);
            }
          }
        }
      } else if (gridDim.x >= units) {
        // One unit per CTA: after its last MMA the stage area is idle, so
        // each warp stages all its columns (32 x BN) at once.
        float *wb = reinterpret_cast<float *>(smem) + (warp - G::kEpiWarp0) * (32 * BN);
#pragma unroll 1
        for (int c0 = 0; row0 < M && c0 < ncols; c0 += 32) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(t_row + (uint32_t)c0, r);
          tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4 *>(wb + lane * BN + c0 + ((q ^ (lane & 7)) << 2)) =
                make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                            __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
        }
        __syncwarp();
        if (row0 < M) {
          if (c_vec) {
            const int q = lane & 7;
#pragma unroll 1
            for (int c0 = 0; c0 < ncols; c0 += 32) {
              const int col = tn * BN + c0 + 4 * q;
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int rr = 4 * i + (lane >> 3);
                const float4 v =
                    *reinterpret_cast<const float4 *>(wb + rr * BN + c0 + ((q ^ (rr & 7)) << 2));
                if (row0 + rr < M) {
                  float *d = C + (int64_t)(row0 + rr) * ldc + col;
                  if (col + 4 <= N) {
                    *reinterpret_cast<float4 *>(d) = v;
                  } else {
                    if (col < N) d[0] = v.x;
                    if (col + 1 < N) d[1] = v.y;
                    if (col + 2 < N) d[2] = v.z;
                  }
                }
              }
            }
          } else {
            // C rows off 16-byte boundaries: along rows first, so that the
            // stores that share a sector (where one 32-column group ends and
            // the next begins) follow one another.
            constexpr int NCH = BN / 32;  // 32-column groups of a staged row
            const int sw = lane & 3, cq = lane >> 2;
#pragma unroll 8
            for (int j = 0; j < 32 * NCH; ++j) {
              const int rr = j / NCH, c0 = (j % NCH) * 32, col = tn * BN + c0 + lane;
              if (row0 + rr < M && col < N)
                C[(int64_t)(row0 + rr) * ldc + col] = wb[rr * BN + c0 + ((cq ^ (rr & 7)) << 2) + sw];
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce_bar(acc));
        break;  // no further unit
      } else {
        // Persistent CTAs (the stage area holds the next tile's operands):
        // through this warp's staging buffer, EPI_COLS columns at a time, two
        // passes per 32-column TMEM load; 64-byte rows, chunk q of row r at
        // q ^ ((r >> 1) & 3).
        static_assert(G::EPI_COLS == 16 && BN % 32 == 0, "two staging passes per TMEM load");
        float *ebuf = reinterpret_cast<float *>(smem + G::STAGES * G::STAGE_BYTES) +
                      (warp - G::kEpiWarp0) * (32 * G::EPI_COLS);
#pragma unroll 1
        for (int c0 = 0; row0 < M && c0 < ncols; c0 += 32) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(t_row + (uint32_t)c0, r);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int cc = c0 + 16 * h;  // first column of this pass, within the tile
            if (cc >= ncols) break;
#pragma unroll
            for (int q = 0; q < 4; ++q)
              *reinterpret_cast<float4 *>(ebuf + lane * 16 + ((q ^ ((lane >> 1) & 3)) << 2)) =
                  make_float4(__uint_as_float(r[16 * h + 4 * q]),
                              __uint_as_float(r[16 * h + 4 * q + 1]),
                              __uint_as_float(r[16 * h + 4 * q + 2]),
                              __uint_as_float(r[16 * h + 4 * q + 3]));
            __syncwarp();
            const int col0 = tn * BN + cc;
            if (c_vec) {
              const int q = lane & 3, col = col0 + 4 * q;
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int rr = 8 * i + (lane >> 2);
                const float4 v = *reinterpret_cast<const float4 *>(
                    ebuf + rr * 16 + ((q ^ ((rr >> 1) & 3)) << 2));
                if (row0 + rr < M) {
                  float *d = C + (int64_t)(row0 + rr) * ldc + col;
                  if (col + 4 <= N) {
                    *reinterpret_cast<float4 *>(d) = v;
                  } else {
                    if (col < N) d[0] = v.x;
                    if (col + 1 < N) d[1] = v.y;
                    if (col + 2 < N) d[2] = v.z;
                  }
                }
              }
            } else {
              const int j = lane & 15, col = col0 + j;
#pragma unroll 4
              for (int i = 0; i < 16; ++i) {
                const int rr = 2 * i + (lane >> 4);
                const float v = ebuf[rr * 16 + (((j >> 2) ^ ((rr >> 1) & 3)) << 2) + (j & 3)];
                if (row0 + rr < M && col < N) C[(int64_t)(row0 + rr) * ldc + col] = v;
              }
            }
            __syncwarp();  // the buffer is rewritten by the next pass
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce_bar(acc));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  } else if constexpr (G::kSplit) {
    // -------------------------------------------- 3xTF32 split (warps 6-9)
    const int t = threadIdx.x - 32 * G::kSplitWarp0;  // 0..127
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      for (int kb = unit_kb0(u); kb < unit_kb1(u); ++kb) {
        // every lane waits: each acquires the TMA-written bytes it reads
        bool got = !*abort_flag && mbar_wait(full_bar(stage), phase);
        if (!got && lane == 0 && !*abort_flag) watchdog_trip(watchdog, kSiteSplitFull, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        // The split is elementwise, so it is independent of the swizzle: the
        // raw value is the hi part, the lo part goes to the same offset of the
        // lo copy.
        uint4 *raw = reinterpret_cast<uint4 *>(smem + stage * G::STAGE_BYTES);
        uint4 *lo = reinterpret_cast<uint4 *>(smem + stage * G::STAGE_BYTES + G::RAW_BYTES);
        float seen = 0.f;
        for (int i = t; i < G::RAW_BYTES / 16; i += 32 * G::kSplitWarps) {
          const uint4 v = raw[i];
          lo[i] = make_uint4(split_lo_tf32_fast(v.x, seen), split_lo_tf32_fast(v.y, seen),
                             split_lo_tf32_fast(v.z, seen), split_lo_tf32_fast(v.w, seen));
        }
        if (seen != seen) {  // an infinity or NaN in this thread's elements
          for (int i = t; i < G::RAW_BYTES / 16; i += 32 * G::kSplitWarps) {
            const uint4 v = raw[i];
            lo[i] = make_uint4(split_lo_tf32(v.x), split_lo_tf32(v.y), split_lo_tf32(v.z),
                               split_lo_tf32(v.w));
          }
        }
        fence_proxy_async_smem();  // generic-proxy writes -> tensor-core reads
        __syncwarp();
        if (lane == 0) mbar_arrive(split_bar(stage));
        if (++stage == G::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  }

  if (splits > 1) {
    // ---------------------------------------- K-split: cluster reduction
    // Every thread of every CTA reaches both cluster barriers, also after a
    // bounded wait gave up (the role loops above all end).
    __syncwarp();
    cluster_sync();  // partials written (release) and visible (acquire)
    bool aborted = false;
    for (int p = 0; p < splits; ++p)
      aborted |= ld_cluster_s32(mapa_shared(smem_u32(const_cast<int *>(abort_flag)),
                                            (uint32_t)p)) != 0;
    if (!aborted) {
      int tm, tn;
      tile_coords(unit_tile(blockIdx.x), tiles_m, tiles_n, group_m, tm, tn);
      const int rank = (int)cluster_ctarank();
      const int r0 = (BM * rank) / splits, r1 = (BM * (rank + 1)) / splits;
      constexpr int Q = BN / 4;  // float4s per tile row
      uint32_t part[G::MAX_SPLITS];
#pragma unroll
      for (int p = 0; p < G::MAX_SPLITS; ++p)
        part[p] = p < splits ? mapa_shared(base, (uint32_t)p) : 0u;
      for (int e = threadIdx.x; e < (r1 - r0) * Q; e += blockDim.x) {
        const int trow = r0 + e / Q, c = 4 * (e % Q);
        const uint32_t off = (uint32_t)((trow * G::PART_PITCH + c) * 4);
        float4 v[G::MAX_SPLITS];
#pragma unroll
        for (int p = 0; p < G::MAX_SPLITS; ++p)
          if (p < splits) v[p] = ld_cluster_f4(part[p] + off);
        float4 sum = v[0];  // parts added in K order
#pragma unroll
        for (int p = 1; p < G::MAX_SPLITS; ++p)
          if (p < splits) sum.x += v[p].x, sum.y += v[p].y, sum.z += v[p].z, sum.w += v[p].w;
        const int row = tm * BM + trow, col = tn * BN + c;
        if (row < M) {
          float *d = C + (int64_t)row * ldc + col;
          if (c_vec && col + 4 <= N) {
            *reinterpret_cast<float4 *>(d) = sum;
          } else {
            if (col < N) d[0] = sum.x;
            if (col + 1 < N) d[1] = sum.y;
            if (col + 2 < N) d[2] = sum.z;
            if (col + 3 < N) d[3] = sum.w;
          }
        }
      }
    }
    __syncwarp();
    cluster_sync();  // no CTA leaves while a peer may still read its partial
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();  // tcgen05.dealloc is .sync.aligned: the whole warp, converged
    tc_fence_after();
    tmem_dealloc(tmem_base, G::TMEM_COLS);
  }
}

// ===================================================================
// CTA-pair variant (cta_group::2), every operand kind.
//
// A cluster of two CTAs on two SMs computes a 256 x 256 tile.  CTA r loads
// rows [128 r, 128 r + 128) of the A panel and columns [128 r, 128 r + 128)
// of the B panel into its own shared memory; one thread of the even CTA
// issues tcgen05.mma.cta_group::2 (M = 256, N = 256), which reads both halves
// of both operands and writes rows [128 r, 128 r + 128) of the accumulator
// into CTA r's tensor memory.  Per SM this halves the B bytes fetched per
// flop compared with the single-CTA 128 x 256 tile.
//  * Both CTAs' TMA loads signal the even CTA's full barrier (pair TMA); its
//    producer posts the expected bytes of both halves.
//  * The MMA thread's commits arrive on the barrier at the same offset in
//    both CTAs (multicast): stage-free and accumulator-ready.
//  * Each CTA's epilogue reads its own TMEM rows and writes them with one
//    128-row TMA store per 32-column chunk, paced over the next tile's main
//    loop; the odd CTA's epilogue releases the accumulator on the even CTA's
//    barrier.
//  * 3xTF32: each producer also loads the lo part of its operand (written by
//    the split pre-pass) into the stage; the MMA thread issues three MMAs per
//    k-step.
//  * Before leaving, each CTA waits (bounded) for every signal still heading
//    its way, then both CTAs meet at a cluster barrier and free TMEM.
template <TcKind KIND, bool AT_ = false, bool BT_ = false>
struct Cfg2 {
  static constexpr bool AT = AT_, BT = BT_;
  // 16-bit operands (BF16 or FP16, tcgen05 kind::f16) vs 32-bit (TF32 kinds)
  static constexpr bool k16 = KIND == TcKind::kBF16 || KIND == TcKind::kF16;
  // 8-bit float operands (tcgen05 kind::f8f6f4), read K-major only
  static constexpr bool k8 = KIND == TcKind::kE4M3 || KIND == TcKind::kE5M2;
  // operand format code of the instruction descriptor: F16 0, BF16 1, TF32 2
  // (kind::f8f6f4 codes: E4M3 0, E5M2 1)
  static constexpr uint32_t kFmt = KIND == TcKind::kF16    ? 0u
                                   : KIND == TcKind::kBF16 ? 1u
                                   : KIND == TcKind::kE4M3 ? 0u
                                   : KIND == TcKind::kE5M2 ? 1u
                                                           : 2u;
  static constexpr bool kSplit = KIND == TcKind::k3xTF32;
  static constexpr int BM = 256, BN = 256;           // pair tile
  static constexpr int HM = 128, HN = 128;           // per-CTA halves
  static constexpr int ES = k8 ? 1 : k16 ? 2 : 4;
  static constexpr int BK = 128 / ES;
  static constexpr int UMMA_K = 32 / ES;
  static constexpr int KSTEPS = BK / UMMA_K;
  static constexpr int BOX = 128 / ES;            // elements in one 128-byte swizzle row
  static constexpr int BOX_N = BOX;
  static constexpr int A_BYTES = HM * 128;        // this CTA's 128 rows of M x BK
  static constexpr int B_BYTES = HN * 128;        // this CTA's 128 columns of N x BK
  static constexpr int A_BOXES = AT ? HM / BOX : 1;
  static constexpr int A_BOX_BYTES = AT ? BK * 128 : A_BYTES;
  static constexpr int B_BOXES = BT ? 1 : HN / BOX;
  static constexpr int B_BOX_BYTES = BT ? B_BYTES : BK * 128;
  static constexpr int RAW_BYTES = A_BYTES + B_BYTES;                // per CTA, per stage
  static constexpr int STAGE_BYTES = RAW_BYTES * (kSplit ? 2 : 1);   // + lo parts (3xTF32)
  static constexpr int STAGES = 196608 / STAGE_BYTES;
  static constexpr int TMEM_COLS = 512;                   // two 256-column accumulators
  static constexpr int kEpiWarps = 4;
  // Two producer threads, one per operand, in warps 0 and kProdBWarp: a TMA
  // instruction takes ~70 cycles to issue whatever its box size, and one
  // thread issuing every box of a stage fell behind the MMAs.
  static constexpr int kProdBWarp = 2 + kEpiWarps;
  static constexpr int THREADS = 32 * (3 + kEpiWarps);
  // full, empty, accf[2], acce[2], drain
  static constexpr int NUM_BARS = 2 * STAGES + 6;  // + the test-stall barrier
  // epilogue staging: two buffers of one 128 x 32 fp32 chunk (one TMA store each)
  static constexpr int EPI_BUF_BYTES = 32 * kEpiWarps * 32 * 4;
  static constexpr int EPI_BYTES = 2 * EPI_BUF_BYTES;
  static constexpr int SMEM_BYTES =
      STAGES * STAGE_BYTES + EPI_BYTES + NUM_BARS * 8 + 16 + 1024;
  static_assert(SMEM_BYTES <= 232448, "fits the 227 KB opt-in shared memory of a CTA");
  static constexpr uint32_t MN_LAYOUT = k16 ? 2u : 1u;
  static constexpr uint32_t MN_SBO = k16 ? 1024u : 512u;
  static_assert(!k8 || (!AT && BT), "8-bit operands are read K-major: A as M x K, B as N x K");
  static constexpr uint32_t IDESC = (1u << 4) | (kFmt << 7) | (kFmt << 10) |
                                    ((AT ? 1u : 0u) << 15) | ((BT ? 0u : 1u) << 16) |
                                    ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
  static_assert(STAGES >= 2, "pipeline needs at least two stages");
};

// Epilogue pacing of the CTA-pair kernel: chunk c (of 8) of a tile's C waits
// until c / kPaceParts of the previous accumulator spacing has passed; the
// spacing is capped at kPaceMaxCycles (about 1 ms), far below the wait limit.
constexpr int kPaceParts = 12;
constexpr long long kPaceMaxCycles = 1ll << 21;

enum : int {
  kSite2ProducerEmpty = 0x51,
  kSite2ProducerTail = 0x52,
  kSite2MmaFull = 0x61,
  kSite2MmaAccEmpty = 0x62,
  kSite2MmaDrain = 0x63,
  kSite2MmaTail = 0x64,
  kSite2EpiAccFull = 0x71,
  kSite2TestStall = 0x66,  // DGEMM_TC_TEST_STALL: the MMA thread's test wait ran out
};

template <TcKind KIND, bool AT, bool BT>
__global__ void __launch_bounds__(Cfg2<KIND, AT, BT>::THREADS, 1)
    tc2_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                    const __grid_constant__ CUtensorMap tmap_b,
                    const __grid_constant__ CUtensorMap tmap_c,
                    const __grid_constant__ CUtensorMap tmap_al,
                    const __grid_constant__ CUtensorMap tmap_bl, float *__restrict__ C, int M,
                    int N, int K, int64_t ldc, int c_tma, int c_vec, int group_m,
                    int *watchdog, int mn3d, int stall, int snake) {
  using G = Cfg2<KIND, AT, BT>;
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw_base);

  const uint32_t epi_base = base + G::STAGES * G::STAGE_BYTES;
  const uint32_t bars = epi_base + G::EPI_BYTES;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (G::STAGES + s); };
  auto accf_bar = [&](int b) { return bars + 8u * (2 * G::STAGES + b); };
  auto acce_bar = [&](int b) { return bars + 8u * (2 * G::STAGES + 2 + b); };
  const uint32_t drain_bar = bars + 8u * (2 * G::STAGES + 4);
  const uint32_t stall_bar = bars + 8u * (2 * G::STAGES + 5);  // nothing ever arrives here
  uint8_t *tail = smem + G::STAGES * G::STAGE_BYTES + G::EPI_BYTES + G::NUM_BARS * 8;
  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(tail);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tail + 4);
  auto a_tile = [&](int s) { return base + (uint32_t)(s * G::STAGE_BYTES); };
  auto b_tile = [&](int s) { return base + (uint32_t)(s * G::STAGE_BYTES + G::A_BYTES); };
  auto a_lo = [&](int s) { return a_tile(s) + (uint32_t)G::RAW_BYTES; };
  auto b_lo = [&](int s) { return b_tile(s) + (uint32_t)G::RAW_BYTES; };

  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cluster = blockIdx.x >> 1, clusters = gridDim.x >> 1;
  const int tiles_m = (M + G::BM - 1) / G::BM;
  const int tiles_n = (N + G::BN - 1) / G::BN;
  const int num_tiles = tiles_m * tiles_n;
  const int kblocks = (K + G::BK - 1) / G::BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < G::STAGES; ++s) {
      mbar_init(full_bar(s), 2);  // one arrival per producer thread
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), 2 * G::kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    mbar_init(stall_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
    if (c_tma) tma_prefetch_desc(&tmap_c);
    if constexpr (G::kSplit) {
      tma_prefetch_desc(&tmap_al);
      tma_prefetch_desc(&tmap_bl);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(const_cast<uint32_t *>(tmem_slot)), G::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  __syncwarp();
  cluster_sync();  // the peer's barriers are initialised before any signal crosses
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // set-up done; the previous kernel on the stream has completed

  if (warp == 0 || warp == G::kProdBWarp) {
    // ----------------------------------------------------------- producers
    // warp 0 loads this CTA's part of op(A), warp kProdBWarp its part of
    // op(B); each arrives once per stage on the full barrier with its bytes.
    // 3xTF32: each also loads the lo part of its operand (written by the
    // split pre-pass, same geometry) into the stage's lo area.
    if (lane == 0) {
      const bool is_a = warp == 0;
      const uint32_t bytes =
          (is_a ? (uint32_t)G::A_BYTES : (uint32_t)G::B_BYTES) * (G::kSplit ? 2u : 1u);
      // Both CTAs' halves signal the even CTA's full barrier (stage s at +8 s).
      const uint32_t fb0 = mapa_shared(full_bar(0), 0);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = cluster; tile < num_tiles && ok; tile += clusters) {
        int tm, tn;
        tile_coords(tile, tiles_m, tiles_n, group_m, tm, tn);
        const int m0 = tm * G::BM + (int)rank * G::HM;  // this CTA's rows of op(A)
        const int n0 = tn * G::BN + (int)rank * G::HN;  // this CTA's columns of op(B)
        const bool rev = snake && (((tile - cluster) / clusters) & 1);
        for (int kq = 0; kq < kblocks; ++kq) {
          const int kb = rev ? kblocks - 1 - kq : kq;
          // The abort flag is only consulted when the stage is not free yet:
          // on the fast path nothing is waiting for this thread to stop.
          if (!mbar_try_wait(empty_bar(stage), phase ^ 1u) &&
              (*abort_flag || !mbar_wait(empty_bar(stage), phase ^ 1u))) {
            if (!*abort_flag) watchdog_trip(watchdog, kSite2ProducerEmpty, abort_flag);
            ok = false;
            break;
          }
          const uint32_t fb = fb0 + 8u * (uint32_t)stage;
          // The copies are issued first and the expected bytes announced after
          // them (the barrier's transaction count may run below zero in
          // between; the phase still needs both producers' arrivals), which
          // takes the arrival off the path from a free stage to its loads.
          // An MN-major operand with a 3-D map comes in one instruction.
          const bool one3d = is_a ? (AT && (mn3d & kA3d)) : (!BT && (mn3d & kB3d));
#pragma unroll
          for (int part = 0; part < (G::kSplit ? 2 : 1); ++part) {  // raw, then lo
            const uint32_t lo_off = part ? (uint32_t)G::RAW_BYTES : 0u;
            if (one3d) {
              const uint32_t dst = (is_a ? a_tile(stage) : b_tile(stage)) + lo_off;
              const CUtensorMap *map =
                  is_a ? (part ? &tmap_al : &tmap_a) : (part ? &tmap_bl : &tmap_b);
              const int z = (is_a ? m0 : n0) / G::BOX;
              tma_load_3d_pair(dst, map, fb, 0, kb * G::BK, z);
            } else if (is_a) {
#pragma unroll
              for (int j = 0; j < G::A_BOXES; ++j) {
                const uint32_t dst = a_tile(stage) + lo_off + j * G::A_BOX_BYTES;
                const int x = AT ? m0 + j * G::BOX : kb * G::BK, y = AT ? kb * G::BK : m0;
                tma_load_2d_pair(dst, part ? &tmap_al : &tmap_a, fb, x, y);
              }
            } else {
#pragma unroll
              for (int j = 0; j < G::B_BOXES; ++j) {
                const uint32_t dst = b_tile(stage) + lo_off + j * G::B_BOX_BYTES;
                const int x = BT ? kb * G::BK : n0 + j * G::BOX, y = BT ? n0 : kb * G::BK;
                tma_load_2d_pair(dst, part ? &tmap_bl : &tmap_b, fb, x, y);
              }
            }
          }
          if (leader) mbar_arrive_expect_tx(full_bar(stage), 2u * bytes);
          if (++stage == G::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Tail: wait until the MMAs have released every stage loaded here, so
      // that all stage-free signals aimed at this CTA have landed (and, on an
      // abort, that no copy is still writing this CTA's shared memory).
      for (int i = 0; i < G::STAGES; ++i) {
        if (!mbar_wait(empty_bar(stage), phase ^ 1u)) {
          atomicCAS(watchdog, 0, kSite2ProducerTail);
          break;
        }
        if (++stage == G::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------- MMA (even CTA only)
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      if (stall && cluster == 0) {
        // Test hook: wait on a barrier that nothing arrives at, so that the
        // bounded wait runs out and the abort path below runs for real.
        if (!mbar_wait(stall_bar, 0)) watchdog_trip(watchdog, kSite2TestStall, abort_flag);
        ok = false;
      }
      for (int tile = cluster; tile < num_tiles && ok; tile += clusters) {
        if (*abort_flag || !mbar_wait(acce_bar(acc), acc_phase ^ 1u)) {
          if (!*abort_flag) watchdog_trip(watchdog, kSite2MmaAccEmpty, abort_flag);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * G::BN);
        for (int kb = 0; kb < kblocks; ++kb) {
          const bool got = mbar_try_wait(full_bar(stage), phase) ||
                           (!*abort_flag && mbar_wait(full_bar(stage), phase));
          if (!got) {
            if (!*abort_flag) watchdog_trip(watchdog, kSite2MmaFull, abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < G::KSTEPS; ++k) {
            const uint64_t ad = operand_desc<G, AT>(a_tile(stage), k, G::A_BOX_BYTES);
            const uint64_t bd = operand_desc<G, !BT>(b_tile(stage), k, G::B_BOX_BYTES);
            const uint32_t accum = (kb > 0 || k > 0) ? 1u : 0u;
            if constexpr (G::kSplit) {
              const uint64_t adl = operand_desc<G, AT>(a_lo(stage), k, G::A_BOX_BYTES);
              const uint64_t bdl = operand_desc<G, !BT>(b_lo(stage), k, G::B_BOX_BYTES);
              umma_tf32_pair(d_tmem, adl, bd, G::IDESC, accum);  // A_lo B_hi
              umma_tf32_pair(d_tmem, ad, bdl, G::IDESC, 1u);     // A_hi B_lo
              umma_tf32_pair(d_tmem, ad, bd, G::IDESC, 1u);      // A_hi B_hi
            } else if constexpr (G::k8) {
              umma_f8_pair(d_tmem, ad, bd, G::IDESC, accum);
            } else if constexpr (G::k16) {
              umma_f16_pair(d_tmem, ad, bd, G::IDESC, accum);
            } else {
              umma_tf32_pair(d_tmem, ad, bd, G::IDESC, accum);
            }
          }
          umma_commit_pair(empty_bar(stage), 0x3);  // frees the stage in both CTAs
          if (++stage == G::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(accf_bar(acc), 0x3);  // accumulator ready in both CTAs
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      umma_commit_pair(drain_bar, 0x1);
      if (!mbar_wait(drain_bar, 0)) atomicCAS(watchdog, 0, kSite2MmaDrain);
      // Tail: both accumulators released by both epilogues, so that every
      // release signal from the odd CTA has landed before this CTA leaves.
      for (int i = 0; i < 2; ++i) {
        if (!mbar_wait(acce_bar(acc), acc_phase ^ 1u)) {
          atomicCAS(watchdog, 0, kSite2MmaTail);
          break;
        }
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
    }
  } else if (warp < 2 + G::kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    // The four epilogue warps work in step (named barrier 1): each 32-column
    // chunk of this CTA's 128 x 256 accumulator goes out as one 128 x 32 TMA
    // store, issued by the first epilogue warp.
    const int quarter = warp & 3;
    const bool issuer = warp == 2 && lane == 0;
    int epi_chunk = 0;  // TMA-store chunks issued by this CTA's epilogue
    const uint32_t acce_leader0 = mapa_shared(acce_bar(0), 0);
    const uint32_t acce_leader1 = mapa_shared(acce_bar(1), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    long long t_prev = 0, t_span = 0;
    for (int tile = cluster; tile < num_tiles; tile += clusters) {
      int tm, tn;
      tile_coords(tile, tiles_m, tiles_n, group_m, tm, tn);
      bool ok = !*abort_flag && mbar_wait(accf_bar(acc), acc_phase);
      if (!ok && lane == 0 && !*abort_flag) watchdog_trip(watchdog, kSite2EpiAccFull, abort_flag);
      // one decision for all four warps: they meet at the barrier below
      if (!named_bar_and<1, 32 * G::kEpiWarps>(ok)) break;
      tc_fence_after();
      // Pacing.  Every CTA finishes its tiles at about the same time, and C
      // written in one burst from all SMs holds up the operand loads of the
      // next tiles.  The chunks of a tile are therefore spread over the first
      // 7/12 of the next tile's main loop (its length taken from the spacing
      // of the last two accumulators, capped), which the second accumulator
      // leaves room for.  The first tile is not paced (no spacing known yet),
      // nor the last one (nothing left to overlap with).
      const long long t_acc = clock64();
      if (t_prev) t_span = min(t_acc - t_prev, kPaceMaxCycles);
      t_prev = t_acc;
      const bool pace = t_span > 0 && tile + clusters < num_tiles;
      const int row0 = tm * G::BM + (int)rank * G::HM;  // this CTA's first row of C
      const uint32_t t_row =
          tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * G::BN);
#pragma unroll 1
      for (int c0 = 0; c0 < G::BN; c0 += 32) {
        if (pace && c0 > 0) {
          const long long due = t_acc + t_span * (c0 / 32) / kPaceParts;
          while (clock64() < due) __nanosleep(100);
        }
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + (uint32_t)c0, r);
        tmem_wait_ld();
        const int col = tn * G::BN + c0;
        // Each warp stages its 32 rows (row = lane) of the chunk in
        // 128B-swizzled shared memory.  A chunk wholly inside N of a C that
        // TMA can write goes out as one 128-row box in one TMA store (full
        // lines; rows past M are dropped by the hardware).  Other chunks (the
        // inner edge, where a TMA store would write whole 16-byte granules
        // and touch the ldc gap when N is not a multiple of 4, or a C that
        // TMA cannot write) are written by the warp itself, row by row from
        // its own 32 rows.  The conditions are the same in all four warps.
        // With TMA stores: two buffers; before one is refilled, the store
        // issued from it two chunks ago must have read it.  Without: buffer
        // 0, which no TMA store reads.
        const bool tma_chunk = c_tma && col + 32 <= N;
        uint32_t buf = epi_base;
        if (c_tma) {
          buf = epi_base + (uint32_t)((epi_chunk & 1) * G::EPI_BUF_BYTES);
          if (issuer && epi_chunk >= 2) bulk_wait_group_read<1>();
          named_bar_sync<1, 32 * G::kEpiWarps>();
        }
        const uint32_t wbuf = buf + (uint32_t)(quarter * 32 * 128);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t dst = wbuf + (uint32_t)(lane * 128 + ((c ^ (lane & 7)) << 4));
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(r[4 * c]),
                       "r"(r[4 * c + 1]), "r"(r[4 * c + 2]), "r"(r[4 * c + 3])
                       : "memory");
        }
        if (tma_chunk) {
          fence_proxy_async_smem();
          named_bar_sync<1, 32 * G::kEpiWarps>();
          if (issuer) {
            // A box wholly outside C is not issued; a (possibly empty) group
            // is committed for every chunk so that "at most one group still
            // reading" always refers to the other buffer.
            if (row0 < M) tma_store_2d(&tmap_c, buf, col, row0);
            bulk_commit_group();
          }
        } else {
          __syncwarp();
          const int wrow0 = row0 + quarter * 32;  // C row of the warp's staged row 0
          const float *wb = reinterpret_cast<const float *>(smem + (wbuf - base));
          if (wrow0 < M && col < N) {
            if (c_vec) {  // 16-byte stores: eight lanes to a row, four rows at a time
              const int q = lane & 7, c4 = col + 4 * q;
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int rr = 4 * i + (lane >> 3);
                const float4 v =
                    *reinterpret_cast<const float4 *>(wb + rr * 32 + ((q ^ (rr & 7)) << 2));
                if (wrow0 + rr < M) {
                  float *d = C + (int64_t)(wrow0 + rr) * ldc + c4;
                  if (c4 + 4 <= N) {
                    *reinterpret_cast<float4 *>(d) = v;
                  } else {
                    if (c4 < N) d[0] = v.x;
                    if (c4 + 1 < N) d[1] = v.y;
                    if (c4 + 2 < N) d[2] = v.z;
                  }
                }
              }
            } else {  // one element per lane, a row per instruction
#pragma unroll 8
              for (int rr = 0; rr < 32; ++rr) {
                const float v = wb[rr * 32 + (((lane >> 2) ^ (rr & 7)) << 2) + (lane & 3)];
                if (wrow0 + rr < M && col + lane < N) C[(int64_t)(wrow0 + rr) * ldc + col + lane] = v;
              }
            }
          }
          __syncwarp();  // the warp's rows are rewritten by the next chunk
          if (c_tma && issuer) bulk_commit_group();  // one group per chunk
        }
        if (c_tma) ++epi_chunk;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc ? acce_leader1 : acce_leader0);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (issuer) bulk_wait_group<0>();  // every TMA store of this CTA complete
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  __syncwarp();
  cluster_sync();  // neither CTA leaves while the other may still signal it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, G::TMEM_COLS);
  }
}

// ------------------------------------------------------------- host side
// Tile rows per raster group: `dflt` unless DGEMM_TC_GROUP_M (1..64)
// overrides it for tuning sweeps; it changes only the order tiles are visited
// in.  Measured best on GB300: 32 rows of 128-row tiles for the single-CTA
// kernel; for the pair kernel 16 rows of 256-row tiles with 16- and 8-bit
// operands, 8 rows with 32-bit operands (as fast as 16 with the snake k
// order, and 2.27 -> 2.21 GB of DRAM reads at 8192^3).
int raster_group_m(int dflt) {
  static const int g = [] {
    const char *e = getenv("DGEMM_TC_GROUP_M");
    const int v = e ? atoi(e) : 0;
    return (v >= 1 && v <= 64) ? v : 0;
  }();
  return g ? g : dflt;
}

// k order of the CTA-pair kernel: with `snake` a pair walks the k-blocks of
// every second tile of its list backwards, so that the tiles starting a
// round read first the k-blocks the previous round read last, which L2 still
// holds.  At 8192^3 TF32 this cut DRAM reads 2.81 -> 2.27 GB per launch
// (2.21 GB with raster groups of 8 tile rows) and ran 1.2% faster (2.2% on
// the transformer-layer shape, paired on one box); for BF16 and E4M3 it was
// 0.2% and 1.1% slower, so it is the default for 32-bit operands only.
// DGEMM_TC_SNAKE=0 / =1 forces it (read at every launch).
int snake_order(bool dflt) {
  const char *e = getenv("DGEMM_TC_SNAKE");
  if (e && (e[0] == '0' || e[0] == '1')) return e[0] - '0';
  return dflt ? 1 : 0;
}

// Small-problem configuration of the single-CTA kernel: 128 x 128 tiles and
// 3 stages (96 KB of stages, 256 TMEM columns), so that two CTAs fit on an
// SM: the next call's CTAs can then start their set-up beside the previous
// call's (programmatic dependent launch), and each CTA writes half the C of a
// 128 x 256 tile.  It pays where 128 x 128 tiles would overfill one CTA per
// SM and a row of K is short (2048^2 x 256 TF32: 8.3 us against 10.0 at one
// CTA per SM); single_tile below decides.
constexpr int kSmallBudget = 3 * 32768;

// Tile of the single-CTA kernel: 128 x BN, one CTA per SM (192 KB of
// stages), or the 128 x 128 two-CTAs-per-SM configuration above; "Deep":
// stages two 128-byte swizzle rows of K deep.
enum class Tile { k64, k64Deep, k128, k128Deep, k128Small, k256 };

// The K-split choose_splits would make, without its occupancy query (every
// cluster size taken to fit).
int expected_splits(int64_t tiles, int kblocks, int64_t slots) {
  if (tiles * 2 > slots) return 1;
  int s = (int)(slots / tiles);
  s = s < 8 ? s : 8;
  s = s < kblocks / 4 ? s : kblocks / 4;
  for (; s >= 2; --s) {
    const int per = (kblocks + s - 1) / s;
    const int w = (kblocks + per - 1) / per;
    if (tiles <= slots / w) return w;
  }
  return 1;
}

// Tile for the single-CTA kernel.  "第八课：GPU 如何完成矩阵乘法" section 十七
// weighs tile size (operand reuse) against concurrency; on GB300 a problem
// this small is bound by how fast each SM can pull its operands from L2
// (about 100 GB/s per CTA measured), so the choice, fitted to a same-process
// sweep of 14 shapes x 3 kinds x 10 configurations (within 5% of the best
// configuration on 40 of the 42 points, 13% faster than the fixed 128 x 256
// / 128 x 128 choice on average) and checked on the same shapes for 8-bit
// operands (within 5% on 13 of 14):
//  - every kind but 3xTF32, in this order: the small configuration when a
//    row of K is at most 1 KB and 128 x 128 tiles would overfill one CTA per
//    SM; else the widest tile (256, 128, 64) whose tile count fills at least
//    half the SMs without a K-split (the 64-wide tile only while a row of K
//    is at most 4 KB: beyond that the K-split's halved operand traffic per
//    CTA wins over its reduction);
//  - otherwise, and always for 3xTF32 (whose split warps favour wide tiles):
//    the width whose expected K-split plan moves the fewest operand bytes
//    through the busiest SM, a K-split counted as 250 KB (its DSMEM
//    reduction, ~2.5 us at that rate);
//  - 128 x 64 and 128 x 128 tiles then take stages two swizzle rows of K
//    deep (48 and 64 KB), when K fills at least four shallow stages and
//    unless that lowers the K-split's part count: a TMA
//    load costs a nearly fixed time per box, so a deep stage fills about
//    twice as fast (measured: 1024^3 TF32 10.6 -> 9.6 us, BF16 1536^3
//    10.9 -> 9.3 us).
// DGEMM_TC_BN=64 / 128 / 256 forces the width (one CTA per SM),
// DGEMM_TC_KD=1 / 2 the stage depth (2: wherever it fits), DGEMM_TC_SMALL=1
// / =0 forces the small configuration / rules it out (read at every launch,
// for tests and tuning).
Tile single_tile(TcKind kind, int M, int N, int K, int num_sms) {
  const int es = (kind == TcKind::kE4M3 || kind == TcKind::kE5M2) ? 1
                 : (kind == TcKind::kBF16 || kind == TcKind::kF16) ? 2
                                                                    : 4;
  const bool split3 = kind == TcKind::k3xTF32;
  const char *kde = getenv("DGEMM_TC_KD");
  const int kd_env = (kde && (kde[0] == '1' || kde[0] == '2') && kde[1] == 0) ? kde[0] - '0' : 0;
  // 128 x 64 and 128 x 128 tiles take deep stages unless that halves the
  // k-blocks a K-split would share out (3xTF32: 128 x 64 only, its deep
  // 128 x 128 stages would not fit twice)
  const int bk = 128 / es, kblocks = (K + bk - 1) / bk;
  const int64_t tm = (M + 127) / 128, kes = (int64_t)K * es;
  auto tiles = [&](int bn) { return tm * ((N + bn - 1) / bn); };
  auto deepen = [&](Tile t) {
    if (kd_env == 1) return t;
    const bool can = t == Tile::k64 || (t == Tile::k128 && !split3);
    // (K of at most three shallow stages: a deep stage would be half empty)
    if (!can || (kd_env != 2 && kblocks < 4)) return t;
    const int64_t n = tiles(t == Tile::k64 ? 64 : 128);
    if (kd_env != 2 && expected_splits(n, (kblocks + 1) / 2, num_sms) !=
                           expected_splits(n, kblocks, num_sms))
      return t;
    return t == Tile::k64 ? Tile::k64Deep : Tile::k128Deep;
  };
  if (const char *e = getenv("DGEMM_TC_BN")) {
    if (strcmp(e, "64") == 0) return kd_env == 2 ? deepen(Tile::k64) : Tile::k64;
    if (strcmp(e, "128") == 0) return kd_env == 2 ? deepen(Tile::k128) : Tile::k128;
    if (strcmp(e, "256") == 0) return Tile::k256;
  }
  const char *sm = getenv("DGEMM_TC_SMALL");
  const int small = (sm && (sm[0] == '0' || sm[0] == '1') && sm[1] == 0) ? sm[0] - '0' : -1;
  if (!split3 && small == 1) return Tile::k128Small;
  if (!split3) {
    if (small != 0 && kes <= 1024 && tiles(128) > num_sms) return Tile::k128Small;
    if (2 * tiles(256) >= num_sms) return Tile::k256;
    if (2 * tiles(128) >= num_sms) return deepen(Tile::k128);
    if (2 * tiles(64) >= num_sms && kes <= (kd_env == 1 ? 2048 : 4096))
      return deepen(Tile::k64);
  }
  Tile best = Tile::k256;
  double best_cost = 0;
  for (int bn : {256, 128, 64}) {
    const int64_t t = tiles(bn);
    const int s = expected_splits(t, kblocks, num_sms);
    const int64_t waves = (t * s + num_sms - 1) / num_sms;
    const double bytes = (double)(128 + bn) * ((kblocks + s - 1) / s) * bk * es;
    const double cost = (double)waves * bytes + (s > 1 ? 250e3 : 0.0);
    if (bn == 256 || cost < best_cost) {
      best_cost = cost;
      best = bn == 256 ? Tile::k256 : bn == 128 ? Tile::k128 : Tile::k64;
    }
  }
  return deepen(best);
}

// DGEMM_TC_TEST_STALL=1 makes the MMA thread of the first CTA (pair) wait on
// a barrier that nothing arrives at: its bounded wait runs out after ~2 s and
// the kernel takes its abort path (watchdog site code, drained copies, freed
// tensor memory, incomplete C).  For the failure-detection test only; read
// at every launch.
int test_stall() {
  const char *e = getenv("DGEMM_TC_TEST_STALL");
  return (e && e[0] == '1') ? 1 : 0;
}

template <TcKind KIND>
constexpr CUtensorMapDataType tma_type() {
  return KIND == TcKind::kBF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
         : KIND == TcKind::kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
         : (KIND == TcKind::kE4M3 || KIND == TcKind::kE5M2) ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
}

// Tensor maps of A and B for configuration G, whose tiles hold `rows_a` rows
// of op(A) and `cols_b` columns of op(B) per CTA.  K-major operands are read
// as boxes of BK (one 128-byte swizzle row) x rows; MN-major operands as
// boxes of 128 bytes of M or N x BK rows, with the 32-byte-atom swizzle for
// 32-bit elements.
// 3-D view of a row-major rows x cols matrix whose cols are a multiple of
// `blk`: (c, r, j) -> X[r][j * blk + c], so that one box of blk x box_rows x
// nblk lands in shared memory exactly as nblk 2-D boxes of blk x box_rows
// side by side.  One TMA instruction then loads what took nblk.
bool make_map3(CUtensorMap *map, const void *ptr, CUtensorMapDataType dt, int es, int64_t rows,
               int64_t cols, int64_t ld, int blk, int box_rows, int nblk, CUtensorMapSwizzle swz) {
  auto enc = get_encode();
  if (!enc || cols % blk != 0) return false;
  cuuint64_t dims[3] = {(cuuint64_t)blk, (cuuint64_t)rows, (cuuint64_t)(cols / blk)};
  cuuint64_t strides[2] = {(cuuint64_t)(ld * es), (cuuint64_t)(blk * es)};
  cuuint32_t box[3] = {(cuuint32_t)blk, (cuuint32_t)box_rows, (cuuint32_t)nblk};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, dt, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <class G, TcKind KIND>
bool make_operand_maps(CUtensorMap *ta, CUtensorMap *tb, int M, int N, int K, const void *A,
                       int64_t lda, const void *B, int64_t ldb, int rows_a, int cols_b,
                       int *mn3d) {
  const CUtensorMapDataType dt = tma_type<KIND>();
  const CUtensorMapSwizzle mn_swz =
      (G::k16 || G::k8) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B;
  *mn3d = 0;
  bool ok_a, ok_b;
  if (G::AT && make_map3(ta, A, dt, G::ES, K, M, lda, G::BOX, G::BK, rows_a / G::BOX, mn_swz)) {
    *mn3d |= kA3d;
    ok_a = true;
  } else {
    ok_a = G::AT ? make_map(ta, A, dt, G::ES, K, M, lda, G::BOX, G::BK, mn_swz)
                 : make_map(ta, A, dt, G::ES, M, K, lda, G::BOX, rows_a, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (!G::BT && make_map3(tb, B, dt, G::ES, K, N, ldb, G::BOX, G::BK, cols_b / G::BOX, mn_swz)) {
    *mn3d |= kB3d;
    ok_b = true;
  } else {
    ok_b = G::BT ? make_map(tb, B, dt, G::ES, N, K, ldb, G::BOX, cols_b, CU_TENSOR_MAP_SWIZZLE_128B)
                 : make_map(tb, B, dt, G::ES, K, N, ldb, G::BOX, G::BK, mn_swz);
  }
  return ok_a && ok_b;
}

// Clusters of `size` CTAs of `kern` that can be resident at once on device
// `dev` (queried once per kernel, device and size).
template <class Kern>
int active_clusters(Kern kern, int threads, int smem, int dev, int size) {
  static std::atomic<int> cache[64][9] = {};
  if (dev < 0 || dev >= 64 || size < 1 || size > 8) return 0;
  int n = cache[dev][size].load(std::memory_order_relaxed);
  if (n == 0) {
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
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 0) {
      cudaGetLastError();  // not sticky; treat as "does not fit"
      n = 0;
    }
    cache[dev][size].store(n > 0 ? n : -1, std::memory_order_relaxed);
  }
  return n > 0 ? n : 0;
}

// Parts per tile for the single-CTA kernel.  "第八课：GPU 如何完成矩阵乘法"
// section 十七 weighs tile size (reuse) against concurrency; here the tile
// keeps its size and a problem whose tiles would leave more than half the
// SMs idle gains concurrency by splitting each tile along K into up to 8
// parts of at least 4 k-blocks (every part non-empty), the largest count whose
// clusters are all resident at once.  DGEMM_TC_SPLITK=0 disables the split;
// DGEMM_TC_SPLITK=2..8 forces that many parts (as far as the k-blocks allow;
// clusters that do not fit run in waves), for tests and tuning.
template <class Kern>
int choose_splits(Kern kern, int threads, int smem, int dev, int64_t tiles, int kblocks,
                  int slots) {
  auto whole = [&](int s) {  // parts actually used when aiming for s
    const int per = (kblocks + s - 1) / s;
    return (kblocks + per - 1) / per;
  };
  const char *env = getenv("DGEMM_TC_SPLITK");
  if (env && env[0] >= '0' && env[0] <= '8' && env[1] == 0) {
    const int f = env[0] - '0';
    return f >= 2 && kblocks >= 2 ? whole(f < kblocks ? f : kblocks) : 1;
  }
  if (tiles * 2 > slots) return 1;
  int s = (int)(slots / tiles);
  s = s < 8 ? s : 8;
  s = s < kblocks / 4 ? s : kblocks / 4;
  for (; s >= 2; --s) {
    const int w = whole(s);
    if (tiles <= (int64_t)active_clusters(kern, threads, smem, dev, w)) return w;
  }
  return 1;
}

template <TcKind KIND, int BN, bool AT, bool BT, int BUDGET = 196608, int KD = 1>
cudaError_t launch_cfg(int M, int N, int K, const void *A, int64_t lda, const void *B,
                       int64_t ldb, float *C, int64_t ldc, bool c_vec, int num_sms,
                       int *watchdog, cudaStream_t stream) {
  using G = Cfg<KIND, BN, AT, BT, BUDGET, KD>;
  CUtensorMap ta, tb;
  int mn3d = 0;
  if (!make_operand_maps<G, KIND>(&ta, &tb, M, N, K, A, lda, B, ldb, BM, BN, &mn3d))
    return cudaErrorInvalidValue;
  auto kern = tc_gemm_kernel<KIND, BN, AT, BT, BUDGET, KD>;
  static std::atomic<bool> attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev].store(true, std::memory_order_release);
  }
  const int64_t tiles = (int64_t)((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  if (tiles > 0x3fffffff) return cudaErrorInvalidValue;
  const int kblocks = (K + G::BK - 1) / G::BK;
  const int64_t slots = (int64_t)num_sms * G::CTAS_PER_SM;
  const int splits = choose_splits(kern, G::THREADS, G::SMEM_BYTES, dev, tiles, kblocks,
                                   (int)slots);
  // K-split: one unit per CTA, the `splits` parts of a tile in one cluster;
  // else a persistent grid of at most CTAS_PER_SM CTAs per SM.
  const int64_t grid = splits > 1 ? tiles * splits : (tiles < slots ? tiles : slots);
  e = launch_kernel(kern, dim3((unsigned)grid), dim3(G::THREADS), G::SMEM_BYTES, stream,
                    splits > 1 ? (unsigned)splits : 1u, ta, tb, C, M, N, K, ldc, c_vec ? 1 : 0,
                    raster_group_m(32), watchdog, splits, mn3d, test_stall());
  if (e == cudaSuccess) count_launch();
  return e;
}

template <TcKind KIND, bool AT, bool BT>
cudaError_t launch_cfg2(int M, int N, int K, const void *A, int64_t lda, const void *B,
                        int64_t ldb, float *C, int64_t ldc, bool c_vec, int *watchdog,
                        cudaStream_t stream, const void *A_lo, const void *B_lo) {
  using G = Cfg2<KIND, AT, BT>;
  CUtensorMap ta, tb, tc, tal, tbl;
  int mn3d = 0;
  if (!make_operand_maps<G, KIND>(&ta, &tb, M, N, K, A, lda, B, ldb, G::HM, G::HN, &mn3d))
    return cudaErrorInvalidValue;
  // 3xTF32: maps of the lo parts, the same geometry (and the same choice of
  // 3-D maps, which the kernel makes once for both)
  memset(&tal, 0, sizeof(tal));
  memset(&tbl, 0, sizeof(tbl));
  if constexpr (G::kSplit) {
    int mn3d_lo = 0;
    if (A_lo == nullptr || B_lo == nullptr ||
        !make_operand_maps<G, KIND>(&tal, &tbl, M, N, K, A_lo, lda, B_lo, ldb, G::HM, G::HN,
                                    &mn3d_lo) ||
        mn3d_lo != mn3d)
      return cudaErrorInvalidValue;
  }
  // C through TMA stores when its rows start on 16-byte boundaries.
  memset(&tc, 0, sizeof(tc));
  const bool c_tma = c_vec && make_map(&tc, C, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, M, N, ldc, 32,
                                       G::HM, CU_TENSOR_MAP_SWIZZLE_128B);
  auto kern = tc2_gemm_kernel<KIND, AT, BT>;
  static std::atomic<int> max_clusters[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(G::THREADS);
  cfg.dynamicSmemBytes = G::SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int maxc = (dev >= 0 && dev < 64) ? max_clusters[dev].load(std::memory_order_acquire) : 0;
  if (maxc == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(2);
    e = cudaOccupancyMaxActiveClusters(&maxc, (void *)kern, &cfg);
    if (e != cudaSuccess) return e;
    if (maxc < 1) return cudaErrorInvalidConfiguration;
    if (dev >= 0 && dev < 64) max_clusters[dev].store(maxc, std::memory_order_release);
  }
  const int64_t tiles = (int64_t)((M + G::BM - 1) / G::BM) * ((N + G::BN - 1) / G::BN);
  if (tiles > 0x3fffffff) return cudaErrorInvalidValue;
  const int clusters = (int)(tiles < maxc ? tiles : maxc);
  e = launch_kernel(kern, dim3(2 * clusters), dim3(G::THREADS), G::SMEM_BYTES, stream, 2u, ta, tb,
                    tc, tal, tbl, C, M, N, K, ldc, c_tma ? 1 : 0, c_vec ? 1 : 0,
                    raster_group_m(G::ES == 4 ? 8 : 16), watchdog,
                    mn3d, test_stall(), snake_order(G::ES == 4));
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

// Pair kernel or single-CTA kernel (tc_use_pair, then single_tile); 3xTF32
// takes the pair kernel only with the lo parts of A and B at hand.
template <TcKind KIND>
cudaError_t launch_kind(int M, int N, int K, const void *A, int64_t lda, const void *B,
                        int64_t ldb, float *C, int64_t ldc, bool c_vec, int num_sms,
                        int *watchdog, cudaStream_t stream, const void *A_lo, const void *B_lo) {
  constexpr bool AT = kUnitAT, BT = kUnitBT;
  const bool lo_ok = KIND != TcKind::k3xTF32 || (A_lo != nullptr && B_lo != nullptr);
  if (lo_ok && tc_use_pair(M, N, num_sms))
    return launch_cfg2<KIND, AT, BT>(M, N, K, A, lda, B, ldb, C, ldc, c_vec, watchdog, stream,
                                     A_lo, B_lo);
  switch (single_tile(KIND, M, N, K, num_sms)) {
    case Tile::k64Deep:
      return launch_cfg<KIND, 64, AT, BT, 196608, 2>(M, N, K, A, lda, B, ldb, C, ldc, c_vec,
                                                      num_sms, watchdog, stream);
    case Tile::k64:
      return launch_cfg<KIND, 64, AT, BT>(M, N, K, A, lda, B, ldb, C, ldc, c_vec, num_sms,
                                          watchdog, stream);
    case Tile::k128Deep:  // (never chosen for 3xTF32)
      if constexpr (KIND != TcKind::k3xTF32)
        return launch_cfg<KIND, 128, AT, BT, 196608, 2>(M, N, K, A, lda, B, ldb, C, ldc, c_vec,
                                                         num_sms, watchdog, stream);
      [[fallthrough]];
    case Tile::k128:
      return launch_cfg<KIND, 128, AT, BT>(M, N, K, A, lda, B, ldb, C, ldc, c_vec, num_sms,
                                           watchdog, stream);
    case Tile::k128Small:
      if constexpr (KIND != TcKind::k3xTF32)
        return launch_cfg<KIND, 128, AT, BT, kSmallBudget>(M, N, K, A, lda, B, ldb, C, ldc, c_vec,
                                                            num_sms, watchdog, stream);
      break;
    case Tile::k256:
      break;
  }
  return launch_cfg<KIND, 256, AT, BT>(M, N, K, A, lda, B, ldb, C, ldc, c_vec, num_sms, watchdog,
                                       stream);
}

#if DGEMM_TC_UNIT == 0
__global__ void read_watchdog_kernel(int *out) {
  pdl_wait();
  *out = g_watchdog;
  g_watchdog = 0;
}
#endif

}  // namespace

// This unit's layout: every tensor-core kind with AT = kUnitAT, BT = kUnitBT.
cudaError_t DG_UNIT_LAUNCHER(TcKind kind, int M, int N, int K, const void *A, int64_t lda,
                             const void *B, int64_t ldb, float *C, int64_t ldc, bool c_vec,
                             int num_sms, int *watchdog, cudaStream_t stream, const void *A_lo,
                             const void *B_lo) {
  switch (kind) {
    case TcKind::kTF32:
      return launch_kind<TcKind::kTF32>(M, N, K, A, lda, B, ldb, C, ldc, c_vec, num_sms, watchdog,
                                        stream, A_lo, B_lo);
    case TcKind::k3xTF32:
      return launch_kind<TcKind::k3xTF32>(M, N, K, A, lda, B, ldb, C, ldc, c_vec, num_sms,
                                          watchdog, stream, A_lo, B_lo);
    case TcKind::kBF16:
      return launch_kind<TcKind::kBF16>(M, N, K, A, lda, B, ldb, C, ldc, c_vec, num_sms, watchdog,
                                        stream, A_lo, B_lo);
    case TcKind::kF16:
      return launch_kind<TcKind::kF16>(M, N, K, A, lda, B, ldb, C, ldc, c_vec, num_sms, watchdog,
                                       stream, A_lo, B_lo);
    case TcKind::kE4M3:
    case TcKind::kE5M2:
      // 8-bit operands exist only K-major (A as M x K, B as N x K): this unit
      if constexpr (!kUnitAT && kUnitBT) {
        if (kind == TcKind::kE4M3)
          return launch_kind<TcKind::kE4M3>(M, N, K, A, lda, B, ldb, C, ldc, c_vec, num_sms,
                                            watchdog, stream, A_lo, B_lo);
        return launch_kind<TcKind::kE5M2>(M, N, K, A, lda, B, ldb, C, ldc, c_vec, num_sms,
                                          watchdog, stream, A_lo, B_lo);
      }
      return cudaErrorInvalidValue;
  }
  return cudaErrorInvalidValue;
}

#if DGEMM_TC_UNIT == 0
// Device address of this device's watchdog word (looked up once per device).
int *watchdog_address() {
  static std::atomic<int *> addr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  int *a = addr[dev].load(std::memory_order_acquire);
  if (a == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_watchdog) != cudaSuccess) return nullptr;
    a = static_cast<int *>(p);
    addr[dev].store(a, std::memory_order_release);
  }
  return a;
}

bool tc_use_pair(int M, int N, int num_sms) {
  const char *e = getenv("DGEMM_TC_PAIR");
  if (e && e[0] == '0') return false;
  if (e && e[0] == '1') return true;
  const int64_t pair_tiles = (int64_t)((M + 255) / 256) * ((N + 255) / 256);
  return pair_tiles * 4 >= num_sms;
}

cudaError_t launch_tc(TcKind kind, bool a_t, bool b_t, int M, int N, int K, const void *A,
                      int64_t lda, const void *B, int64_t ldb, float *C, int64_t ldc, bool c_vec,
                      int num_sms, cudaStream_t stream, const void *A_lo, const void *B_lo) {
  int *wd = watchdog_address();
  if (wd == nullptr) return cudaErrorInvalidSymbol;
  const int unit = (a_t ? 2 : 0) + (b_t ? 1 : 0);
  switch (unit) {
    case 0:
      return launch_tc_unit_0(kind, M, N, K, A, lda, B, ldb, C, ldc, c_vec, num_sms, wd, stream,
                              A_lo, B_lo);
    case 1:
      return launch_tc_unit_1(kind, M, N, K, A, lda, B, ldb, C, ldc, c_vec, num_sms, wd, stream,
                              A_lo, B_lo);
    case 2:
      return launch_tc_unit_2(kind, M, N, K, A, lda, B, ldb, C, ldc, c_vec, num_sms, wd, stream,
                              A_lo, B_lo);
    default:
      return launch_tc_unit_3(kind, M, N, K, A, lda, B, ldb, C, ldc, c_vec, num_sms, wd, stream,
                              A_lo, B_lo);
  }
}

cudaError_t read_watchdog(cudaStream_t stream, int *code) {
  int *d = nullptr;
  cudaError_t e = scratch_alloc(reinterpret_cast<void **>(&d), sizeof(int), stream);
  if (e != cudaSuccess) return e;
  e = launch_kernel(read_watchdog_kernel, dim3(1), dim3(1), 0, stream, 1, d);
  if (e == cudaSuccess) count_launch();
  int h = 0;
  if (e == cudaSuccess) e = cudaMemcpyAsync(&h, d, sizeof(int), cudaMemcpyDeviceToHost, stream);
  cudaError_t e2 = scratch_free(d, stream);
  if (e == cudaSuccess) e = e2;
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) *code = h;
  return e;
}
#endif

}  // namespace dg
