// api.cu -- the exported C ABI: argument validation, path choice, launch.
//
// Every check that can fail is done on the host before anything is
// enqueued, so an invalid call never launches a kernel.  Order of checks:
//   1. mode (gemm_f32_tc only)                      -> DGEMM_ERR_UNSUPPORTED
//   2. sizes and leading dimensions                 -> DGEMM_ERR_INVALID_VALUE
//   3. M == 0 or N == 0                             -> DGEMM_OK, nothing launched
//   4. NULL pointers where there is work            -> DGEMM_ERR_NULL_POINTER
//   5. pointer alignment to the element size        -> DGEMM_ERR_MISALIGNED
//   6. C overlapping A or B                         -> DGEMM_ERR_ALIAS
//   7. current device is compute capability 10.3    -> DGEMM_ERR_ARCH / DGEMM_ERR_CUDA
//   8. A, B, C are device memory of this device     -> DGEMM_ERR_INVALID_POINTER
// Steps 1-6 touch no CUDA API, so they behave the same on a machine without
// a GPU.
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <cuda_runtime.h>

#include "../../include/dgemm.h"
#include "kernels.h"

namespace dg {
namespace {
std::atomic<unsigned long long> g_launches{0};
}
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
}  // namespace dg

namespace {

thread_local char g_cuda_err[512];

int cuda_fail(cudaError_t e, const char *where) {
  snprintf(g_cuda_err, sizeof g_cuda_err, "%s: %s (%s)", where, cudaGetErrorString(e),
           cudaGetErrorName(e));
  return DGEMM_ERR_CUDA;
}

// Per-device facts, looked up once.  state: 0 unknown, 1 supported, 2 not CC 10.3.
struct DeviceInfo {
  std::atomic<int> state{0};
  int num_sms = 0;
};
constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];

int current_device(int *dev, int *num_sms) {
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (d < 0 || d >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice, "device ordinal");
  DeviceInfo &info = g_devices[d];
  int st = info.state.load(std::memory_order_acquire);
  if (st == 0) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, d)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(major)");
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, d)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(minor)");
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    info.num_sms = sms;
    st = (major == 10 && minor == 3) ? 1 : 2;
    info.state.store(st, std::memory_order_release);
  }
  if (st != 1) return DGEMM_ERR_ARCH;
  *dev = d;
  *num_sms = info.num_sms;
  return DGEMM_OK;
}

// A, B and C must be memory that this device's kernels can address directly.
int check_device_pointer(const void *p, int dev) {
  cudaPointerAttributes at;
  cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();  // the failed query's own, non-sticky error
    return DGEMM_ERR_INVALID_POINTER;
  }
  if (at.type == cudaMemoryTypeManaged) return DGEMM_OK;
  if (at.type == cudaMemoryTypeDevice && at.device == dev) return DGEMM_OK;
  return DGEMM_ERR_INVALID_POINTER;
}

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Byte range [lo, hi) spanned by a rows x cols row-major matrix.
struct Span {
  uintptr_t lo, hi;
};
inline Span span(const void *p, int64_t rows, int64_t cols, int64_t ld, int64_t es) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  if (rows <= 0 || cols <= 0) return {lo, lo};
  return {lo, lo + static_cast<uintptr_t>(((rows - 1) * ld + cols) * es)};
}
inline bool overlap(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }

// Steps 2-8 of the check list.  *nothing_to_do is set when M or N is zero.
// a_t / b_t: A is stored K x M (op(A) = A^T) / B is stored N x K.
int validate(int M, int N, int K, bool a_t, bool b_t, const void *A, int lda, const void *B,
             int ldb, const void *C, int ldc, int in_bytes, bool *nothing_to_do, int *dev,
             int *num_sms) {
  *nothing_to_do = false;
  if (M < 0 || N < 0 || K < 0) return DGEMM_ERR_INVALID_VALUE;
  const int a_rows = a_t ? K : M, a_cols = a_t ? M : K;
  const int b_rows = b_t ? N : K, b_cols = b_t ? K : N;
  if (lda < (a_cols > 1 ? a_cols : 1) || ldb < (b_cols > 1 ? b_cols : 1) ||
      ldc < (N > 1 ? N : 1))
    return DGEMM_ERR_INVALID_VALUE;
  if (M == 0 || N == 0) {
    *nothing_to_do = true;
    return DGEMM_OK;
  }
  if (C == nullptr || (K > 0 && (A == nullptr || B == nullptr))) return DGEMM_ERR_NULL_POINTER;
  if (!aligned(C, 4)) return DGEMM_ERR_MISALIGNED;
  if (K > 0 && (!aligned(A, in_bytes) || !aligned(B, in_bytes))) return DGEMM_ERR_MISALIGNED;
  if (K > 0) {
    const Span c = span(C, M, N, ldc, 4);
    if (overlap(c, span(A, a_rows, a_cols, lda, in_bytes)) ||
        overlap(c, span(B, b_rows, b_cols, ldb, in_bytes)))
      return DGEMM_ERR_ALIAS;
  }
  int st = current_device(dev, num_sms);
  if (st != DGEMM_OK) return st;
  if ((st = check_device_pointer(C, *dev)) != DGEMM_OK) return st;
  if (K > 0) {
    if ((st = check_device_pointer(A, *dev)) != DGEMM_OK) return st;
    if ((st = check_device_pointer(B, *dev)) != DGEMM_OK) return st;
  }
  return DGEMM_OK;
}

}  // namespace

// ------------------------------------------------------------------------
// Scratch: a library-owned stream-ordered memory pool per device.  Freed
// scratch is reused by the next allocations on the stream; at the next
// synchronisation the pool returns what it holds beyond its release threshold
// to the system, so at most kPoolKeepBytes (32 MiB: the re-pitched operands of
// the small workloads, the SIMT tail split's partial tiles at 8192^3) stays
// reserved between calls.  DGEMM_POOL_KEEP_BYTES overrides the bound (read
// once per device, when its pool is created).
namespace dg {
namespace {
constexpr uint64_t kPoolKeepBytes = 32ull << 20;
std::mutex g_pool_mutex;
cudaMemPool_t g_pools[64] = {};

uint64_t pool_keep_bytes() {
  const char *e = getenv("DGEMM_POOL_KEEP_BYTES");
  if (e == nullptr || e[0] < '0' || e[0] > '9') return kPoolKeepBytes;
  return strtoull(e, nullptr, 10);
}
}  // namespace

cudaError_t scratch_alloc(void **ptr, size_t bytes, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaMemPool_t pool;
  {
    std::lock_guard<std::mutex> lock(g_pool_mutex);
    if (g_pools[dev] == nullptr) {
      cudaMemPoolProps props = {};
      props.allocType = cudaMemAllocationTypePinned;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      cudaMemPool_t p = nullptr;
      if ((e = cudaMemPoolCreate(&p, &props)) != cudaSuccess) return e;
      uint64_t keep = pool_keep_bytes();
      if ((e = cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess) {
        cudaMemPoolDestroy(p);
        return e;
      }
      g_pools[dev] = p;
    }
    pool = g_pools[dev];
  }
  return cudaMallocFromPoolAsync(ptr, bytes, pool, stream);
}

cudaError_t scratch_free(void *ptr, cudaStream_t stream) { return cudaFreeAsync(ptr, stream); }
}  // namespace dg

namespace {

int after_launch(cudaError_t e, const char *what) {
  if (e != cudaSuccess) return cuda_fail(e, what);
  return DGEMM_OK;
}

// TMA needs 16-byte aligned bases and row pitches that are multiples of 16 B.
inline bool tma_ok(const void *p, int64_t ld, int es) { return aligned(p, 16) && (ld * es) % 16 == 0; }

inline bool is_f8(dg::TcKind k) { return k == dg::TcKind::kE4M3 || k == dg::TcKind::kE5M2; }

int run_tc(dg::TcKind kind, bool a_t, bool b_t, int M, int N, int K, const void *A, int lda,
           const void *B, int ldb, float *C, int ldc, int num_sms, cudaStream_t stream);

// 8-bit operands: the tensor cores read them K-major only, so A stored K x M
// and B stored K x N are transposed into scratch (A as M x K, B as N x K,
// pitch rounded up to 16 bytes), and a K-major operand whose rows are not
// 16-byte aligned is re-pitched there, both operands in one staging launch.
int run_tc_f8(dg::TcKind kind, bool a_t, bool b_t, int M, int N, int K, const void *A, int lda,
              const void *B, int ldb, float *C, int ldc, int num_sms, cudaStream_t stream) {
  if (!a_t && b_t)
    return run_tc(kind, false, true, M, N, K, A, lda, B, ldb, C, ldc, num_sms, stream);
  const int64_t kp = (K + 15) / 16 * 16;  // K-major pitch of a staged operand
  const bool a_stage = a_t || !tma_ok(A, lda, 1);
  const bool b_stage = !b_t || !tma_ok(B, ldb, 1);
  const size_t a_bytes = a_stage ? (size_t)(((int64_t)M * kp + 255) / 256 * 256) : 0;
  const size_t b_bytes = b_stage ? (size_t)(((int64_t)N * kp + 255) / 256 * 256) : 0;
  void *scratch = nullptr;
  cudaError_t e = dg::scratch_alloc(&scratch, a_bytes + b_bytes, stream);
  if (e != cudaSuccess) return cuda_fail(e, "scratch allocation (8-bit staging)");
  char *s = static_cast<char *>(scratch);
  const void *Ause = A, *Buse = B;
  int lda_use = lda, ldb_use = ldb;
  dg::StageJob jobs[2];
  int njobs = 0;
  if (a_stage) {  // A stored K x M -> M x K, or M x K re-pitched
    jobs[njobs++] = a_t ? dg::StageJob{A, lda, s, kp, K, M, true}
                        : dg::StageJob{A, lda, s, kp, M, K, false};
    Ause = s;
    lda_use = (int)kp;
  }
  if (b_stage) {  // B stored K x N -> N x K, or N x K re-pitched
    jobs[njobs++] = b_t ? dg::StageJob{B, ldb, s + a_bytes, kp, N, K, false}
                        : dg::StageJob{B, ldb, s + a_bytes, kp, K, N, true};
    Buse = s + a_bytes;
    ldb_use = (int)kp;
  }
  e = dg::launch_stage(jobs, njobs, 1, num_sms, stream);
  int st = DGEMM_OK;
  if (e != cudaSuccess)
    st = cuda_fail(e, "8-bit staging launch");
  else
    st = run_tc(kind, false, true, M, N, K, Ause, lda_use, Buse, ldb_use, C, ldc, num_sms, stream);
  const cudaError_t e2 = dg::scratch_free(scratch, stream);
  if (st == DGEMM_OK && e2 != cudaSuccess) return cuda_fail(e2, "scratch release");
  return st;
}

// Tensor-core GEMM with operands re-pitched into stream-ordered scratch when
// their rows do not start on 16-byte boundaries.
int run_tc(dg::TcKind kind, bool a_t, bool b_t, int M, int N, int K, const void *A, int lda,
           const void *B, int ldb, float *C, int ldc, int num_sms, cudaStream_t stream) {
  const int es = is_f8(kind) ? 1
                 : (kind == dg::TcKind::kBF16 || kind == dg::TcKind::kF16) ? 2
                                                                            : 4;
  const int64_t pitch_elems = 16 / es;
  const int a_rows = a_t ? K : M, a_cols = a_t ? M : K;  // storage shapes
  const int b_rows = b_t ? N : K, b_cols = b_t ? K : N;
  const void *Ause = A, *Buse = B;
  int64_t lda_use = lda, ldb_use = ldb;
  void *scratch = nullptr, *lo_scratch = nullptr;
  const bool a_ok = tma_ok(A, lda, es), b_ok = tma_ok(B, ldb, es);
  cudaError_t e = cudaSuccess;
  if (!a_ok || !b_ok) {
    const int64_t lda2 = (a_cols + pitch_elems - 1) / pitch_elems * pitch_elems;
    const int64_t ldb2 = (b_cols + pitch_elems - 1) / pitch_elems * pitch_elems;
    const size_t a_bytes = a_ok ? 0 : (size_t)((int64_t)a_rows * lda2 * es + 255) / 256 * 256;
    const size_t b_bytes = b_ok ? 0 : (size_t)((int64_t)b_rows * ldb2 * es + 255) / 256 * 256;
    e = dg::scratch_alloc(&scratch, a_bytes + b_bytes, stream);
    if (e != cudaSuccess) return cuda_fail(e, "scratch allocation (re-pitch)");
    char *s = static_cast<char *>(scratch);
    dg::StageJob jobs[2];
    int njobs = 0;
    if (!a_ok) {
      jobs[njobs++] = {A, lda, s, lda2, a_rows, a_cols, false};
      Ause = s;
      lda_use = lda2;
    }
    if (!b_ok) {
      jobs[njobs++] = {B, ldb, s + a_bytes, ldb2, b_rows, b_cols, false};
      Buse = s + a_bytes;
      ldb_use = ldb2;
    }
    e = dg::launch_stage(jobs, njobs, es, num_sms, stream);  // both operands, one launch
    if (e != cudaSuccess) goto done;
  }
  {
    // 3xTF32 on the CTA-pair kernel: the split pre-pass writes lo(A) and
    // lo(B) into scratch with the operands' own leading dimensions.  If that
    // scratch cannot be had, the single-CTA kernel splits in shared memory.
    const void *Alo = nullptr, *Blo = nullptr;
    if (kind == dg::TcKind::k3xTF32 && dg::tc_use_pair(M, N, num_sms)) {
      const size_t al = (size_t)(((int64_t)a_rows * lda_use * 4 + 255) / 256 * 256);
      const size_t bl = (size_t)(((int64_t)b_rows * ldb_use * 4 + 255) / 256 * 256);
      if (dg::scratch_alloc(&lo_scratch, al + bl, stream) == cudaSuccess) {
        char *l = static_cast<char *>(lo_scratch);
        e = dg::launch_split_lo(static_cast<const float *>(Ause), lda_use,
                                reinterpret_cast<float *>(l), a_rows, a_cols,
                                static_cast<const float *>(Buse), ldb_use,
                                reinterpret_cast<float *>(l + al), b_rows, b_cols, num_sms,
                                stream);
        if (e != cudaSuccess) goto done;
        Alo = l;
        Blo = l + al;
      } else {
        lo_scratch = nullptr;
        (void)cudaGetLastError();  // the failed allocation is not this call's error
      }
    }
    e = dg::launch_tc(kind, a_t, b_t, M, N, K, Ause, lda_use, Buse, ldb_use, C, ldc,
                      aligned(C, 16) && (ldc % 4) == 0, num_sms, stream, Alo, Blo);
  }
done:
  for (void *p : {lo_scratch, scratch}) {
    if (p == nullptr) continue;
    cudaError_t e2 = dg::scratch_free(p, stream);
    if (e == cudaSuccess && e2 != cudaSuccess) return cuda_fail(e2, "scratch release");
  }
  return after_launch(e, "tensor-core GEMM launch");
}

// ------------------------------------------------------------------------
// Fixed scratch for gemm_f32_tc_noalloc: the re-pitch target of operands
// whose rows do not start on 16-byte boundaries, held by every GPU that loads
// the library.  In host code `g_noalloc_scratch` names a host-side stand-in,
// not the device array: only the address from cudaGetSymbolAddress (looked
// up once per device, with that device current) is passed to kernels.
static __device__ __align__(256) unsigned char g_noalloc_scratch[DGEMM_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mutex;
void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of this device's scratch array (set-up on first use).
int noalloc_scratch(int dev, void **ptr) {
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress (no-alloc scratch)");
    g_noalloc_ptr[dev] = p;
  }
  *ptr = g_noalloc_ptr[dev];
  return DGEMM_OK;
}

// run_tc with the fixed scratch array in place of the scratch pool.
int run_tc_noalloc(dg::TcKind kind, int M, int N, int K, const float *A, int lda, const float *B,
                   int ldb, float *C, int ldc, int dev, int num_sms, cudaStream_t stream) {
  const int es = 4;
  const int64_t pitch_elems = 16 / es;
  const void *Ause = A, *Buse = B;
  int64_t lda_use = lda, ldb_use = ldb;
  const bool a_ok = tma_ok(A, lda, es), b_ok = tma_ok(B, ldb, es);
  cudaError_t e = cudaSuccess;
  uint64_t used = 0;  // bytes of the fixed scratch taken by re-pitched copies
  if (!a_ok || !b_ok) {
    const int64_t lda2 = (K + pitch_elems - 1) / pitch_elems * pitch_elems;
    const int64_t ldb2 = (N + pitch_elems - 1) / pitch_elems * pitch_elems;
    const uint64_t a_bytes = a_ok ? 0 : ((uint64_t)M * lda2 * es + 255) / 256 * 256;
    const uint64_t b_bytes = b_ok ? 0 : ((uint64_t)K * ldb2 * es + 255) / 256 * 256;
    if (a_bytes + b_bytes > (uint64_t)DGEMM_NOALLOC_SCRATCH_BYTES) return DGEMM_ERR_SCRATCH_LIMIT;
    used = a_bytes + b_bytes;
    void *base = nullptr;
    const int st = noalloc_scratch(dev, &base);
    if (st != DGEMM_OK) return st;
    char *s = static_cast<char *>(base);
    dg::StageJob jobs[2];
    int njobs = 0;
    if (!a_ok) {
      jobs[njobs++] = {A, lda, s, lda2, M, K, false};
      Ause = s;
      lda_use = lda2;
    }
    if (!b_ok) {
      jobs[njobs++] = {B, ldb, s + a_bytes, ldb2, K, N, false};
      Buse = s + a_bytes;
      ldb_use = ldb2;
    }
    e = dg::launch_stage(jobs, njobs, es, num_sms, stream);
    if (e != cudaSuccess) return cuda_fail(e, "re-pitch launch (no-alloc)");
  }
  // 3xTF32 on the CTA-pair kernel when the lo parts fit in the rest of the
  // fixed scratch; otherwise the single-CTA kernel splits in shared memory.
  const void *Alo = nullptr, *Blo = nullptr;
  if (kind == dg::TcKind::k3xTF32 && dg::tc_use_pair(M, N, num_sms)) {
    const uint64_t al = ((uint64_t)M * lda_use * 4 + 255) / 256 * 256;
    const uint64_t bl = ((uint64_t)K * ldb_use * 4 + 255) / 256 * 256;
    if (used + al + bl <= (uint64_t)DGEMM_NOALLOC_SCRATCH_BYTES) {
      void *base = nullptr;
      const int st = noalloc_scratch(dev, &base);
      if (st != DGEMM_OK) return st;
      char *l = static_cast<char *>(base) + used;
      e = dg::launch_split_lo(static_cast<const float *>(Ause), lda_use,
                              reinterpret_cast<float *>(l), M, K, static_cast<const float *>(Buse),
                              ldb_use, reinterpret_cast<float *>(l + al), K, N, num_sms, stream);
      if (e != cudaSuccess) return cuda_fail(e, "split pre-pass launch (no-alloc)");
      Alo = l;
      Blo = l + al;
    }
  }
  e = dg::launch_tc(kind, false, false, M, N, K, Ause, lda_use, Buse, ldb_use, C, ldc,
                    aligned(C, 16) && (ldc % 4) == 0, num_sms, stream, Alo, Blo);
  return after_launch(e, "tensor-core GEMM launch (no-alloc)");
}

}  // namespace

extern "C" {

int gemm_f32_tc_noalloc(int mode, int M, int N, int K, const float *A, int lda, const float *B,
                        int ldb, float *C, int ldc, cudaStream_t stream) {
  if (mode != DGEMM_TC_TF32 && mode != DGEMM_TC_3XTF32) return DGEMM_ERR_UNSUPPORTED;
  bool none = false;
  int dev = 0, sms = 0;
  int st = validate(M, N, K, false, false, A, lda, B, ldb, C, ldc, 4, &none, &dev, &sms);
  if (st != DGEMM_OK || none) return st;
  if (K == 0) return after_launch(dg::launch_zero_fill(C, M, N, ldc, sms, stream), "zero fill");
  return run_tc_noalloc(mode == DGEMM_TC_TF32 ? dg::TcKind::kTF32 : dg::TcKind::k3xTF32, M, N, K,
                        A, lda, B, ldb, C, ldc, dev, sms, stream);
}

int gemm_f32_simt(int M, int N, int K, const float *A, int lda, const float *B, int ldb,
                  float *C, int ldc, cudaStream_t stream) {
  bool none = false;
  int dev = 0, sms = 0;
  int st = validate(M, N, K, false, false, A, lda, B, ldb, C, ldc, 4, &none, &dev, &sms);
  if (st != DGEMM_OK || none) return st;
  if (K == 0) return after_launch(dg::launch_zero_fill(C, M, N, ldc, sms, stream), "zero fill");
  const bool ab_vec = aligned(A, 16) && aligned(B, 16) && lda % 4 == 0 && ldb % 4 == 0;
  const bool c_vec = aligned(C, 16) && ldc % 4 == 0;
  return after_launch(
      dg::launch_simt(false, false, M, N, K, A, lda, B, ldb, C, ldc, ab_vec, c_vec, sms, stream),
      "SIMT GEMM launch");
}

int gemm_f32_tc(int mode, int M, int N, int K, const float *A, int lda, const float *B, int ldb,
                float *C, int ldc, cudaStream_t stream) {
  if (mode != DGEMM_TC_TF32 && mode != DGEMM_TC_3XTF32) return DGEMM_ERR_UNSUPPORTED;
  bool none = false;
  int dev = 0, sms = 0;
  int st = validate(M, N, K, false, false, A, lda, B, ldb, C, ldc, 4, &none, &dev, &sms);
  if (st != DGEMM_OK || none) return st;
  if (K == 0) return after_launch(dg::launch_zero_fill(C, M, N, ldc, sms, stream), "zero fill");
  return run_tc(mode == DGEMM_TC_TF32 ? dg::TcKind::kTF32 : dg::TcKind::k3xTF32, false, false, M,
                N, K, A, lda, B, ldb, C, ldc, sms, stream);
}

int gemm_bf16_tc(int M, int N, int K, const unsigned short *A, int lda, const unsigned short *B,
                 int ldb, float *C, int ldc, cudaStream_t stream) {
  bool none = false;
  int dev = 0, sms = 0;
  int st = validate(M, N, K, false, false, A, lda, B, ldb, C, ldc, 2, &none, &dev, &sms);
  if (st != DGEMM_OK || none) return st;
  if (K == 0) return after_launch(dg::launch_zero_fill(C, M, N, ldc, sms, stream), "zero fill");
  return run_tc(dg::TcKind::kBF16, false, false, M, N, K, A, lda, B, ldb, C, ldc, sms, stream);
}

int gemm_f16_tc(int M, int N, int K, const unsigned short *A, int lda, const unsigned short *B,
                int ldb, float *C, int ldc, cudaStream_t stream) {
  bool none = false;
  int dev = 0, sms = 0;
  int st = validate(M, N, K, false, false, A, lda, B, ldb, C, ldc, 2, &none, &dev, &sms);
  if (st != DGEMM_OK || none) return st;
  if (K == 0) return after_launch(dg::launch_zero_fill(C, M, N, ldc, sms, stream), "zero fill");
  return run_tc(dg::TcKind::kF16, false, false, M, N, K, A, lda, B, ldb, C, ldc, sms, stream);
}

int gemm_f8_tc(int format, int M, int N, int K, const unsigned char *A, int lda,
               const unsigned char *B, int ldb, float *C, int ldc, cudaStream_t stream) {
  if (format != DGEMM_F8_E4M3 && format != DGEMM_F8_E5M2) return DGEMM_ERR_UNSUPPORTED;
  bool none = false;
  int dev = 0, sms = 0;
  int st = validate(M, N, K, false, false, A, lda, B, ldb, C, ldc, 1, &none, &dev, &sms);
  if (st != DGEMM_OK || none) return st;
  if (K == 0) return after_launch(dg::launch_zero_fill(C, M, N, ldc, sms, stream), "zero fill");
  return run_tc_f8(format == DGEMM_F8_E4M3 ? dg::TcKind::kE4M3 : dg::TcKind::kE5M2, false, false,
                   M, N, K, A, lda, B, ldb, C, ldc, sms, stream);
}

int dgemm_gemm_ex(int path, int op_a, int op_b, int M, int N, int K, const void *A, int lda,
                  const void *B, int ldb, float *C, int ldc, cudaStream_t stream) {
  if (path < DGEMM_PATH_SIMT || path > DGEMM_PATH_F8_E5M2) return DGEMM_ERR_UNSUPPORTED;
  if ((op_a != DGEMM_OP_N && op_a != DGEMM_OP_T) || (op_b != DGEMM_OP_N && op_b != DGEMM_OP_T))
    return DGEMM_ERR_UNSUPPORTED;
  const bool a_t = op_a == DGEMM_OP_T, b_t = op_b == DGEMM_OP_T;
  const bool f8 = path == DGEMM_PATH_F8_E4M3 || path == DGEMM_PATH_F8_E5M2;
  const int es = f8 ? 1 : (path == DGEMM_PATH_BF16 || path == DGEMM_PATH_FP16) ? 2 : 4;
  bool none = false;
  int dev = 0, sms = 0;
  int st = validate(M, N, K, a_t, b_t, A, lda, B, ldb, C, ldc, es, &none, &dev, &sms);
  if (st != DGEMM_OK || none) return st;
  if (K == 0) return after_launch(dg::launch_zero_fill(C, M, N, ldc, sms, stream), "zero fill");
  if (path == DGEMM_PATH_SIMT) {
    const bool ab_vec = aligned(A, 16) && aligned(B, 16) && lda % 4 == 0 && ldb % 4 == 0;
    const bool c_vec = aligned(C, 16) && ldc % 4 == 0;
    return after_launch(dg::launch_simt(a_t, b_t, M, N, K, static_cast<const float *>(A), lda,
                                        static_cast<const float *>(B), ldb, C, ldc, ab_vec,
                                        c_vec, sms, stream),
                        "SIMT GEMM launch");
  }
  if (f8)
    return run_tc_f8(path == DGEMM_PATH_F8_E4M3 ? dg::TcKind::kE4M3 : dg::TcKind::kE5M2, a_t, b_t,
                     M, N, K, A, lda, B, ldb, C, ldc, sms, stream);
  const dg::TcKind kind = path == DGEMM_PATH_TF32    ? dg::TcKind::kTF32
                          : path == DGEMM_PATH_3XTF32 ? dg::TcKind::k3xTF32
                          : path == DGEMM_PATH_BF16   ? dg::TcKind::kBF16
                                                      : dg::TcKind::kF16;
  return run_tc(kind, a_t, b_t, M, N, K, A, lda, B, ldb, C, ldc, sms, stream);
}

const char *dgemm_status_string(int status) {
  switch (status) {
    case DGEMM_OK: return "success";
    case DGEMM_ERR_INVALID_VALUE: return "invalid value: negative size or leading dimension too small";
    case DGEMM_ERR_NULL_POINTER: return "null pointer for A, B or C";
    case DGEMM_ERR_ALIAS: return "C overlaps A or B";
    case DGEMM_ERR_UNSUPPORTED: return "unsupported mode";
    case DGEMM_ERR_CUDA: return "CUDA error (see dgemm_last_cuda_error)";
    case DGEMM_ERR_ARCH: return "current device is not compute capability 10.3 (sm_103a)";
    case DGEMM_ERR_MISALIGNED: return "pointer not aligned to its element size";
    case DGEMM_ERR_INVALID_POINTER: return "A, B or C is not device memory of the current device";
    case DGEMM_ERR_WATCHDOG: return "a kernel gave up a bounded wait; its output is incomplete";
    case DGEMM_ERR_SCRATCH_LIMIT:
      return "operands need more re-pitch scratch than gemm_f32_tc_noalloc's fixed 16 MiB; "
             "use gemm_f32_tc";
    default: return "unknown status";
  }
}

const char *dgemm_last_cuda_error(void) { return g_cuda_err; }

int dgemm_watchdog_status(cudaStream_t stream, int *where) {
  int code = 0;
  cudaError_t e = dg::read_watchdog(stream, &code);
  if (e != cudaSuccess) return cuda_fail(e, "watchdog read");
  if (where) *where = code;
  return code ? DGEMM_ERR_WATCHDOG : DGEMM_OK;
}

int dgemm_version(void) { return 100; }

unsigned long long dgemm_kernel_launches(void) {
  return dg::g_launches.load(std::memory_order_relaxed);
}

}  // extern "C"
