"""ctypes binding of libdgemm.so: the C entry points under the same names.

Argument marshalling only -- every step of the product runs in the library's
CUDA kernels.  Pointers are integers (device addresses), `stream` is a
cudaStream_t handle as an integer (0 = legacy default stream).  Each function
returns the library's status code; see include/dgemm.h for the semantics.
"""
import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdgemm.so")

# Status codes (dgemm_status_t in include/dgemm.h).
OK = 0
ERR_INVALID_VALUE = 1
ERR_NULL_POINTER = 2
ERR_ALIAS = 3
ERR_UNSUPPORTED = 4
ERR_CUDA = 5
ERR_ARCH = 6
ERR_MISALIGNED = 7
ERR_INVALID_POINTER = 8
ERR_WATCHDOG = 9
ERR_SCRATCH_LIMIT = 10
NOALLOC_SCRATCH_BYTES = 16 << 20

TC_TF32 = 0
TC_3XTF32 = 1

OP_N = 0
OP_T = 1
PATH_SIMT, PATH_TF32, PATH_3XTF32, PATH_BF16, PATH_FP16, PATH_F8_E4M3, PATH_F8_E5M2 = range(7)
F8_E4M3 = 0
F8_E5M2 = 1

EXPORTED = ("gemm_f32_simt", "gemm_f32_tc", "gemm_bf16_tc", "dgemm_status_string",
            "dgemm_last_cuda_error", "dgemm_watchdog_status", "dgemm_version",
            "dgemm_kernel_launches", "gemm_f32_tc_noalloc", "gemm_f16_tc", "dgemm_gemm_ex",
            "gemm_f8_tc")

_lib = None


class LibraryMissing(RuntimeError):
    pass


def load():
    """Load libdgemm.so (built by dense_gemm_f32_gb300.build); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise LibraryMissing(
            f"{LIB_PATH} is missing: build it first with "
            "`python -c 'import __graft_entry__ as g; g.build()'` "
            "(there is no fallback implementation)")
    lib = ctypes.CDLL(LIB_PATH)
    i, p = ctypes.c_int, ctypes.c_void_p
    gemm_args = [i, i, i, p, i, p, i, p, i, p]
    lib.gemm_f32_simt.argtypes = gemm_args
    lib.gemm_f32_simt.restype = i
    lib.gemm_f32_tc.argtypes = [i] + gemm_args
    lib.gemm_f32_tc.restype = i
    lib.gemm_bf16_tc.argtypes = gemm_args
    lib.gemm_bf16_tc.restype = i
    lib.dgemm_status_string.argtypes = [i]
    lib.dgemm_status_string.restype = ctypes.c_char_p
    lib.dgemm_last_cuda_error.argtypes = []
    lib.dgemm_last_cuda_error.restype = ctypes.c_char_p
    lib.dgemm_watchdog_status.argtypes = [p, ctypes.POINTER(ctypes.c_int)]
    lib.dgemm_watchdog_status.restype = i
    lib.dgemm_version.argtypes = []
    lib.dgemm_version.restype = i
    lib.dgemm_kernel_launches.argtypes = []
    lib.dgemm_kernel_launches.restype = ctypes.c_ulonglong
    lib.gemm_f32_tc_noalloc.argtypes = [i] + gemm_args
    lib.gemm_f32_tc_noalloc.restype = i
    lib.gemm_f16_tc.argtypes = gemm_args
    lib.gemm_f16_tc.restype = i
    lib.dgemm_gemm_ex.argtypes = [i, i, i] + gemm_args
    lib.dgemm_gemm_ex.restype = i
    lib.gemm_f8_tc.argtypes = [i] + gemm_args
    lib.gemm_f8_tc.restype = i
    _lib = lib
    return lib


def gemm_f32_simt(M, N, K, A, lda, B, ldb, C, ldc, stream=0):
    return load().gemm_f32_simt(M, N, K, A, lda, B, ldb, C, ldc, stream)


def gemm_f32_tc(mode, M, N, K, A, lda, B, ldb, C, ldc, stream=0):
    return load().gemm_f32_tc(mode, M, N, K, A, lda, B, ldb, C, ldc, stream)


def gemm_f32_tc_noalloc(mode, M, N, K, A, lda, B, ldb, C, ldc, stream=0):
    """gemm_f32_tc without allocating: re-pitch scratch is the library's fixed
    16 MiB device array (see include/dgemm.h)."""
    return load().gemm_f32_tc_noalloc(mode, M, N, K, A, lda, B, ldb, C, ldc, stream)


def gemm_bf16_tc(M, N, K, A, lda, B, ldb, C, ldc, stream=0):
    return load().gemm_bf16_tc(M, N, K, A, lda, B, ldb, C, ldc, stream)


def gemm_f16_tc(M, N, K, A, lda, B, ldb, C, ldc, stream=0):
    return load().gemm_f16_tc(M, N, K, A, lda, B, ldb, C, ldc, stream)


def gemm_f8_tc(fmt, M, N, K, A, lda, B, ldb, C, ldc, stream=0):
    return load().gemm_f8_tc(fmt, M, N, K, A, lda, B, ldb, C, ldc, stream)


def dgemm_gemm_ex(path, op_a, op_b, M, N, K, A, lda, B, ldb, C, ldc, stream=0):
    return load().dgemm_gemm_ex(path, op_a, op_b, M, N, K, A, lda, B, ldb, C, ldc, stream)


def dgemm_status_string(status):
    return load().dgemm_status_string(status).decode()


def dgemm_last_cuda_error():
    return load().dgemm_last_cuda_error().decode()


def dgemm_watchdog_status(stream=0):
    """(status, site code)."""
    where = ctypes.c_int(0)
    st = load().dgemm_watchdog_status(stream, ctypes.byref(where))
    return st, where.value


def dgemm_version():
    return load().dgemm_version()


def dgemm_kernel_launches():
    return load().dgemm_kernel_launches()
