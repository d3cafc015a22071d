"""GB300-native dense GEMM: C = A x B, row-major, on sm_103a.

The library is the C ABI in include/dgemm.h (libdgemm.so, built from csrc/ by
`build.py`).  This package binds it with ctypes under the same names
(`gemm_f32_simt`, `gemm_f32_tc`, `gemm_bf16_tc`, ...: raw device pointers,
status codes) and adds `matmul`, a convenience over torch CUDA tensors that
only derives pointers, leading dimensions and the stream, allocates C, and
raises on a non-zero status.  PyTorch is used for device memory and streams;
all arithmetic runs in the library's kernels.  There is no fallback: without
libdgemm.so every call raises.
"""
from ._lib import (  # noqa: F401  (re-exported C entry points)
    ERR_ALIAS, ERR_ARCH, ERR_CUDA, ERR_INVALID_POINTER, ERR_INVALID_VALUE, ERR_MISALIGNED,
    ERR_NULL_POINTER, ERR_SCRATCH_LIMIT, ERR_UNSUPPORTED, ERR_WATCHDOG, EXPORTED, F8_E4M3,
    F8_E5M2, LIB_PATH, NOALLOC_SCRATCH_BYTES, OK, OP_N, OP_T, PATH_3XTF32, PATH_BF16,
    PATH_F8_E4M3, PATH_F8_E5M2, PATH_FP16, PATH_SIMT, PATH_TF32, TC_3XTF32, TC_TF32,
    LibraryMissing, dgemm_gemm_ex, dgemm_kernel_launches, dgemm_last_cuda_error,
    dgemm_status_string, dgemm_version, dgemm_watchdog_status, gemm_bf16_tc, gemm_f16_tc,
    gemm_f32_simt, gemm_f32_tc, gemm_f32_tc_noalloc, gemm_f8_tc, load,
)

MODES = ("simt", "tf32", "3xtf32", "bf16", "fp16", "e4m3", "e5m2")


class DgemmError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        msg = dgemm_status_string(status)
        if status == ERR_CUDA:
            msg += ": " + dgemm_last_cuda_error()
        super().__init__(f"{what}: {msg}" if what else msg)


def check(status, what=""):
    if status != OK:
        raise DgemmError(status, what)


def _ld(X, cols):
    """Leading dimension (elements) of a 2-D row-major tensor view."""
    if X.dim() != 2:
        raise ValueError("expected a 2-D matrix")
    rows = X.shape[0]
    if cols > 1 and X.stride(1) != 1:
        raise ValueError("rows must be contiguous (stride(1) == 1)")
    if rows <= 1:
        return max(cols, 1)
    return X.stride(0)


_PATH = {"simt": PATH_SIMT, "tf32": PATH_TF32, "3xtf32": PATH_3XTF32, "bf16": PATH_BF16,
         "fp16": PATH_FP16, "e4m3": PATH_F8_E4M3, "e5m2": PATH_F8_E5M2}


def input_dtype(mode):
    """The torch dtype of A and B for a mode."""
    import torch

    return {"bf16": torch.bfloat16, "fp16": torch.float16, "e4m3": torch.float8_e4m3fn,
            "e5m2": torch.float8_e5m2}.get(mode, torch.float32)


def matmul(A, B, mode="tf32", out=None, stream=None, trans_a=False, trans_b=False):
    """C = op(A) @ op(B) on the GPU through the C ABI.

    A, B: CUDA tensors as stored, float32 for modes simt / tf32 / 3xtf32,
    bfloat16 for mode bf16, float16 for mode fp16, float8_e4m3fn / float8_e5m2
    for modes e4m3 / e5m2; rows may be strided
    (leading dimension = stride(0)).  op(A) = A.T when trans_a (A stored
    K x M), else A (M x K); op(B) = B.T when trans_b (B stored N x K), else B.
    out: optional float32 (M, N) CUDA tensor view to overwrite.
    stream: a torch.cuda.Stream or raw handle; default the current stream.
    """
    import torch

    if mode not in MODES:
        raise ValueError(f"mode must be one of {MODES}")
    want = input_dtype(mode)
    if A.dtype != want or B.dtype != want:
        raise TypeError(f"mode {mode} takes {want} inputs, got {A.dtype} and {B.dtype}")
    if A.dim() != 2 or B.dim() != 2:
        raise ValueError("expected 2-D matrices")
    M, K = (A.shape[1], A.shape[0]) if trans_a else (A.shape[0], A.shape[1])
    K2, N = (B.shape[1], B.shape[0]) if trans_b else (B.shape[0], B.shape[1])
    if K != K2:
        raise ValueError(f"inner dimensions differ: op(A) is {M}x{K}, op(B) is {K2}x{N}")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    elif out.dtype != torch.float32 or tuple(out.shape) != (M, N):
        raise ValueError("out must be a float32 (M, N) tensor")
    if stream is None:
        stream = torch.cuda.current_stream(A.device).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    lda, ldb, ldc = _ld(A, A.shape[1]), _ld(B, B.shape[1]), _ld(out, N)
    pa, pb, pc = A.data_ptr(), B.data_ptr(), out.data_ptr()
    if trans_a or trans_b:
        st = dgemm_gemm_ex(_PATH[mode], OP_T if trans_a else OP_N, OP_T if trans_b else OP_N,
                           M, N, K, pa, lda, pb, ldb, pc, ldc, stream)
    elif mode == "simt":
        st = gemm_f32_simt(M, N, K, pa, lda, pb, ldb, pc, ldc, stream)
    elif mode == "tf32":
        st = gemm_f32_tc(TC_TF32, M, N, K, pa, lda, pb, ldb, pc, ldc, stream)
    elif mode == "3xtf32":
        st = gemm_f32_tc(TC_3XTF32, M, N, K, pa, lda, pb, ldb, pc, ldc, stream)
    elif mode == "bf16":
        st = gemm_bf16_tc(M, N, K, pa, lda, pb, ldb, pc, ldc, stream)
    elif mode == "fp16":
        st = gemm_f16_tc(M, N, K, pa, lda, pb, ldb, pc, ldc, stream)
    else:
        st = gemm_f8_tc(F8_E4M3 if mode == "e4m3" else F8_E5M2, M, N, K, pa, lda, pb, ldb, pc,
                        ldc, stream)
    check(st, f"gemm ({mode})")
    return out
