"""The C ABI without a GPU: the library loads, exports every entry point that
include/dgemm.h declares, and rejects invalid calls on the host before any
CUDA call (the validation order is documented in csrc/api.cu)."""
import ctypes
import os
import re

import pytest

import dense_gemm_f32_gb300 as dg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "dgemm.h"), encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = "\n".join(ln for ln in text.splitlines() if not ln.lstrip().startswith("#"))
    return sorted(set(re.findall(r"(\w+)\s*\([^;{}]*\)\s*;", text)))


@pytest.fixture(scope="module")
def lib():
    from dense_gemm_f32_gb300 import build

    build.build()
    return dg.load()


def test_header_declares_the_documented_entry_points():
    assert _declared_functions() == sorted(dg.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"libdgemm.so does not export {name}"
        ctypes.cast(getattr(lib, name), ctypes.c_void_p)


def test_status_strings_and_version(lib):
    for st in range(0, 11):
        s = dg.dgemm_status_string(st)
        assert s and s != "unknown status"
    assert dg.dgemm_status_string(99) == "unknown status"
    assert dg.dgemm_version() >= 100


P = 0x10000  # a fake, 16-byte aligned address: never dereferenced by these calls


@pytest.mark.parametrize("fn", ["simt", "tf32", "3xtf32", "bf16", "fp16", "noalloc-tf32", "noalloc-3xtf32"])
def test_invalid_sizes_rejected(lib, fn):
    call = _caller(fn)
    E = dg.ERR_INVALID_VALUE
    assert call(-1, 4, 4, P, 4, P * 2, 4, P * 3, 4) == E
    assert call(4, -1, 4, P, 4, P * 2, 4, P * 3, 4) == E
    assert call(4, 4, -1, P, 4, P * 2, 4, P * 3, 4) == E
    assert call(4, 4, 8, P, 7, P * 2, 4, P * 3, 4) == E     # lda < K
    assert call(4, 8, 4, P, 4, P * 2, 7, P * 3, 8) == E     # ldb < N
    assert call(4, 8, 4, P, 4, P * 2, 8, P * 3, 7) == E     # ldc < N
    assert call(4, 4, 0, P, 0, P * 2, 4, P * 3, 4) == E     # lda must be >= 1


@pytest.mark.parametrize("fn", ["simt", "tf32", "3xtf32", "bf16", "fp16", "noalloc-tf32", "noalloc-3xtf32"])
def test_empty_output_is_a_no_op(lib, fn):
    call = _caller(fn)
    # nothing to do: pointers are not looked at, no CUDA call is made
    assert call(0, 5, 5, 0, 5, 0, 5, 0, 5) == dg.OK
    assert call(5, 0, 5, 0, 5, 0, 1, 0, 1) == dg.OK


@pytest.mark.parametrize("fn", ["simt", "tf32", "3xtf32", "bf16", "fp16", "noalloc-tf32", "noalloc-3xtf32"])
def test_null_pointers_rejected(lib, fn):
    call = _caller(fn)
    E = dg.ERR_NULL_POINTER
    assert call(4, 4, 4, 0, 4, P, 4, P * 4, 4) == E
    assert call(4, 4, 4, P, 4, 0, 4, P * 4, 4) == E
    assert call(4, 4, 4, P, 4, P * 2, 4, 0, 4) == E
    assert call(4, 4, 0, P, 1, P * 2, 4, 0, 4) == E       # K == 0 still writes C


@pytest.mark.parametrize("fn", ["simt", "tf32", "3xtf32", "bf16", "fp16", "noalloc-tf32", "noalloc-3xtf32"])
def test_misaligned_pointers_rejected(lib, fn):
    call = _caller(fn)
    es = 2 if fn in ("bf16", "fp16") else 4
    E = dg.ERR_MISALIGNED
    assert call(4, 4, 4, P + 1, 4, P * 2, 4, P * 4, 4) == E
    assert call(4, 4, 4, P, 4, P * 2 + 1, 4, P * 4, 4) == E
    assert call(4, 4, 4, P, 4, P * 2, 4, P * 4 + 2, 4) == E   # C is fp32: 4-byte aligned
    if es == 4:
        assert call(4, 4, 4, P + 2, 4, P * 2, 4, P * 4, 4) == E


@pytest.mark.parametrize("fn", ["simt", "tf32", "3xtf32", "bf16", "fp16", "noalloc-tf32", "noalloc-3xtf32"])
def test_alias_rejected(lib, fn):
    call = _caller(fn)
    es = 2 if fn in ("bf16", "fp16") else 4
    E = dg.ERR_ALIAS
    # C starts inside A's span / B's span
    assert call(8, 8, 8, P, 8, P * 4, 8, P + 8 * 8 * es - 4, 8) == E
    assert call(8, 8, 8, P, 8, P * 4, 8, P * 4 + 16, 8) == E
    # A inside C's span
    assert call(8, 8, 8, P * 4 + 64, 8, P * 8, 8, P * 4, 8) == E


@pytest.mark.parametrize("fn", ["gemm_f32_tc", "gemm_f32_tc_noalloc"])
def test_unknown_mode_rejected(lib, fn):
    f = getattr(dg, fn)
    assert f(7, 4, 4, 4, P, 4, P * 2, 4, P * 4, 4, 0) == dg.ERR_UNSUPPORTED
    assert f(-1, 4, 4, 4, P, 4, P * 2, 4, P * 4, 4, 0) == dg.ERR_UNSUPPORTED
    # the mode is checked before anything else, even with sizes that are invalid too
    assert f(2, -1, 4, 4, P, 4, P * 2, 4, P * 4, 4, 0) == dg.ERR_UNSUPPORTED


def test_scratch_limit_status_names_the_limit(lib):
    s = dg.dgemm_status_string(dg.ERR_SCRATCH_LIMIT)
    assert "16 MiB" in s and "gemm_f32_tc_noalloc" in s
    assert dg.NOALLOC_SCRATCH_BYTES == 16 << 20


def test_matmul_argument_checks_need_no_gpu():
    import torch

    with pytest.raises(ValueError):
        dg.matmul(torch.zeros(2, 3), torch.zeros(3, 2), mode="fp64")
    with pytest.raises(TypeError):
        dg.matmul(torch.zeros(2, 3), torch.zeros(3, 2, dtype=torch.float64), mode="simt")
    with pytest.raises(ValueError):
        dg.matmul(torch.zeros(2, 3), torch.zeros(4, 2), mode="simt")


def test_watchdog_site_codes_documented():
    """Every bounded wait of every kernel has its own site code, across files."""
    codes = []
    for f in ("tc.cu", "simt.cu"):
        src = open(os.path.join(ROOT, "dense_gemm_f32_gb300", "csrc", f), encoding="utf-8").read()
        codes += re.findall(r"kSite\w+ = (0x[0-9a-f]+)", src)
    assert len(codes) == len(set(codes)) >= 9


def _caller(fn):
    if fn == "simt":
        return lambda *a: dg.gemm_f32_simt(*a, 0)
    if fn == "tf32":
        return lambda *a: dg.gemm_f32_tc(dg.TC_TF32, *a, 0)
    if fn == "3xtf32":
        return lambda *a: dg.gemm_f32_tc(dg.TC_3XTF32, *a, 0)
    if fn == "fp16":
        return lambda *a: dg.gemm_f16_tc(*a, 0)
    if fn == "noalloc-tf32":
        return lambda *a: dg.gemm_f32_tc_noalloc(dg.TC_TF32, *a, 0)
    if fn == "noalloc-3xtf32":
        return lambda *a: dg.gemm_f32_tc_noalloc(dg.TC_3XTF32, *a, 0)
    return lambda *a: dg.gemm_bf16_tc(*a, 0)


@pytest.mark.parametrize("path", range(5))
def test_gemm_ex_leading_dimensions_follow_the_stored_shape(lib, path):
    """op_a = T: A is stored K x M, so lda >= M; op_b = T: B is N x K, ldb >= K."""
    call = lambda oa, ob, *a: dg.dgemm_gemm_ex(path, oa, ob, *a, 0)  # noqa: E731
    E = dg.ERR_INVALID_VALUE
    N_, T_ = dg.OP_N, dg.OP_T
    # M=8, N=16, K=4: A^T stored 4 x 8 needs lda >= 8; B^T stored 16 x 4 needs ldb >= 4
    assert call(T_, N_, 8, 16, 4, P, 4, P * 2, 16, P * 4, 16) == E
    assert call(N_, T_, 8, 16, 4, P, 4, P * 2, 3, P * 4, 16) == E
    assert call(N_, N_, 8, 16, 4, P, 3, P * 2, 16, P * 4, 16) == E
    # C overlapping A's stored span (4 rows of 8 when transposed)
    es = 2 if path >= 3 else 4
    assert call(T_, N_, 8, 16, 4, P, 8, P * 4, 16, P + 2 * 8 * es, 16) == dg.ERR_ALIAS


def test_gemm_ex_rejects_unknown_path_or_op(lib):
    assert dg.dgemm_gemm_ex(7, 0, 0, 4, 4, 4, P, 4, P * 2, 4, P * 4, 4, 0) == dg.ERR_UNSUPPORTED
    assert dg.dgemm_gemm_ex(-1, 0, 0, 4, 4, 4, P, 4, P * 2, 4, P * 4, 4, 0) == dg.ERR_UNSUPPORTED
    assert dg.dgemm_gemm_ex(1, 2, 0, 4, 4, 4, P, 4, P * 2, 4, P * 4, 4, 0) == dg.ERR_UNSUPPORTED
    assert dg.dgemm_gemm_ex(1, 0, -1, 4, 4, 4, P, 4, P * 2, 4, P * 4, 4, 0) == dg.ERR_UNSUPPORTED
    assert dg.dgemm_gemm_ex(1, 0, 1, 0, 4, 4, 0, 4, 0, 4, 0, 4, 0) == dg.OK


def test_f8_rejects_unknown_format_and_checks_arguments(lib):
    """gemm_f8_tc: unknown format first, then the common checks (element
    alignment is one byte, so any address is aligned)."""
    assert dg.gemm_f8_tc(2, 4, 4, 4, P, 4, P * 2, 4, P * 4, 4, 0) == dg.ERR_UNSUPPORTED
    assert dg.gemm_f8_tc(-1, 4, 4, 4, P, 4, P * 2, 4, P * 4, 4, 0) == dg.ERR_UNSUPPORTED
    assert dg.gemm_f8_tc(dg.F8_E4M3, 4, 4, 4, P, 3, P * 2, 4, P * 4, 4, 0) == dg.ERR_INVALID_VALUE
    assert dg.gemm_f8_tc(dg.F8_E5M2, 4, 4, 4, 0, 4, P * 2, 4, P * 4, 4, 0) == dg.ERR_NULL_POINTER
    assert dg.gemm_f8_tc(dg.F8_E4M3, 0, 4, 4, 0, 4, 0, 4, 0, 4, 0) == dg.OK
    # C overlapping B
    assert dg.gemm_f8_tc(dg.F8_E4M3, 4, 4, 4, P + 1, 4, P * 2 + 1, 4, P * 2 + 4, 4, 0) == dg.ERR_ALIAS
    # the FP8 paths of dgemm_gemm_ex validate the transposed storage shapes
    assert dg.dgemm_gemm_ex(dg.PATH_F8_E4M3, dg.OP_T, dg.OP_N, 4, 8, 2, P, 3, P * 2, 8,
                            P * 4, 8, 0) == dg.ERR_INVALID_VALUE


def test_matmul_transposed_shape_checks_need_no_gpu():
    import torch

    with pytest.raises(ValueError):
        dg.matmul(torch.zeros(3, 2), torch.zeros(3, 4), mode="simt", trans_a=False)
