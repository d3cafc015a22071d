"""gemm_f32_tc_noalloc, the entry point for callers that cannot allocate.

Some callers must not allocate device memory during a call: a process that
reserved all of HBM up front, code running inside an allocator callback, a
latency-critical loop that cannot afford an allocation failing mid-run.  For
them the library keeps a fixed 16 MiB scratch array on each GPU and
gemm_f32_tc_noalloc re-pitches unaligned operands into it instead of calling
cudaMallocAsync.  These tests call it through the C ABI and check that it
gives what gemm_f32_tc gives (bit for bit wherever both run the same kernel,
within the tolerances the other tests use otherwise) and what the CPU oracle
gives, on two calls in a row (the second with different inputs, so that a
stale scratch would show), and that it refuses operands that do not fit.

This file is collected last on purpose; it also passes when run on its own.
"""
import numpy as np
import pytest
import torch

import gpu_util as gu
from dense_gemm_f32_gb300 import inputs
import dense_gemm_f32_gb300 as dg

pytestmark = pytest.mark.gpu

MODES = {"tf32": dg.TC_TF32, "3xtf32": dg.TC_3XTF32}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _call(fn, mode, A, B, C, stream):
    M, K = A.shape
    N = B.shape[1]
    return fn(MODES[mode], M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0),
              C.data_ptr(), C.stride(0), stream)


def _pair(mode, A, B):
    """(existing entry point's C, no-alloc entry point's C) on the same inputs."""
    stream = torch.cuda.current_stream().cuda_stream
    M, N = A.shape[0], B.shape[1]
    C_ref = torch.full((M, N), float("nan"), device="cuda")
    C_new = torch.full((M, N), float("nan"), device="cuda")
    assert _call(dg.gemm_f32_tc, mode, A, B, C_ref, stream) == dg.OK
    assert _call(dg.gemm_f32_tc_noalloc, mode, A, B, C_new, stream) == dg.OK
    torch.cuda.synchronize()
    return C_ref.cpu().numpy(), C_new.cpu().numpy()


def _s(A, B):
    import oracle

    return oracle.abs_gemm(A.float().cpu().numpy(), B.float().cpu().numpy())


def _oracle(A, B):
    import oracle

    return oracle.gemm(A.float().cpu().numpy(), B.float().cpu().numpy())


@pytest.mark.parametrize("mode", ["tf32", "3xtf32"])
def test_matches_existing_entry_point_on_two_calls(mode):
    """Ragged shapes with rows that are not 16-byte aligned, so both operands
    go through the fixed scratch; two calls in a row with different inputs."""
    shapes = [(1000, 1013, 997, 2), (333, 517, 259, 5)]
    for (M, N, K, seed) in shapes:
        A, B = inputs.make_random(M, N, K, seed=seed, dist="normal")
        Ad, Bd = A.cuda(), B.cuda()
        ref, new = _pair(mode, Ad, Bd)
        assert np.isfinite(new).all()
        # the same kernel on the same operands: identical bits
        assert np.array_equal(new, ref), f"{mode} {M}x{N}x{K}: differs from gemm_f32_tc"
        gu.assert_close(new, _oracle(A, B), _s(A, B), gu.TOL[mode], f"{mode} {M}x{N}x{K}")
    gu.check_watchdog()


def test_only_b_misaligned_and_aligned_operands():
    """Only B re-pitched (A aligned), then no re-pitch at all."""
    M, N, K = 256, 301, 128
    A, B = inputs.make_random(M, N, K, seed=8)
    Ad = A.cuda()
    Bd = gu.device_view(*inputs.embed(B, N, offset=1))
    assert Bd.data_ptr() % 16 != 0
    ref, new = _pair("tf32", Ad, Bd)
    assert np.array_equal(new, ref)
    gu.assert_close(new, _oracle(A, B), _s(A, B), gu.TOL["tf32"], "only B re-pitched")
    A2, B2 = inputs.make_random(512, 512, 512, seed=9)
    ref, new = _pair("tf32", A2.cuda(), B2.cuda())
    assert np.array_equal(new, ref)
    gu.assert_close(new, _oracle(A2, B2), _s(A2, B2), gu.TOL["tf32"], "aligned")


def test_rejects_operands_beyond_the_scratch():
    """Misaligned operands whose re-pitched copies exceed 16 MiB: a clear
    status code, and nothing launched."""
    M, N, K = 2049, 2049, 2049          # 2049 x 2052 fp32 ~ 16.8 MB per copy
    A = torch.zeros((M, K), device="cuda")
    B = torch.zeros((K, N), device="cuda")
    C = torch.zeros((M, N), device="cuda")
    n0 = dg.dgemm_kernel_launches()
    st = _call(dg.gemm_f32_tc_noalloc, "tf32", A, B, C, torch.cuda.current_stream().cuda_stream)
    assert st == dg.ERR_SCRATCH_LIMIT
    assert "16 MiB" in dg.dgemm_status_string(st)
    assert dg.dgemm_kernel_launches() == n0


@pytest.mark.parametrize("K, launches", [(512, 2), (2048, 1)])
def test_3xtf32_lo_parts_in_the_fixed_scratch(K, launches):
    """3xTF32 on a problem the CTA-pair kernel takes (2048 x 2048): with
    K = 512 the lo parts of A and B (8 MiB) fit in the fixed scratch, so the
    split pre-pass writes them there and the pair kernel loads them (two
    launches); with K = 2048 (32 MiB) they do not, and the single-CTA kernel
    splits in shared memory (one launch).  With K = 512 both entry points run
    the same kernel on the same operands and agree bit for bit; with K = 2048
    gemm_f32_tc runs the pair kernel, which sums in another order, so the two
    agree within the 3xTF32 tolerance.  Both match the oracle."""
    M = N = 2048
    A, B = inputs.make_random(M, N, K, seed=K, dist="normal")
    Ad, Bd = A.cuda(), B.cuda()
    stream = torch.cuda.current_stream().cuda_stream
    C = torch.full((M, N), float("nan"), device="cuda")
    torch.cuda.synchronize()
    n0 = dg.dgemm_kernel_launches()
    assert _call(dg.gemm_f32_tc_noalloc, "3xtf32", Ad, Bd, C, stream) == dg.OK
    assert dg.dgemm_kernel_launches() - n0 == launches
    ref, new = _pair("3xtf32", Ad, Bd)
    S = _s(A, B)
    if launches == 2:
        assert np.array_equal(new, ref)
    err = np.abs(new.astype(np.float64) - ref.astype(np.float64))
    assert np.all(err <= gu.TOL["3xtf32"] * S)
    assert np.array_equal(C.cpu().numpy(), new)
    gu.assert_close(new, _oracle(A, B), S, gu.TOL["3xtf32"], f"3xtf32 K={K}")
    gu.check_watchdog()
