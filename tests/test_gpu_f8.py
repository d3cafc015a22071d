"""FP8 operands (E4M3, E5M2) on the tcgen05 kernels, against the CPU oracle.

The 8-bit values are the operands as given (no scaling); the oracle widens
them exactly.  The tensor cores read 8-bit operands K-major only: A as M x K
and B as N x K (dgemm_gemm_ex with op_b = T) go straight to the GEMM kernel,
any other layout is transposed into scratch first by a byte-transpose kernel
(32-bit words and in-register byte permutes for aligned 64 x 64 tiles, bytes
at the edges and for unaligned operands).  Tolerance 2e-4 * S: the inputs and
their products are exact in fp32, only the accumulation rounds.
"""
import numpy as np
import pytest
import torch

import gpu_util as gu
from dense_gemm_f32_gb300 import inputs
import dense_gemm_f32_gb300 as dg

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    gu.check_watchdog()


def _check(mode, A, B, Ad, Bd, ta, tb, what):
    C = dg.matmul(Ad, Bd, mode=mode, trans_a=ta, trans_b=tb)
    torch.cuda.synchronize()
    ref, S = gu.oracle_full(A, B)
    gu.assert_close(C.cpu().numpy(), ref, S, gu.TOL[mode], what)
    return C


@pytest.mark.parametrize("mode", gu.F8_MODES)
def test_native_layout_needs_no_transpose(mode):
    """A as M x K and B as N x K: one launch, the GEMM kernel alone."""
    M, N, K = 640, 768, 512
    A, B = inputs.make_random(M, N, K, seed=3, dist="normal", dtype=gu.in_dtype(mode))
    Ad, Bt = A.cuda(), B.t().contiguous().cuda()
    n0 = dg.dgemm_kernel_launches()
    _check(mode, A, B, Ad, Bt, False, True, f"{mode} NT")
    assert dg.dgemm_kernel_launches() - n0 == 1


@pytest.mark.parametrize("mode", gu.F8_MODES)
def test_transpose_tiles_edges_and_alignment(mode):
    """B (K x N) transposed by the byte-transpose kernel: whole 64 x 64 tiles
    only, edge tiles, and unaligned rows (byte path); A stored K x M likewise."""
    for (M, N, K, pad) in [(256, 192, 128, 0), (200, 136, 72, 0), (65, 130, 193, 1),
                           (300, 517, 640, 3), (128, 64, 64, 0)]:
        A, B = inputs.make_random(M, N, K, seed=M + N + K, dist="normal", dtype=gu.in_dtype(mode))
        Bd = gu.device_view(*inputs.embed(B, N + pad))
        _check(mode, A, B, A.cuda(), Bd, False, False, f"{mode} NN {M}x{N}x{K} pad {pad}")
        At = A.t().contiguous()
        Ad = gu.device_view(*inputs.embed(At, M + pad, offset=pad))
        _check(mode, A, B, Ad, B.t().contiguous().cuda(), True, True,
               f"{mode} TT {M}x{N}x{K} pad {pad}")


@pytest.mark.parametrize("mode", gu.F8_MODES)
def test_long_k_error_bound(mode):
    """K = 16384, the longest K the tolerance is stated for, on both kernels."""
    A, B = inputs.make_random(256, 384, 16384, seed=19, dist="normal", dtype=gu.in_dtype(mode))
    for pair in ("0", "1"):
        import os

        os.environ["DGEMM_TC_PAIR"] = pair
        try:
            _check(mode, A, B, A.cuda(), B.cuda(), False, False, f"{mode} K=16384 pair={pair}")
        finally:
            del os.environ["DGEMM_TC_PAIR"]


def test_e5m2_wide_range():
    """E5M2 covers 2^-16 .. 57344: operands spanning that range, products
    far apart in magnitude (exact in fp32), against the oracle."""
    g = torch.Generator().manual_seed(5)
    M, N, K = 192, 160, 256
    ea = torch.randint(-14, 12, (M, K), generator=g).float()
    eb = torch.randint(-14, 4, (K, N), generator=g).float()
    sa = torch.where(torch.rand(M, K, generator=g) < 0.5, -1.0, 1.0)
    A = (sa * torch.exp2(ea) * (1 + torch.randint(0, 4, (M, K), generator=g) / 4)).to(
        torch.float8_e5m2)
    B = (torch.exp2(eb) * (1 + torch.randint(0, 4, (K, N), generator=g) / 4)).to(torch.float8_e5m2)
    assert torch.isfinite(A.float()).all() and torch.isfinite(B.float()).all()
    _check("e5m2", A, B, A.cuda(), B.cuda(), False, False, "e5m2 wide range")


@pytest.mark.parametrize("mode", gu.F8_MODES)
def test_integer_inputs_exact_every_layout(mode):
    A, B = inputs.make_integer(520, 1030, 1024, seed=21)
    A, B = A.to(gu.in_dtype(mode)), B.to(gu.in_dtype(mode))
    exact = A.float().numpy().astype(np.int64) @ B.float().numpy().astype(np.int64)
    for ta, tb in [(False, False), (False, True), (True, False), (True, True)]:
        Ad = (A.t().contiguous() if ta else A).cuda()
        Bd = (B.t().contiguous() if tb else B).cuda()
        C = dg.matmul(Ad, Bd, mode=mode, trans_a=ta, trans_b=tb).cpu().numpy()
        assert np.array_equal(C.astype(np.float64), exact.astype(np.float64)), (ta, tb)
