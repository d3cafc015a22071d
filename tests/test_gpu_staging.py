"""Staging of operands TMA cannot read as stored: re-pitch and byte transpose.

A re-pitched row is assembled from the aligned 16-byte blocks it straddles
(blocks wholly inside the row by vector loads, the partial blocks at its two
ends byte by byte, nothing outside the row read).  Rows of every length
against the 16-byte chunk (shorter than one chunk, exactly one, many, more
chunks than a block's 256 threads) at several offsets from the 16-byte
boundary, in every element size, go through the GEMM and are compared with
the CPU oracle.  For 8-bit operands a transpose and a re-pitch (or two of
either) go out in one staging launch before the GEMM.
"""
import pytest
import torch

import gpu_util as gu
import dense_gemm_f32_gb300 as dg
from dense_gemm_f32_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    gu.check_watchdog()


@pytest.mark.parametrize("mode", ("tf32", "bf16", "e4m3"))
@pytest.mark.parametrize("K", [1, 3, 4, 5, 8, 15, 16, 17, 33, 100, 1000, 4100])
def test_repitch_row_lengths_and_offsets(mode, K):
    """A (M x K) with its rows off 16-byte boundaries by 1 .. 3 elements plus
    a pitch that moves every row's offset; B re-pitched too in one case.  The
    8-bit case reads B stored N x K (re-pitch only)."""
    M, N = 70, 24
    f8 = mode in gu.F8_MODES
    A, B = inputs.make_random(M, N, K, seed=K, dist="normal", dtype=gu.in_dtype(mode))
    ref, S = gu.oracle_full(A, B)
    Bs = B.t().contiguous() if f8 else B
    for off, extra, b_mis in [(1, 1, False), (2, 3, True), (3, 0, False)]:
        Ad = gu.device_view(*inputs.embed(A, K + extra, offset=off))
        if b_mis:
            Bd = gu.device_view(*inputs.embed(Bs, Bs.shape[1] + 1, offset=1))
        else:
            Bd = Bs.cuda()
        C = dg.matmul(Ad, Bd, mode=mode, trans_b=f8)
        torch.cuda.synchronize()
        gu.assert_close(C.cpu().numpy(), ref, S, gu.TOL[mode],
                        f"{mode} K={K} offset={off} lda=K+{extra} B misaligned={b_mis}")


@pytest.mark.parametrize("mode", gu.F8_MODES)
@pytest.mark.parametrize("ta, tb, a_mis, b_mis", [
    (False, False, True, False),  # B transposed, A re-pitched
    (False, False, False, False),  # B transposed alone
    (True, True, False, True),  # A transposed, B re-pitched
    (True, False, False, False),  # both transposed
    (False, True, True, True),  # both re-pitched
])
def test_f8_staging_in_one_launch(mode, ta, tb, a_mis, b_mis):
    """Every 8-bit layout that needs staging: one staging launch for both
    operands, then the GEMM."""
    M, N, K = 300, 259, 301
    A, B = inputs.make_random(M, N, K, seed=7 + ta + 2 * tb, dist="normal", dtype=gu.in_dtype(mode))
    ref, S = gu.oracle_full(A, B)
    As = A.t().contiguous() if ta else A
    Bs = B.t().contiguous() if tb else B
    Ad = gu.device_view(*inputs.embed(As, As.shape[1] + 3, offset=5)) if a_mis else As.cuda()
    Bd = gu.device_view(*inputs.embed(Bs, Bs.shape[1] + 1, offset=2)) if b_mis else Bs.cuda()
    torch.cuda.synchronize()
    n0 = dg.dgemm_kernel_launches()
    C = dg.matmul(Ad, Bd, mode=mode, trans_a=ta, trans_b=tb)
    torch.cuda.synchronize()
    assert dg.dgemm_kernel_launches() - n0 == 2, (ta, tb, a_mis, b_mis)
    gu.assert_close(C.cpu().numpy(), ref, S, gu.TOL[mode], f"{mode} ta={ta} tb={tb}")
