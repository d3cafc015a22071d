"""The two tile configurations of the FP32 SIMT kernel, each forced on shapes
the other one would normally take, against the CPU oracle.

The library runs 128 x 256 x 16 block tiles, and 64 x 64 x 16 ones (4 x 8
outputs per thread, up to 4 CTAs per SM) when the large tiles would be fewer
than an eighth of the SMs or a third of their area padding.
DGEMM_SIMT_SMALL=0 / =1 forces one of them.  Both give every output element
the same sequence of multiply-adds in K order unless K is split, so with
K = 64 (4 k-blocks: never split) they must agree bit for bit.
"""
import numpy as np
import pytest
import torch

import gpu_util as gu
from dense_gemm_f32_gb300 import inputs
import dense_gemm_f32_gb300 as dg

pytestmark = pytest.mark.gpu

SHAPES = [(1, 1, 1), (64, 64, 64), (65, 130, 33), (300, 64, 1000), (64, 700, 512),
          (1000, 1013, 997), (257, 513, 4096)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    gu.check_watchdog()


@pytest.mark.parametrize("small", ["0", "1"])
@pytest.mark.parametrize("M, N, K", SHAPES)
def test_both_configurations_match_the_oracle(M, N, K, small, monkeypatch):
    monkeypatch.setenv("DGEMM_SIMT_SMALL", small)
    A, B = inputs.make_random(M, N, K, seed=M * 7 + N + K, dist="normal")
    C = gu.run("simt", A.cuda(), B.cuda())
    ref, S = gu.oracle_full(A, B)
    gu.assert_close(C.cpu().numpy(), ref, S, gu.TOL["simt"], f"simt small={small} {M}x{N}x{K}")


@pytest.mark.parametrize("small", ["0", "1"])
def test_transposed_and_unaligned_operands(small, monkeypatch):
    """op(A) = A^T, op(B) = B^T and rows that are not 16-byte aligned (scalar
    loads at the edges) on each configuration."""
    monkeypatch.setenv("DGEMM_SIMT_SMALL", small)
    M, N, K = 130, 75, 301
    A, B = inputs.make_random(M, N, K, seed=5, dist="normal")
    ref, S = gu.oracle_full(A, B)
    for ta, tb in [(False, False), (True, False), (False, True), (True, True)]:
        As = A.t().contiguous() if ta else A
        Bs = B.t().contiguous() if tb else B
        Ad = gu.device_view(*inputs.embed(As, As.shape[1] + 1, offset=1))
        Bd = gu.device_view(*inputs.embed(Bs, Bs.shape[1] + 3, offset=3))
        C = dg.matmul(Ad, Bd, mode="simt", trans_a=ta, trans_b=tb)
        torch.cuda.synchronize()
        gu.assert_close(C.cpu().numpy(), ref, S, gu.TOL["simt"],
                        f"simt small={small} ta={ta} tb={tb}")


def test_unsplit_results_identical_across_configurations(monkeypatch):
    M, N, K = 333, 517, 64
    A, B = inputs.make_random(M, N, K, seed=77, dist="normal")
    Ad, Bd = A.cuda(), B.cuda()
    out = {}
    for small in ("0", "1"):
        monkeypatch.setenv("DGEMM_SIMT_SMALL", small)
        out[small] = gu.run("simt", Ad, Bd).cpu()
    assert torch.equal(out["0"], out["1"])
