"""K-split of the single-CTA tensor-core kernel.

When a problem has too few 128 x 256 output tiles to fill half the GPU, the
single-CTA kernel divides each tile's K range into parts (at most 8, each at
least 4 k-blocks), writes one fp32 partial tile per part to scratch, and a
second kernel adds the parts in a fixed order into C.  DGEMM_TC_SPLITK=0
turns the split off.  These tests run shapes that split evenly, unevenly and
not at all, with and without the split, against the CPU oracle, and check that
the split result does not depend on the order the parts finish in.
"""
import pytest
import torch

import gpu_util as gu
from dense_gemm_f32_gb300 import inputs
import dense_gemm_f32_gb300 as dg

pytestmark = pytest.mark.gpu

TC_MODES = ["tf32", "3xtf32", "bf16", "fp16"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    gu.check_watchdog()


@pytest.fixture(autouse=True)
def _single_cta(monkeypatch):
    monkeypatch.setenv("DGEMM_TC_PAIR", "0")


# (M, N, K): one tile with 8 parts; 34 k-blocks of fp32 (7 uneven parts);
# 32 tiles (4 parts); too short a K to split; a ragged tile grid.
SHAPES = [(128, 256, 1000), (100, 200, 1061), (1024, 1024, 1024), (300, 500, 96),
          (333, 777, 2345)]


@pytest.mark.parametrize("mode", TC_MODES)
def test_split_and_unsplit_match_oracle(mode, monkeypatch):
    for (M, N, K) in SHAPES:
        A, B = inputs.make_random(M, N, K, seed=M + N + K, dist="normal",
                                  dtype=gu.in_dtype(mode))
        Ad, Bd = A.cuda(), B.cuda()
        ref, S = gu.oracle_full(A, B)
        monkeypatch.delenv("DGEMM_TC_SPLITK", raising=False)
        C1 = gu.run(mode, Ad, Bd).clone()
        C2 = gu.run(mode, Ad, Bd)
        assert torch.equal(C1, C2), f"{mode} {M}x{N}x{K}: split sums must be deterministic"
        gu.assert_close(C1.cpu().numpy(), ref, S, gu.TOL[mode], f"{mode} split {M}x{N}x{K}")
        monkeypatch.setenv("DGEMM_TC_SPLITK", "0")
        C0 = gu.run(mode, Ad, Bd)
        gu.assert_close(C0.cpu().numpy(), ref, S, gu.TOL[mode], f"{mode} unsplit {M}x{N}x{K}")


@pytest.mark.parametrize("mode", TC_MODES)
def test_split_adds_one_reduce_launch(mode, monkeypatch):
    """A split call launches the GEMM kernel and the reduce kernel; an unsplit
    call launches the GEMM kernel alone."""
    A, B = inputs.make_random(128, 256, 1000, seed=5, dtype=gu.in_dtype(mode))
    Ad, Bd = A.cuda(), B.cuda()
    n0 = dg.dgemm_kernel_launches()
    gu.run(mode, Ad, Bd)
    assert dg.dgemm_kernel_launches() - n0 == 2
    monkeypatch.setenv("DGEMM_TC_SPLITK", "0")
    n0 = dg.dgemm_kernel_launches()
    gu.run(mode, Ad, Bd)
    assert dg.dgemm_kernel_launches() - n0 == 1


@pytest.mark.parametrize("mode", TC_MODES)
def test_split_guard_bands_and_unaligned_ldc(mode):
    """The reduce kernel writes C through an ldc that breaks 16-byte row
    alignment (scalar stores) and leaves the gap columns untouched."""
    M, N, K = 301, 517, 2000
    A, B = inputs.make_random(M, N, K, seed=33, dist="normal", dtype=gu.in_dtype(mode))
    for ldc in (N + 6, 520):  # 2092-byte rows (scalar stores), 2080-byte rows
        buf, C = gu.guarded_output(M, N, ldc)
        Cr = gu.run(mode, A.cuda(), B.cuda(), C)
        ref, S = gu.oracle_full(A, B)
        gu.assert_close(Cr.cpu().numpy(), ref, S, gu.TOL[mode], f"{mode} split ldc={ldc}")
        gu.assert_guards_intact(buf, M, N, ldc)


@pytest.mark.parametrize("mode", ["tf32", "bf16"])
def test_split_integer_bit_exact(mode):
    """Integer entries in {-4..4}: every partial sum is exact, so the split
    result equals the exact product bit for bit."""
    import numpy as np

    A, B = inputs.make_integer(200, 300, 1024, seed=12)
    A, B = A.to(gu.in_dtype(mode)), B.to(gu.in_dtype(mode))
    C = gu.run(mode, A.cuda(), B.cuda()).cpu().numpy()
    exact = A.float().numpy().astype(np.int64) @ B.float().numpy().astype(np.int64)
    assert np.array_equal(C.astype(np.float64), exact.astype(np.float64))
