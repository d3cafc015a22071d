"""K-split of the single-CTA tensor-core kernel.

When a problem has too few 128 x BN output tiles to fill half the GPU, the
single-CTA kernel divides each tile's K range into parts (2 to 8, each at
least 4 k-blocks) and runs the parts of one tile as one thread-block cluster.
Every CTA parks its partial tile in its own shared memory; after a cluster
barrier the CTAs add the partials in part order through distributed shared
memory, each writing a slice of the tile's rows to C.  DGEMM_TC_SPLITK=0
turns the split off and DGEMM_TC_SPLITK=n (2..8) forces n parts.  These tests
run every cluster size and the automatic choice against the CPU oracle, and
check that the split result does not depend on scheduling.
"""
import numpy as np
import pytest
import torch

import gpu_util as gu
from dense_gemm_f32_gb300 import inputs
import dense_gemm_f32_gb300 as dg

pytestmark = pytest.mark.gpu

TC_MODES = list(gu.TC_MODES)


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


# (M, N, K): one tile with 8 parts; 34 fp32 k-blocks (7 uneven parts);
# 32 tiles (4 parts); too short a K to split; a ragged tile grid.
SHAPES = [(128, 256, 1000), (100, 200, 1061), (1024, 1024, 1024), (300, 500, 96),
          (333, 777, 2345)]


@pytest.mark.parametrize("mode", TC_MODES)
def test_automatic_split_and_unsplit_match_oracle(mode, monkeypatch):
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
@pytest.mark.parametrize("parts", [2, 3, 4, 5, 6, 7, 8])
def test_every_cluster_size(mode, parts, monkeypatch):
    """Forced part counts, so every cluster size and every row slicing of
    the 128-row tile (128 / parts need not be whole) runs; ragged M, N, K;
    more clusters than fit at once for the larger sizes."""
    monkeypatch.setenv("DGEMM_TC_SPLITK", str(parts))
    for (M, N, K) in [(200, 300, 777), (1300, 700, 515)]:
        A, B = inputs.make_random(M, N, K, seed=parts * 1000 + M, dist="normal",
                                  dtype=gu.in_dtype(mode))
        Ad, Bd = A.cuda(), B.cuda()
        C1 = gu.run(mode, Ad, Bd).clone()
        C2 = gu.run(mode, Ad, Bd)
        assert torch.equal(C1, C2)
        ref, S = gu.oracle_full(A, B)
        gu.assert_close(C1.cpu().numpy(), ref, S, gu.TOL[mode], f"{mode} parts={parts} {M}x{N}x{K}")


@pytest.mark.parametrize("mode", TC_MODES)
def test_split_is_one_launch(mode, monkeypatch):
    """The split needs no second kernel and no scratch (the FP8 paths add one
    launch either way: the transpose of the row-major B into K-major form)."""
    A, B = inputs.make_random(128, 256, 1024, seed=5, dtype=gu.in_dtype(mode))
    Ad, Bd = A.cuda(), B.cuda()
    want = 2 if mode in gu.F8_MODES else 1
    for env in ("8", "0"):
        monkeypatch.setenv("DGEMM_TC_SPLITK", env)
        n0 = dg.dgemm_kernel_launches()
        gu.run(mode, Ad, Bd)
        assert dg.dgemm_kernel_launches() - n0 == want


@pytest.mark.parametrize("mode", TC_MODES)
def test_split_guard_bands_and_unaligned_ldc(mode):
    """The cluster reduction writes C through an ldc that breaks 16-byte row
    alignment (scalar stores) and leaves the gap columns untouched."""
    M, N, K = 301, 517, 2000
    A, B = inputs.make_random(M, N, K, seed=33, dist="normal", dtype=gu.in_dtype(mode))
    for ldc in (N + 6, 520):  # 2092-byte rows (scalar stores), 2080-byte rows
        buf, C = gu.guarded_output(M, N, ldc)
        Cr = gu.run(mode, A.cuda(), B.cuda(), C)
        ref, S = gu.oracle_full(A, B)
        gu.assert_close(Cr.cpu().numpy(), ref, S, gu.TOL[mode], f"{mode} split ldc={ldc}")
        gu.assert_guards_intact(buf, M, N, ldc)


@pytest.mark.parametrize("mode", TC_MODES)
def test_split_transposed_operands(mode, monkeypatch):
    """The split with A stored K x M and B stored N x K."""
    monkeypatch.setenv("DGEMM_TC_SPLITK", "4")
    M, N, K = 260, 390, 1100
    A, B = inputs.make_random(M, N, K, seed=77, dist="normal", dtype=gu.in_dtype(mode))
    At, Bt = A.t().contiguous().cuda(), B.t().contiguous().cuda()
    C = dg.matmul(At, Bt, mode=mode, trans_a=True, trans_b=True)
    torch.cuda.synchronize()
    ref, S = gu.oracle_full(A, B)
    gu.assert_close(C.cpu().numpy(), ref, S, gu.TOL[mode], f"{mode} split TT")


@pytest.mark.parametrize("mode", TC_MODES)
def test_split_integer_bit_exact(mode, monkeypatch):
    """Integer entries in {-4..4}: every partial sum is exact, so the split
    result equals the exact product bit for bit."""
    A, B = inputs.make_integer(200, 300, 1024, seed=12)
    A, B = A.to(gu.in_dtype(mode)), B.to(gu.in_dtype(mode))
    exact = A.float().numpy().astype(np.int64) @ B.float().numpy().astype(np.int64)
    for env in ("", "3", "8"):
        if env:
            monkeypatch.setenv("DGEMM_TC_SPLITK", env)
        C = gu.run(mode, A.cuda(), B.cuda()).cpu().numpy()
        assert np.array_equal(C.astype(np.float64), exact.astype(np.float64)), env
