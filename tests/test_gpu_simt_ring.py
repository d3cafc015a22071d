"""The FP32 SIMT path's TMA ring kernel (sgemm_ring_kernel) against the CPU
oracle, in both of its configurations, and against the register-staged
kernel it replaced for TMA-readable operands.

The ring kernel runs when A's and B's rows start on 16-byte boundaries and
B is stored K x N (A either way).  DGEMM_SIMT_RING=1 forces the 128 x 256
configuration (one CTA per SM), =2 the 128 x 128 one (two CTAs per SM), =0
the register-staged kernel; DGEMM_SIMT_SMALL=0 keeps small problems on the
large tiles, so that the K-split paths (partials through scratch for a
partial last wave, through distributed shared memory when every tile is
split) run too.
"""
import numpy as np
import pytest
import torch

import gpu_util as gu
from dense_gemm_f32_gb300 import inputs
import dense_gemm_f32_gb300 as dg

pytestmark = pytest.mark.gpu

RINGS = ["1", "2"]

# Several tiles with ragged edges in M, N and K (K % 32 != 0 but lda % 4 == 0,
# so TMA can still read the rows), a single partial tile, long K.
SHAPES = [(1, 4, 4), (64, 64, 64), (129, 260, 36), (300, 516, 1000), (1000, 1012, 1000),
          (257, 516, 4096)]
# The tail split: 200 tiles of 128 x 256 on 152 SMs (48 in the last wave),
# 320 tiles of 128 x 128 on 304 slots (16 in the last wave).
TAIL_SHAPES = [(1024, 6400, 1024), (1024, 5120, 1024)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    gu.check_watchdog()


@pytest.mark.parametrize("ring", RINGS)
@pytest.mark.parametrize("M, N, K", SHAPES)
def test_ring_matches_the_oracle(M, N, K, ring, monkeypatch):
    monkeypatch.setenv("DGEMM_SIMT_RING", ring)
    monkeypatch.setenv("DGEMM_SIMT_SMALL", "0")
    A, B = inputs.make_random(M, N, K, seed=M * 3 + N + K, dist="normal")
    C = gu.run("simt", A.cuda(), B.cuda())
    ref, S = gu.oracle_full(A, B)
    gu.assert_close(C.cpu().numpy(), ref, S, gu.TOL["simt"], f"ring={ring} {M}x{N}x{K}")
    gu.check_watchdog()


@pytest.mark.parametrize("ring", RINGS)
@pytest.mark.parametrize("M, N, K", TAIL_SHAPES)
def test_ring_tail_split_matches_the_oracle(M, N, K, ring, monkeypatch):
    monkeypatch.setenv("DGEMM_SIMT_RING", ring)
    A, B = inputs.make_random(M, N, K, seed=11, dist="uniform")
    Ad, Bd = A.cuda(), B.cuda()
    C1 = gu.run("simt", Ad, Bd).cpu()
    C2 = gu.run("simt", Ad, Bd).cpu()
    assert torch.equal(C1, C2), "two calls differ"
    rows = np.unique(np.concatenate([np.arange(0, 8), np.arange(M - 8, M),
                                     np.random.default_rng(3).integers(0, M, 48)]))
    ref, S = gu.oracle_rows(A, B, rows)
    gu.assert_close(C1.numpy()[rows], ref, S, gu.TOL["simt"], f"ring={ring} tail {M}x{N}x{K}")


@pytest.mark.parametrize("ring", RINGS)
@pytest.mark.parametrize("M, N, K", [(128, 256, 4096), (256, 256, 2048), (300, 520, 1024)])
def test_ring_cluster_split_matches_the_oracle(M, N, K, ring, monkeypatch):
    """Few tiles: every tile split along K over a thread-block cluster."""
    monkeypatch.setenv("DGEMM_SIMT_RING", ring)
    monkeypatch.setenv("DGEMM_SIMT_SMALL", "0")
    A, B = inputs.make_random(M, N, K, seed=5, dist="normal")
    Ad, Bd = A.cuda(), B.cuda()
    C1 = gu.run("simt", Ad, Bd).cpu()
    C2 = gu.run("simt", Ad, Bd).cpu()
    assert torch.equal(C1, C2), "two calls differ"
    ref, S = gu.oracle_full(A, B)
    gu.assert_close(C1.numpy(), ref, S, gu.TOL["simt"], f"ring={ring} cluster {M}x{N}x{K}")


@pytest.mark.parametrize("ring", RINGS)
def test_ring_integer_inputs_exact(ring, monkeypatch):
    """Integers in [-4, 4] with K <= 1024: every partial sum is exact in
    fp32, so C equals the oracle bit for bit (also through the K-split)."""
    monkeypatch.setenv("DGEMM_SIMT_RING", ring)
    monkeypatch.setenv("DGEMM_SIMT_SMALL", "0")
    for (M, N, K) in [(300, 516, 1024), (128, 256, 1024), (1024, 5120, 1024)]:
        g = torch.Generator().manual_seed(M + N)
        A = torch.randint(-4, 5, (M, K), generator=g).float()
        B = torch.randint(-4, 5, (K, N), generator=g).float()
        C = gu.run("simt", A.cuda(), B.cuda()).cpu().numpy().astype(np.float64)
        ref = A.double().numpy() @ B.double().numpy()
        assert np.array_equal(C, ref), f"ring={ring} {M}x{N}x{K}: not exact"


@pytest.mark.parametrize("ring", RINGS)
def test_ring_transposed_a_matches_the_oracle(ring, monkeypatch):
    """op(A) = A^T (A stored K x M): A's boxes land k-major."""
    monkeypatch.setenv("DGEMM_SIMT_RING", ring)
    monkeypatch.setenv("DGEMM_SIMT_SMALL", "0")
    for (M, N, K) in [(260, 516, 1000), (128, 256, 2048)]:
        A, B = inputs.make_random(M, N, K, seed=9, dist="normal")
        At = A.t().contiguous().cuda()
        C = dg.matmul(At, B.cuda(), mode="simt", trans_a=True)
        torch.cuda.synchronize()
        ref, S = gu.oracle_full(A, B)
        gu.assert_close(C.cpu().numpy(), ref, S, gu.TOL["simt"], f"ring={ring} A^T {M}x{N}x{K}")


def test_ring_and_register_staged_kernels_agree_bitwise(monkeypatch):
    """Unsplit (K = 64: too few k-blocks to split), every kernel gives each
    output element the same multiply-adds in K order: identical bits."""
    M, N, K = 333, 520, 64
    A, B = inputs.make_random(M, N, K, seed=21, dist="normal")
    Ad, Bd = A.cuda(), B.cuda()
    monkeypatch.setenv("DGEMM_SIMT_SMALL", "0")
    out = {}
    for ring in ("0", "1", "2"):
        monkeypatch.setenv("DGEMM_SIMT_RING", ring)
        out[ring] = gu.run("simt", Ad, Bd).cpu()
    assert torch.equal(out["0"], out["1"]) and torch.equal(out["0"], out["2"])


def test_ring_leaves_the_ldc_gap_and_guard_bands_untouched(monkeypatch):
    """C written through a strided view: the columns between N and ldc and the
    rows around C keep their sentinel."""
    monkeypatch.setenv("DGEMM_SIMT_SMALL", "0")
    M, N, K, ldc = 300, 516, 1000, 532
    A, B = inputs.make_random(M, N, K, seed=4, dist="normal")
    ref, S = gu.oracle_full(A, B)
    for ring in RINGS:
        monkeypatch.setenv("DGEMM_SIMT_RING", ring)
        buf = torch.full(((M + 2) * ldc,), 7.0, device="cuda")
        C = buf[ldc:ldc + M * ldc].view(M, ldc)[:, :N]
        dg.matmul(A.cuda(), B.cuda(), mode="simt", out=C)
        torch.cuda.synchronize()
        gu.assert_close(C.cpu().numpy(), ref, S, gu.TOL["simt"], f"ring={ring} strided C")
        host = buf.cpu().view(M + 2, ldc)
        assert torch.all(host[0] == 7.0) and torch.all(host[M + 1] == 7.0), "guard rows written"
        assert torch.all(host[1:M + 1, N:] == 7.0), "ldc gap written"
