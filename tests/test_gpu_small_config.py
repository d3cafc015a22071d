"""The single-CTA tensor-core kernel's small-problem configuration.

Problems below the CTA-pair kernel's threshold run on the single-CTA kernel
with 128 x 128 tiles and 3 stages, two CTAs per SM, for 8-bit operands and
when K is short (DGEMM_TC_SMALL=1 / =0 forces it on / off).  Against the CPU oracle in every mode,
including the cluster K-split, ragged and unaligned operands (re-pitched, both
operands in one launch); and, with the K-split off, bit for bit equal to the
large configuration (every output element sees the same multiply-adds in the
same order).
"""
import pytest
import torch

import gpu_util as gu
from dense_gemm_f32_gb300 import inputs
import dense_gemm_f32_gb300 as dg

pytestmark = pytest.mark.gpu

MODES = ("tf32", "bf16", "fp16", "e4m3", "e5m2")
SHAPES = [(1, 1, 1), (64, 64, 64), (130, 200, 70), (1000, 1013, 997), (1024, 1024, 1024),
          (512, 384, 4096)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    gu.check_watchdog()


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("M, N, K", SHAPES)
def test_small_configuration_matches_the_oracle(M, N, K, mode, monkeypatch):
    monkeypatch.setenv("DGEMM_TC_PAIR", "0")
    monkeypatch.setenv("DGEMM_TC_SMALL", "1")
    A, B = inputs.make_random(M, N, K, seed=M + 2 * N + K, dist="normal", dtype=gu.in_dtype(mode))
    Ad, Bd = A.cuda(), B.cuda()
    C1 = gu.run(mode, Ad, Bd).cpu()
    C2 = gu.run(mode, Ad, Bd).cpu()
    assert torch.equal(C1, C2), "two calls differ"
    ref, S = gu.oracle_full(A, B)
    gu.assert_close(C1.numpy(), ref, S, gu.TOL[mode], f"{mode} small config {M}x{N}x{K}")


@pytest.mark.parametrize("mode", MODES)
def test_small_and_large_configurations_agree_without_split(mode, monkeypatch):
    monkeypatch.setenv("DGEMM_TC_PAIR", "0")
    monkeypatch.setenv("DGEMM_TC_SPLITK", "0")
    for (M, N, K) in [(300, 520, 256), (1000, 1013, 997)]:
        A, B = inputs.make_random(M, N, K, seed=9, dist="normal", dtype=gu.in_dtype(mode))
        Ad, Bd = A.cuda(), B.cuda()
        out = {}
        for small in ("1", "0"):
            monkeypatch.setenv("DGEMM_TC_SMALL", small)
            out[small] = gu.run(mode, Ad, Bd).cpu()
        assert torch.equal(out["1"], out["0"]), f"{mode} {M}x{N}x{K}"


@pytest.mark.parametrize("mode", ("tf32", "bf16"))
def test_one_re_pitch_launch_for_both_operands(mode):
    """A and B with rows off 16-byte boundaries: one re-pitch launch for both,
    then the GEMM; only one of them misaligned: still one re-pitch launch."""
    M, N, K = 300, 259, 301
    A, B = inputs.make_random(M, N, K, seed=4, dist="normal", dtype=gu.in_dtype(mode))
    ref, S = gu.oracle_full(A, B)
    up8 = lambda x: (x + 7) // 8 * 8  # noqa: E731  (16-byte rows for fp32 and bf16)
    # (lda, A offset, ldb, B offset): both misaligned, only A, only B
    cases = [(K + 1, 1, N + 1, 1), (K + 1, 1, up8(N), 0), (up8(K), 0, N + 1, 1)]
    for lda, oa, ldb, ob in cases:
        Ad = gu.device_view(*inputs.embed(A, lda, offset=oa))
        Bd = gu.device_view(*inputs.embed(B, ldb, offset=ob))
        torch.cuda.synchronize()
        n0 = dg.dgemm_kernel_launches()
        C = gu.run(mode, Ad, Bd)
        assert dg.dgemm_kernel_launches() - n0 == 2, f"lda={lda} ldb={ldb}"
        gu.assert_close(C.cpu().numpy(), ref, S, gu.TOL[mode], f"{mode} lda={lda} ldb={ldb}")
