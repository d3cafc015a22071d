"""Tile widths of the single-CTA tensor-core kernel.

Below the CTA-pair threshold the library picks a 128 x BN tile (BN = 64, 128
or 256 with one CTA per SM, or the 128 x 128 two-CTAs-per-SM configuration),
and for 128 x 64 / 128 x 128 tiles stages one or two swizzle rows of K deep,
by problem shape; DGEMM_TC_BN=64 / 128 / 256 forces a width and
DGEMM_TC_KD=1 / 2 the depth.  Every width in
every tensor-core mode (8-bit operands read K-major, B transposed first)
against the CPU oracle, through ragged and unaligned operands,
the K-split and guarded C; without the K-split all widths give the same bits
(each output element sees the same multiply-adds in the same order); and the
default choice on a few shapes whose best width is known.
"""
import numpy as np
import pytest
import torch

import gpu_util as gu
from dense_gemm_f32_gb300 import inputs
import dense_gemm_f32_gb300 as dg

pytestmark = pytest.mark.gpu

WIDTHS = ("64", "128", "256")
MODES = ("tf32", "3xtf32", "bf16", "fp16", "e4m3", "e5m2")
SHAPES = [(1, 1, 1), (64, 64, 64), (130, 200, 70), (1000, 1013, 997), (512, 384, 4096),
          (1024, 1024, 256)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    gu.check_watchdog()


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("kd", ["1", "2"])
@pytest.mark.parametrize("bn", WIDTHS)
@pytest.mark.parametrize("M, N, K", SHAPES)
def test_every_width_matches_the_oracle(M, N, K, bn, kd, mode, monkeypatch):
    monkeypatch.setenv("DGEMM_TC_PAIR", "0")
    monkeypatch.setenv("DGEMM_TC_BN", bn)
    monkeypatch.setenv("DGEMM_TC_KD", kd)
    A, B = inputs.make_random(M, N, K, seed=M + 3 * N + K, dist="normal", dtype=gu.in_dtype(mode))
    Ad, Bd = A.cuda(), B.cuda()
    C1 = gu.run(mode, Ad, Bd).cpu()
    C2 = gu.run(mode, Ad, Bd).cpu()
    assert torch.equal(C1, C2), "two calls differ"
    ref, S = gu.oracle_full(A, B)
    gu.assert_close(C1.numpy(), ref, S, gu.TOL[mode], f"{mode} BN={bn} KD={kd} {M}x{N}x{K}")


@pytest.mark.parametrize("mode", MODES)
def test_widths_agree_bit_for_bit_without_split(mode, monkeypatch):
    monkeypatch.setenv("DGEMM_TC_PAIR", "0")
    monkeypatch.setenv("DGEMM_TC_SPLITK", "0")
    for (M, N, K) in [(300, 520, 256), (1000, 1013, 997)]:
        A, B = inputs.make_random(M, N, K, seed=7, dist="normal", dtype=gu.in_dtype(mode))
        Ad, Bd = A.cuda(), B.cuda()
        out = {}
        for bn in WIDTHS:
            for kd in ("1", "2"):
                monkeypatch.setenv("DGEMM_TC_BN", bn)
                monkeypatch.setenv("DGEMM_TC_KD", kd)
                out[bn + "/" + kd] = gu.run(mode, Ad, Bd).cpu()
        first = out["64/1"]
        for key, c in out.items():
            assert torch.equal(first, c), f"{mode} {M}x{N}x{K} {key}"


@pytest.mark.parametrize("mode", ("tf32", "bf16", "e4m3"))
@pytest.mark.parametrize("kd", ["1", "2"])
@pytest.mark.parametrize("bn", WIDTHS)
@pytest.mark.parametrize("split", ["0", "4"])
def test_widths_guard_bands_unaligned_operands_and_ldc(mode, bn, kd, split, monkeypatch):
    """A and B with rows off 16-byte boundaries (re-pitched), C through an
    ldc that breaks 16-byte rows with sentinels around and between its rows:
    nothing outside the M x N window is written."""
    monkeypatch.setenv("DGEMM_TC_PAIR", "0")
    monkeypatch.setenv("DGEMM_TC_BN", bn)
    monkeypatch.setenv("DGEMM_TC_KD", kd)
    monkeypatch.setenv("DGEMM_TC_SPLITK", split)
    M, N, K, ldc = 301, 517, 700, 523
    A, B = inputs.make_random(M, N, K, seed=23, dist="normal", dtype=gu.in_dtype(mode))
    ref, S = gu.oracle_full(A, B)
    Ad = gu.device_view(*inputs.embed(A, K + 1, offset=1))
    Bd = gu.device_view(*inputs.embed(B, N + 1, offset=1))
    buf, view = gu.guarded_output(M, N, ldc)
    gu.run(mode, Ad, Bd, out=view)
    gu.assert_guards_intact(buf, M, N, ldc)
    gu.assert_close(view.cpu().numpy(), ref, S, gu.TOL[mode], f"{mode} BN={bn} split={split}")


@pytest.mark.parametrize("bn", WIDTHS)
def test_integer_inputs_exact_every_width(bn, monkeypatch):
    monkeypatch.setenv("DGEMM_TC_PAIR", "0")
    monkeypatch.setenv("DGEMM_TC_BN", bn)
    A, B = inputs.make_integer(333, 444, 1000, seed=5)
    exact = A.numpy().astype(np.int64) @ B.numpy().astype(np.int64)
    for kd in ("1", "2"):
        monkeypatch.setenv("DGEMM_TC_KD", kd)
        for mode in ("tf32", "3xtf32"):
            C = gu.run(mode, A.cuda(), B.cuda()).cpu().numpy()
            assert np.array_equal(C.astype(np.int64), exact), (mode, bn, kd)


@pytest.mark.parametrize("mode", MODES)
def test_default_choice_matches_the_oracle(mode, monkeypatch):
    """The shapes of the measured sweep, through the library's own choice of
    kernel and width."""
    monkeypatch.delenv("DGEMM_TC_BN", raising=False)
    for (M, N, K) in [(256, 256, 256), (512, 512, 512), (1024, 1024, 64), (2048, 1024, 1024),
                      (1024, 2048, 512), (512, 512, 4096)]:
        A, B = inputs.make_random(M, N, K, seed=M ^ N ^ K, dist="normal", dtype=gu.in_dtype(mode))
        C = gu.run(mode, A.cuda(), B.cuda()).cpu().numpy()
        rows = np.arange(0, M, 37)
        ref, S = gu.oracle_rows(A, B, rows)
        gu.assert_close(C[rows], ref, S, gu.TOL[mode], f"{mode} default {M}x{N}x{K}")


@pytest.mark.parametrize("mode", ("tf32", "bf16", "e4m3"))
@pytest.mark.parametrize("kd", ["1", "2"])
@pytest.mark.parametrize("bn", WIDTHS)
def test_persistent_ctas_guard_bands_and_unaligned_ldc(mode, bn, kd, monkeypatch):
    """More tiles than CTA slots: persistent CTAs, whose epilogue stages C
    through a small per-warp buffer while the next tile's operands arrive;
    with an ldc that breaks 16-byte rows, sentinels around and between the
    rows of C, and a ragged last tile row and column."""
    monkeypatch.setenv("DGEMM_TC_PAIR", "0")
    monkeypatch.setenv("DGEMM_TC_BN", bn)
    monkeypatch.setenv("DGEMM_TC_KD", kd)
    monkeypatch.setenv("DGEMM_TC_SPLITK", "0")
    M, N, K, ldc = 4001, 1030, 200, 1033
    A, B = inputs.make_random(M, N, K, seed=29, dist="normal", dtype=gu.in_dtype(mode))
    buf, view = gu.guarded_output(M, N, ldc)
    gu.run(mode, A.cuda(), B.cuda(), out=view)
    gu.assert_guards_intact(buf, M, N, ldc)
    rows = np.concatenate([np.arange(0, M, 61), [M - 1]])
    ref, S = gu.oracle_rows(A, B, rows)
    gu.assert_close(view.cpu().numpy()[rows], ref, S, gu.TOL[mode], f"{mode} BN={bn} persistent")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("kd", ["1", "2"])
@pytest.mark.parametrize("bn", WIDTHS)
@pytest.mark.parametrize("ta, tb", [(False, True), (True, False), (True, True)])
def test_every_width_transposed_operands(ta, tb, bn, kd, mode, monkeypatch):
    """op(A) = A^T and / or op(B) = B^T (the MMA reads such operands MN- or
    K-major as stored; 8-bit ones are transposed into K-major form first) at
    every width, ragged sizes, with and without the K-split."""
    monkeypatch.setenv("DGEMM_TC_PAIR", "0")
    monkeypatch.setenv("DGEMM_TC_BN", bn)
    monkeypatch.setenv("DGEMM_TC_KD", kd)
    for (M, N, K, split) in [(300, 259, 301, "0"), (257, 385, 1030, "4")]:
        monkeypatch.setenv("DGEMM_TC_SPLITK", split)
        A, B = inputs.make_random(M, N, K, seed=M + N + K + ta + 2 * tb, dist="normal",
                                  dtype=gu.in_dtype(mode))
        Ad = (A.t().contiguous() if ta else A).cuda()
        Bd = (B.t().contiguous() if tb else B).cuda()
        C = dg.matmul(Ad, Bd, mode=mode, trans_a=ta, trans_b=tb)
        torch.cuda.synchronize()
        ref, S = gu.oracle_full(A, B)
        gu.assert_close(C.cpu().numpy(), ref, S, gu.TOL[mode],
                        f"{mode} BN={bn} KD={kd} ta={ta} tb={tb} {M}x{N}x{K} split={split}")
