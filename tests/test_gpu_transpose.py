"""C = op(A) op(B) with transposed operands (dgemm_gemm_ex), every path.

A transposed A is stored K x M and a transposed B is stored N x K, both
row-major (Lesson 8 section 二十八: a column-major matrix is a row-major
transpose).  Every path (SIMT, TF32, 3xTF32, BF16, FP16, FP8) and, for the tensor
cores, both kernels (single CTA and CTA pair, forced with DGEMM_TC_PAIR) are
compared with the CPU oracle on op(A) and op(B), at the same tolerances as
the plain product, over ragged shapes, padded leading dimensions,
misaligned bases (re-pitched for TMA) and guard bands around C.
"""
import numpy as np
import pytest
import torch

import gpu_util as gu
from dense_gemm_f32_gb300 import inputs

pytestmark = pytest.mark.gpu

LAYOUTS = [(False, True), (True, False), (True, True), (False, False)]
LAYOUT_IDS = ["NT", "TN", "TT", "NN"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    gu.check_watchdog()


def _stored(X, trans):
    """The matrix as stored: X itself, or X^T laid out row-major."""
    return X.t().contiguous() if trans else X


def _run(mode, A, B, ta, tb, ld_pad=0, offset=0, out=None):
    As, Bs = _stored(A, ta), _stored(B, tb)
    Ad = gu.device_view(*inputs.embed(As, As.shape[1] + ld_pad, offset=offset))
    Bd = gu.device_view(*inputs.embed(Bs, Bs.shape[1] + ld_pad, offset=offset))
    import dense_gemm_f32_gb300 as dg

    C = dg.matmul(Ad, Bd, mode=mode, out=out, trans_a=ta, trans_b=tb)
    torch.cuda.synchronize()
    return C


def _modes_and_kernels():
    for mode in gu.ALL_MODES:
        for pair in (["0", "1"] if mode != "simt" else ["-"]):
            yield mode, pair


@pytest.mark.parametrize("layout", LAYOUTS, ids=LAYOUT_IDS)
@pytest.mark.parametrize("mode,pair", list(_modes_and_kernels()))
def test_transposed_operands(mode, pair, layout, monkeypatch):
    if pair != "-":
        monkeypatch.setenv("DGEMM_TC_PAIR", pair)
    ta, tb = layout
    for (M, N, K, pad, off) in [(300, 517, 173, 0, 0), (257, 129, 333, 8, 0), (130, 260, 97, 3, 1),
                               (1, 300, 65, 0, 0), (600, 2, 40, 4, 0)]:
        A, B = inputs.make_random(M, N, K, seed=M + N + K, dist="normal", dtype=gu.in_dtype(mode))
        buf, C = gu.guarded_output(M, N, N + 5)
        C = _run(mode, A, B, ta, tb, ld_pad=pad, offset=off, out=C)
        ref, S = gu.oracle_full(A, B)
        gu.assert_close(C.cpu().numpy(), ref, S, gu.TOL[mode],
                        f"{mode} pair={pair} {'T' if ta else 'N'}{'T' if tb else 'N'} {M}x{N}x{K}")
        gu.assert_guards_intact(buf, M, N, N + 5)


@pytest.mark.parametrize("layout", LAYOUTS, ids=LAYOUT_IDS)
@pytest.mark.parametrize("mode", gu.ALL_MODES)
def test_transposed_integer_bit_exact_large(mode, layout):
    """Integer inputs in {-4..4}, K = 1024, many tiles (the kernel picks its
    own path): exact in every layout."""
    ta, tb = layout
    A, B = inputs.make_integer(1030, 1100, 1024, seed=11)
    A, B = A.to(gu.in_dtype(mode)), B.to(gu.in_dtype(mode))
    C = _run(mode, A, B, ta, tb).cpu().numpy()
    exact = A.float().numpy().astype(np.int64) @ B.float().numpy().astype(np.int64)
    assert np.array_equal(C.astype(np.float64), exact.astype(np.float64))


@pytest.mark.parametrize("layout", LAYOUTS, ids=LAYOUT_IDS)
@pytest.mark.parametrize("mode,pair", [mp for mp in _modes_and_kernels() if mp[0] != "simt"])
def test_mn_major_operands_whole_blocks(mode, pair, layout, monkeypatch):
    """M and N multiples of 128: an MN-major operand (A stored K x M, B
    stored K x N) is read through a 3-D tensor map, one TMA load per stage
    for all its 128-byte column blocks; K stays ragged."""
    monkeypatch.setenv("DGEMM_TC_PAIR", pair)
    ta, tb = layout
    for (M, N, K) in [(256, 512, 200), (640, 384, 333), (128, 128, 1000)]:
        A, B = inputs.make_random(M, N, K, seed=M + 2 * N + K, dist="normal",
                                  dtype=gu.in_dtype(mode))
        buf, C = gu.guarded_output(M, N, N + 4)
        C = _run(mode, A, B, ta, tb, out=C)
        ref, S = gu.oracle_full(A, B)
        gu.assert_close(C.cpu().numpy(), ref, S, gu.TOL[mode],
                        f"{mode} pair={pair} {'T' if ta else 'N'}{'T' if tb else 'N'} {M}x{N}x{K}")
        gu.assert_guards_intact(buf, M, N, N + 4)
