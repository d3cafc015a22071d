"""The TF32 and BF16 paths have two tensor-core kernels: a single-CTA kernel
(128 x 256 tiles) and a CTA-pair kernel (256 x 256 tiles on two SMs).  The
library picks one by problem size; DGEMM_TC_PAIR=0 / =1 forces either, and
these tests run the edge cases through both against the CPU oracle."""
import numpy as np
import pytest
import torch

import gpu_util as gu
from dense_gemm_f32_gb300 import inputs
import dense_gemm_f32_gb300 as dg

pytestmark = pytest.mark.gpu

KERNELS = ["0", "1"]  # single-CTA, pair


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    gu.check_watchdog()


def _check(mode, A, B, what, Ad=None, Bd=None, out=None):
    C = gu.run(mode, A.cuda() if Ad is None else Ad, B.cuda() if Bd is None else Bd, out)
    ref, S = gu.oracle_full(A, B)
    gu.assert_close(C.cpu().numpy(), ref, S, gu.TOL[mode], what)
    return C


@pytest.mark.parametrize("pair", KERNELS)
@pytest.mark.parametrize("mode", gu.TC_MODES)
def test_shapes_both_kernels(mode, pair, monkeypatch):
    monkeypatch.setenv("DGEMM_TC_PAIR", pair)
    for (M, N, K) in [(1, 1, 1), (7, 300, 33), (129, 257, 65), (255, 129, 100), (256, 256, 32),
                      (257, 513, 200), (600, 130, 1000), (1000, 1013, 997)]:
        A, B = inputs.make_random(M, N, K, seed=M + 3 * N + 7 * K, dist="normal",
                                  dtype=gu.in_dtype(mode))
        _check(mode, A, B, f"{mode} pair={pair} {M}x{N}x{K}")


@pytest.mark.parametrize("pair", KERNELS)
@pytest.mark.parametrize("mode", gu.TC_MODES)
def test_many_tiles_and_long_k(mode, pair, monkeypatch):
    """More pair tiles than clusters (several tiles per cluster, both
    accumulator buffers, pipeline wrap-around) and a long ragged K."""
    monkeypatch.setenv("DGEMM_TC_PAIR", pair)
    A, B = inputs.make_random(4100, 2100, 100, seed=24, dtype=gu.in_dtype(mode))
    _check(mode, A, B, f"{mode} pair={pair} many tiles")
    A, B = inputs.make_random(300, 520, 5000, seed=25, dtype=gu.in_dtype(mode))
    _check(mode, A, B, f"{mode} pair={pair} long K")


@pytest.mark.parametrize("pair", KERNELS)
@pytest.mark.parametrize("mode", gu.TC_MODES)
def test_guard_bands_and_misaligned(mode, pair, monkeypatch):
    monkeypatch.setenv("DGEMM_TC_PAIR", pair)
    M, N, K = 301, 517, 173
    A, B = inputs.make_random(M, N, K, seed=31, dist="normal", dtype=gu.in_dtype(mode))
    ldc = N + 7
    Ad = gu.device_view(*inputs.embed(A, K + 8))
    Bd = gu.device_view(*inputs.embed(B, N + 3, offset=1))
    buf, C = gu.guarded_output(M, N, ldc)
    _check(mode, A, B, f"{mode} pair={pair} ld/guard", Ad, Bd, C)
    gu.assert_guards_intact(buf, M, N, ldc)


@pytest.mark.parametrize("mode", gu.TC_MODES)
def test_integer_bit_exact_both_kernels(mode, monkeypatch):
    A, B = inputs.make_integer(300, 520, 1024, seed=9)
    A, B = A.to(gu.in_dtype(mode)), B.to(gu.in_dtype(mode))
    exact = (A.float().numpy().astype(np.int64) @ B.float().numpy().astype(np.int64))
    for pair in KERNELS:
        monkeypatch.setenv("DGEMM_TC_PAIR", pair)
        C = gu.run(mode, A.cuda(), B.cuda()).cpu().numpy()
        assert np.array_equal(C.astype(np.float64), exact.astype(np.float64)), pair


@pytest.mark.parametrize("mode", gu.TC_MODES)
def test_pair_deterministic_and_counted(mode, monkeypatch):
    monkeypatch.setenv("DGEMM_TC_PAIR", "1")
    A, B = inputs.make_random(1024, 1024, 512, seed=41, dtype=gu.in_dtype(mode))
    Ad, Bd = A.cuda(), B.cuda()
    n0 = dg.dgemm_kernel_launches()
    C1 = gu.run(mode, Ad, Bd).clone()
    C2 = gu.run(mode, Ad, Bd)
    # FP8 transposes B first, 3xTF32 writes the lo parts of A and B first
    assert dg.dgemm_kernel_launches() - n0 == (4 if mode in gu.F8_MODES or mode == "3xtf32" else 2)
    assert torch.equal(C1, C2)
