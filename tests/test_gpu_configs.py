"""Parity of every GPU path with the CPU oracle on the benchmark workloads.

Shapes, seeds and distributions are the five workloads of the benchmark
configuration (dense_gemm_f32_gb300.inputs).  Small and medium shapes are
compared element by element against the full oracle; the two large ones
(8192^3 and the 16384 x 14336 x 4096 transformer layer), run through the same
call and launch configuration bench.py times, are compared on sampled rows
that the oracle computes one by one.  Tolerances: |C - C_exact| <= tol * S,
S = |A| x |B|, tol 1e-5 (SIMT, 3xTF32), 2e-3 (TF32), 8e-3 (BF16).
"""
import numpy as np
import pytest
import torch

import gpu_util as gu
from dense_gemm_f32_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    gu.check_watchdog()


def _full_case(w, mode):
    A, B = inputs.make(w)
    if mode in gu.LOW_MODES and A.dtype != gu.in_dtype(mode):
        A, B = A.float().to(gu.in_dtype(mode)), B.float().to(gu.in_dtype(mode))
    C = gu.run(mode, A.cuda(), B.cuda())
    ref, S = gu.oracle_full(A, B)
    gu.assert_close(C.cpu().numpy(), ref, S, gu.TOL[mode], f"{w.name} {mode}")
    return C, ref, S


@pytest.mark.parametrize("mode", gu.ALL_MODES)
def test_square_64(mode):
    _full_case(inputs.SQUARE_64, mode)


@pytest.mark.parametrize("mode", gu.ALL_MODES)
def test_square_64_integer_bit_exact(mode):
    """Entries in {-4..4}, K = 64: every product and partial sum is an integer
    below 2^24, exact in fp32, TF32 and BF16 alike, so C must equal the exact
    product bit for bit (the 3xTF32 lo parts are zero)."""
    A, B = inputs.make_integer(64, 64, 64, seed=inputs.SQUARE_64.seed)
    A, B = A.to(gu.in_dtype(mode)), B.to(gu.in_dtype(mode))
    C = gu.run(mode, A.cuda(), B.cuda()).cpu().numpy()
    exact = (A.float().numpy().astype(np.int64) @ B.float().numpy().astype(np.int64))
    assert np.array_equal(C.astype(np.float64), exact.astype(np.float64))


@pytest.mark.parametrize("mode", gu.ALL_MODES)
def test_integer_bit_exact_k1024(mode):
    """The bit-exact case at its largest K (1024): |partial sums| <= 16 * 1024."""
    A, B = inputs.make_integer(300, 260, 1024, seed=9)
    A, B = A.to(gu.in_dtype(mode)), B.to(gu.in_dtype(mode))
    C = gu.run(mode, A.cuda(), B.cuda()).cpu().numpy()
    exact = (A.float().numpy().astype(np.int64) @ B.float().numpy().astype(np.int64))
    assert np.array_equal(C.astype(np.float64), exact.astype(np.float64))


@pytest.mark.parametrize("mode", gu.ALL_MODES)
def test_square_1024(mode):
    _full_case(inputs.SQUARE_1024, mode)


@pytest.mark.parametrize("mode", gu.ALL_MODES)
def test_ragged_1000x1013x997(mode):
    """lda = 997, ldb = ldc = 1013: no row after the first starts on a 16-byte
    boundary, so the tensor-core paths re-pitch A and B and every path
    stores C with masked scalar writes."""
    _full_case(inputs.RAGGED_1000, mode)


def _sampled(w, mode, nrows=48):
    A, B = inputs.make(w)
    if mode in gu.LOW_MODES and A.dtype != gu.in_dtype(mode):
        A, B = A.float().to(gu.in_dtype(mode)), B.float().to(gu.in_dtype(mode))
    C = gu.run(mode, A.cuda(), B.cuda())
    g = np.random.default_rng(w.seed)
    rows = np.unique(np.concatenate([[0, 127, 128, w.M - 1],
                                     g.choice(w.M, nrows, replace=False)]))
    Cr = C[torch.from_numpy(rows).cuda()].cpu().numpy()
    del C
    ref, S = gu.oracle_rows(A, B, rows)
    gu.assert_close(Cr, ref, S, gu.TOL[mode], f"{w.name} {mode} (rows {len(rows)})")


@pytest.mark.parametrize("mode", ["simt", "tf32", "3xtf32"])
def test_square_8192_sampled_rows(mode):
    _sampled(inputs.SQUARE_8192, mode)


def test_transformer_bf16_sampled_rows():
    _sampled(inputs.TRANSFORMER_BF16, "bf16", nrows=24)


def test_transformer_tf32_sampled_rows():
    _sampled(inputs.TRANSFORMER_F32, "tf32", nrows=24)


def test_transformer_fp16_sampled_rows():
    """The transformer-layer draws rounded to fp16 instead of bf16."""
    _sampled(inputs.TRANSFORMER_F16, "fp16", nrows=24)


@pytest.mark.parametrize("mode", ["e4m3", "e5m2"])
def test_transformer_fp8_sampled_rows(mode):
    """The transformer-layer draws rounded to FP8 (scale 1), through the
    default row-major B (transposed into K-major scratch first)."""
    _sampled(inputs.TRANSFORMER_E4M3 if mode == "e4m3" else inputs.TRANSFORMER_E5M2, mode,
             nrows=24)
