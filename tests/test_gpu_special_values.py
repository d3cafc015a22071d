"""Infinities and NaNs in A and B, on every path, against the CPU oracle.

The oracle sums in IEEE double, so an infinite product makes its entry of C
infinite, opposite infinities or an infinity times zero make it NaN, and a
NaN operand makes NaN.  Every GPU path must give the same class (NaN, +Inf,
-Inf, finite) in every entry, and the finite entries must meet the mode's
tolerance.  E4M3 has no infinities (they round to NaN), so it gets NaNs only.

One exception, inherent in split precision: 3xTF32 adds the cross products
a_hi*b_lo and a_lo*b_hi, so an infinite a meeting a finite b whose low part is
exactly zero (b already a TF32 value, about one b in 8192) gives inf * 0 =
NaN where the exact entry is infinite.  The split keeps infinities and NaNs
out of the low parts, which leaves that coincidence as the only difference.
"""
import numpy as np
import pytest
import torch

import gpu_util as gu
from dense_gemm_f32_gb300 import inputs
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    gu.check_watchdog()


def _plant(A, B, mode):
    A, B = A.float().clone(), B.float().clone()
    inf = float("inf") if mode != "e4m3" else float("nan")
    A[3, 5] = inf          # row 3 of C infinite where B[5, j] != 0 ...
    B[5, 11] = 0.0         # ... and NaN at (3, 11): inf * 0
    A[7, 2] = float("nan")  # row 7 of C all NaN
    B[4, 9] = -inf         # column 9 of C -inf where A[i, 4] != 0 (NaN where it meets +inf)
    A[10, 4] = 0.0
    return A.to(gu.in_dtype(mode)), B.to(gu.in_dtype(mode))


def _classes(X):
    return np.where(np.isnan(X), 0, np.where(np.isposinf(X), 1, np.where(np.isneginf(X), 2, 3)))


@pytest.mark.parametrize("pair", ["0", "1"])
@pytest.mark.parametrize("mode", gu.ALL_MODES)
def test_special_values_propagate_like_ieee(mode, pair, monkeypatch):
    monkeypatch.setenv("DGEMM_TC_PAIR", pair)
    for (M, N, K) in [(64, 80, 48), (300, 260, 1024)]:
        A, B = inputs.make_random(M, N, K, seed=M + N, dist="normal", dtype=torch.float32)
        A, B = _plant(A, B, mode)
        C = gu.run(mode, A.cuda(), B.cuda()).cpu().numpy().astype(np.float64)
        An, Bn = A.float().numpy(), B.float().numpy()
        ref, S = oracle.gemm(An, Bn), oracle.abs_gemm(An, Bn)
        assert np.isnan(ref[7]).all() and np.isnan(ref[3, 11])
        bad = _classes(C) != _classes(ref)
        if mode == "3xtf32":
            bad &= ~(np.isinf(ref) & np.isnan(C))
        assert not bad.any(), (f"{mode} pair={pair} {M}x{N}x{K}: {int(bad.sum())} entries of the "
                               f"wrong class, first {np.argwhere(bad)[0].tolist()}")
        fin = np.isfinite(ref) & np.isfinite(S)
        gu.assert_close(np.where(fin, C, 0.0), np.where(fin, ref, 0.0), np.where(fin, S, 0.0),
                        gu.TOL[mode], f"{mode} pair={pair} finite entries")
