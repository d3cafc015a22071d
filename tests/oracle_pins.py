"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each pin takes a candidate `gemm(A, B) -> C` (float32 numpy inputs, float64
output) and raises AssertionError when the candidate disagrees with what
the pages or the mathematics fix.  tests/test_oracle.py runs every pin on
the oracle and also on deliberately broken candidates (a transposed
operand, a dropped term, a wrong sign, a shifted index, float32
accumulation) to show that each plausible mistake is caught by some pin.

Definition being pinned: "第八课：GPU 如何完成矩阵乘法" (Lesson 8), section 一,
C[i][j] = sum_{k<K} A[i][k]*B[k][j].
"""
from fractions import Fraction

import numpy as np

import golden_io

U53 = 2.0 ** -53


def _rng(seed):
    return np.random.default_rng(seed)


def _rand(rng, shape, kind="uniform"):
    if kind == "uniform":
        return (2 * rng.random(shape) - 1).astype(np.float32)
    if kind == "normal":
        return rng.standard_normal(shape).astype(np.float32)
    if kind == "int":
        return rng.integers(-4, 5, size=shape).astype(np.float32)
    raise ValueError(kind)


def _exact(A, B):
    """Exact rational product by brute force (pure Python; tiny inputs only)."""
    M, K = A.shape
    N = B.shape[1]
    Af = [[Fraction(float(A[i, k])) for k in range(K)] for i in range(M)]
    Bf = [[Fraction(float(B[k, j])) for j in range(N)] for k in range(K)]
    return [[sum((Af[i][k] * Bf[k][j] for k in range(K)), Fraction(0)) for j in range(N)]
            for i in range(M)]


def pin_golden(gemm):
    """Hand-computed products in tests/golden/ are reproduced exactly."""
    cases = golden_io.all_cases()
    assert cases, "no golden fixtures found"
    for path in cases:
        blk = golden_io.load(path)
        A = blk["A"].astype(np.float32)
        B = blk["B"].astype(np.float32)
        C = np.asarray(gemm(A, B))
        assert C.shape == blk["C"].shape, f"{path}: shape {C.shape} != {blk['C'].shape}"
        assert np.array_equal(C, blk["C"]), f"{path}: got\n{C}\nexpected\n{blk['C']}"


def pin_exact_rational(gemm):
    """Within the rounding bound of the exact rational product, brute force.
    With products exact in double and K-1 rounded additions the error is at
    most (K-1)*u*S with u = 2^-53; float32 accumulation would exceed it."""
    rng = _rng(11)
    for (M, N, K) in [(3, 4, 5), (5, 3, 9), (4, 6, 17), (2, 2, 33)]:
        A = _rand(rng, (M, K), "normal")
        B = _rand(rng, (K, N), "normal")
        E = _exact(A, B)
        C = np.asarray(gemm(A, B))
        assert C.shape == (M, N)
        for i in range(M):
            for j in range(N):
                S = sum(abs(float(A[i, k])) * abs(float(B[k, j])) for k in range(K))
                err = abs(Fraction(float(C[i, j])) - E[i][j])
                bound = Fraction(max(K - 1, 1) * 1.01 * U53 * S)
                assert err <= bound, f"({M},{N},{K}) [{i},{j}] err {float(err):.3e} > {float(bound):.3e}"


def pin_integer_exact(gemm):
    """Integer-valued inputs give the exact integer product (brute force on
    tiny shapes, numpy's exact int64 matmul on larger ones)."""
    rng = _rng(12)
    A = _rand(rng, (4, 7), "int")
    B = _rand(rng, (7, 5), "int")
    E = _exact(A, B)
    C = np.asarray(gemm(A, B))
    assert all(C[i, j] == E[i][j] for i in range(4) for j in range(5))
    for (M, N, K) in [(64, 64, 64), (33, 17, 129)]:
        A = _rand(rng, (M, K), "int")
        B = _rand(rng, (K, N), "int")
        E = A.astype(np.int64) @ B.astype(np.int64)
        assert np.array_equal(np.asarray(gemm(A, B)), E.astype(np.float64))


def pin_identity_zero(gemm):
    """A*I = A and I*B = B exactly; a zero factor gives zero; K = 0 gives the
    empty sum, zero."""
    rng = _rng(13)
    A = _rand(rng, (5, 7))
    B = _rand(rng, (7, 6))
    assert np.array_equal(np.asarray(gemm(A, np.eye(7, dtype=np.float32))), A.astype(np.float64))
    assert np.array_equal(np.asarray(gemm(np.eye(5, dtype=np.float32), A)), A.astype(np.float64))
    assert np.array_equal(np.asarray(gemm(np.zeros((5, 7), np.float32), B)), np.zeros((5, 6)))
    C0 = np.asarray(gemm(np.zeros((3, 0), np.float32), np.zeros((0, 4), np.float32)))
    assert C0.shape == (3, 4) and np.array_equal(C0, np.zeros((3, 4)))


def pin_transpose(gemm):
    """(A B)^T = B^T A^T.  The same products are added in the same k order on
    both sides, so the identity holds bit for bit."""
    rng = _rng(14)
    A = _rand(rng, (6, 9), "normal")
    B = _rand(rng, (9, 4), "normal")
    C = np.asarray(gemm(A, B))
    Ct = np.asarray(gemm(np.ascontiguousarray(B.T), np.ascontiguousarray(A.T)))
    assert np.array_equal(C.T, Ct)


def pin_k_slabs(gemm):
    """Lesson 8 section 九: a tile's result is the sum over K-slabs of the
    slab products; K = 64 as 4 slabs of 16.  Exact on integer inputs, within
    the rounding bound on real-valued ones."""
    rng = _rng(15)
    for kind in ("int", "uniform"):
        A = _rand(rng, (16, 64), kind)
        B = _rand(rng, (64, 16), kind)
        C = np.asarray(gemm(A, B))
        parts = [np.asarray(gemm(np.ascontiguousarray(A[:, 16 * t:16 * t + 16]),
                                 np.ascontiguousarray(B[16 * t:16 * t + 16, :]))) for t in range(4)]
        Csum = parts[0] + parts[1] + parts[2] + parts[3]
        if kind == "int":
            assert np.array_equal(C, Csum)
        else:
            S = np.abs(A).astype(np.float64) @ np.abs(B).astype(np.float64)
            assert np.all(np.abs(C - Csum) <= 64 * 2 * U53 * S)


def pin_numpy_f64(gemm):
    """numpy's float64 matmul of the widened inputs agrees within the rounding
    bound 2*K*u*S (both sides round; neither is exact)."""
    rng = _rng(16)
    for (M, N, K) in [(31, 47, 129), (64, 1, 300), (1, 50, 77)]:
        A = _rand(rng, (M, K), "normal")
        B = _rand(rng, (K, N), "normal")
        ref = A.astype(np.float64) @ B.astype(np.float64)
        S = np.abs(A).astype(np.float64) @ np.abs(B).astype(np.float64)
        C = np.asarray(gemm(A, B))
        assert C.shape == (M, N)
        assert np.all(np.abs(C - ref) <= 2.0 * K * U53 * S + 1e-300)


ALL_PINS = [pin_golden, pin_exact_rational, pin_integer_exact, pin_identity_zero,
            pin_transpose, pin_k_slabs, pin_numpy_f64]


def failures(gemm):
    """Names of the pins that `gemm` fails (an exception counts as a failure)."""
    bad = []
    for pin in ALL_PINS:
        try:
            pin(gemm)
        except Exception:  # noqa: BLE001 - any failure of a candidate counts
            bad.append(pin.__name__)
    return bad
