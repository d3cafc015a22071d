"""The CPU oracle against its pins (CPU only).

The oracle is what every GPU result is judged by, so before it is trusted
it is checked against things other than itself: hand-computed products
(tests/golden/), exact rational brute force, integer inputs, identity and
zero factors, the transpose identity, the K-slab decomposition of
Lesson 8 section 九, and numpy's float64 matmul.  A second group plants
plausible mistakes in copies of the oracle and shows that the pins catch
every one of them.
"""
import numpy as np
import pytest

import oracle
import oracle_pins
import golden_io
from dense_gemm_f32_gb300 import inputs


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_passes_pin(pin):
    pin(oracle.gemm)


def test_abs_gemm_golden():
    """S = |A| x |B| on the hand-computed 3x3 case."""
    blk = golden_io.load(golden_io.GOLDEN_DIR + "/hand_3x3_frac.txt")
    S = oracle.abs_gemm(blk["A"].astype(np.float32), blk["B"].astype(np.float32))
    assert np.array_equal(S, blk["S"])


def test_abs_gemm_properties():
    """S(A, B) = C(|A|, |B|) bit for bit, S >= |C|, and S = C for nonnegative
    factors."""
    rng = np.random.default_rng(21)
    A = rng.standard_normal((13, 29)).astype(np.float32)
    B = rng.standard_normal((29, 11)).astype(np.float32)
    S = oracle.abs_gemm(A, B)
    assert np.array_equal(S, oracle.gemm(np.abs(A), np.abs(B)))
    assert np.all(S >= np.abs(oracle.gemm(A, B)))
    assert np.array_equal(oracle.abs_gemm(np.abs(A), np.abs(B)), oracle.gemm(np.abs(A), np.abs(B)))


def test_leading_dimensions():
    """A matrix read through a leading dimension larger than its width (the
    rest of each row is NaN padding) gives the compact result bit for bit."""
    rng = np.random.default_rng(22)
    A = rng.standard_normal((9, 13)).astype(np.float32)
    B = rng.standard_normal((13, 10)).astype(np.float32)
    ref = oracle.gemm(A, B)
    Abuf = np.full((9, 21), np.nan, dtype=np.float32)
    Bbuf = np.full((13, 17), np.nan, dtype=np.float32)
    Abuf[:, :13] = A
    Bbuf[:, :10] = B
    got = oracle.gemm(Abuf[:, :13], Bbuf[:, :10])
    assert np.array_equal(got, ref)


def test_rows_variant_matches_full():
    rng = np.random.default_rng(23)
    A = rng.standard_normal((40, 70)).astype(np.float32)
    B = rng.standard_normal((70, 33)).astype(np.float32)
    C = oracle.gemm(A, B)
    S = oracle.abs_gemm(A, B)
    rows = np.array([0, 7, 39, 7, 12])
    Cr, Sr = oracle.gemm_rows(A, B, rows)
    assert np.array_equal(Cr, C[rows])
    assert np.array_equal(Sr, S[rows])


def test_thread_count_does_not_change_results():
    A, B = inputs.make_random(70, 50, 90, seed=5)
    A, B = A.numpy(), B.numpy()
    n0 = oracle.max_threads()
    try:
        oracle.set_threads(1)
        c1 = oracle.gemm(A, B)
        oracle.set_threads(max(n0, 2))
        c2 = oracle.gemm(A, B)
    finally:
        oracle.set_threads(n0)
    assert np.array_equal(c1, c2)


def test_shape_mismatch_rejected():
    with pytest.raises(ValueError):
        oracle.gemm(np.zeros((2, 3), np.float32), np.zeros((4, 2), np.float32))
    with pytest.raises(TypeError):
        oracle.gemm(np.zeros((2, 3), np.float64), np.zeros((3, 2), np.float32))


# ---------------------------------------------------------------------------
# Planted mistakes: each broken copy of the definition must fail some pin.
# ---------------------------------------------------------------------------

def _f64(X):
    return np.asarray(X, dtype=np.float64)


def _mut_transposed_b(A, B):
    return _f64(A) @ _f64(B).T


def _mut_transposed_a(A, B):
    return _f64(A).T @ _f64(B)


def _mut_drop_last_k(A, B):
    return _f64(A)[:, :-1] @ _f64(B)[:-1, :]


def _mut_drop_first_k(A, B):
    return _f64(A)[:, 1:] @ _f64(B)[1:, :]


def _mut_sign_last_k(A, B):
    A, B = _f64(A), _f64(B)
    if A.shape[1] == 0:
        return np.zeros((A.shape[0], B.shape[1]))
    return A[:, :-1] @ B[:-1, :] - np.outer(A[:, -1], B[-1, :])


def _mut_shifted_column(A, B):
    return _f64(A) @ np.roll(_f64(B), 1, axis=1)


def _mut_output_transposed(A, B):
    return (_f64(A) @ _f64(B)).T


def _mut_f32_accumulate(A, B):
    A = np.asarray(A, np.float32)
    B = np.asarray(B, np.float32)
    C = np.zeros((A.shape[0], B.shape[1]), np.float32)
    for k in range(A.shape[1]):
        C = C + np.outer(A[:, k], B[k, :]).astype(np.float32)
    return C.astype(np.float64)


MUTANTS = [_mut_transposed_b, _mut_transposed_a, _mut_drop_last_k, _mut_drop_first_k,
           _mut_sign_last_k, _mut_shifted_column, _mut_output_transposed, _mut_f32_accumulate]


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda f: f.__name__)
def test_pins_catch_planted_mistake(mutant):
    assert oracle_pins.failures(mutant), f"{mutant.__name__} passed every pin"


def test_pins_accept_float64_library_product():
    """Sanity of the pins themselves: numpy's float64 matmul of the widened
    inputs (a different but correct summation) passes every pin except the
    bit-level ones that fix the k order."""
    bad = oracle_pins.failures(lambda A, B: _f64(A) @ _f64(B))
    assert set(bad) <= {"pin_transpose", "pin_k_slabs"}, bad
