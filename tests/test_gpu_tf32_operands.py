"""How the tensor core reads fp32 operands in TF32 mode, pinned on the GPU.

The 3xTF32 split relies on it: the raw fp32 tile serves as the hi part, so
the tensor core must read an fp32 value x as trunc_tf32(x), x with its low 13
mantissa bits dropped (rounding toward zero).  With x = 1 + 2^-11 + 2^-12
(0.75 of a TF32 unit above 1) truncation gives exactly 1 while rounding to
nearest would give 1 + 2^-10; both are exact fp32 results of a 1 x 1 x 1
product, so the check is bit-exact and independent of accumulation order.
"""
import numpy as np
import pytest
import torch

import gpu_util as gu

pytestmark = pytest.mark.gpu

X = 1.0 + 2.0 ** -11 + 2.0 ** -12


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.mark.parametrize("pair", ["0", "1"])
def test_tf32_reads_operands_by_truncation(pair, monkeypatch):
    monkeypatch.setenv("DGEMM_TC_PAIR", pair)
    # 3 + 7 * 2^-11 is 1.75 TF32 units (2^-9 each in [2, 4)) above 3: truncation
    # gives 3 + 2^-9, rounding to nearest would give 3 + 2^-8.
    for a, b, want in [(X, 1.0, 1.0), (-X, 1.0, -1.0), (1.0, X, 1.0), (X, X, 1.0),
                       (3.0 + 7 * 2.0 ** -11, 1.0, 3.0 + 2.0 ** -9)]:
        A = torch.tensor([[a]], dtype=torch.float32, device="cuda")
        B = torch.tensor([[b]], dtype=torch.float32, device="cuda")
        C = gu.run("tf32", A, B).item()
        assert C == want, f"tf32({a!r} x {b!r}) = {C!r}, truncation gives {want!r}"


def test_3xtf32_recovers_the_dropped_bits():
    """The same operands through 3xTF32 give the fp32-exact product."""
    A = torch.tensor([[X, -X]], dtype=torch.float32, device="cuda")
    B = torch.tensor([[1.0], [2.0 ** -12]], dtype=torch.float32, device="cuda")
    want = np.float32(X) * 1.0 + np.float32(-X) * np.float32(2.0 ** -12)
    C = gu.run("3xtf32", A, B).item()
    assert abs(C - float(want)) <= 2.0 ** -22 * abs(float(want))
