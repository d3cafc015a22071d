"""Helpers for the GPU parity tests: tolerances, comparison, guarded buffers."""
import numpy as np
import torch

import oracle

# |C - C_exact| <= tol * S elementwise, S = |A| x |B|; one tolerance per mode.
# fp16 and fp8: the inputs are exact and so are their products in fp32; only
# the fp32 accumulation rounds (once per MMA instruction, K/16 or K/32 times:
# below 6e-5 at K = 16384), plus the rounding inside one instruction's sum.
TOL = {"simt": 1e-5, "3xtf32": 1e-5, "tf32": 2e-3, "bf16": 8e-3, "fp16": 2e-4,
       "e4m3": 2e-4, "e5m2": 2e-4}
FP32_MODES = ("simt", "tf32", "3xtf32")
HALF_MODES = ("bf16", "fp16")
F8_MODES = ("e4m3", "e5m2")
LOW_MODES = HALF_MODES + F8_MODES  # inputs narrower than fp32
ALL_MODES = ("simt", "tf32", "3xtf32", "bf16", "fp16", "e4m3", "e5m2")
TC_MODES = ("tf32", "3xtf32", "bf16", "fp16", "e4m3", "e5m2")


def in_dtype(mode):
    return {"bf16": torch.bfloat16, "fp16": torch.float16, "e4m3": torch.float8_e4m3fn,
            "e5m2": torch.float8_e5m2}.get(mode, torch.float32)


def elem_bytes(mode):
    return 1 if mode in F8_MODES else 2 if mode in HALF_MODES else 4


def np_inputs(A, B):
    """float32 numpy copies of CPU tensors (bf16, fp16 and fp8 widen exactly)."""
    return A.float().numpy(), B.float().numpy()


def assert_close(got, ref, S, tol, what=""):
    """Elementwise err <= tol * S; finite everywhere; exact zero where S == 0."""
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} != {ref.shape}"
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = ~(err <= tol * S)
    if bad.any():
        i, j = np.argwhere(bad)[0]
        ratio = float(np.max(err / np.where(S > 0, S, 1.0)))
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements beyond {tol}*S "
            f"(max err/S {ratio:.3e}); first ({i},{j}): got {got[i, j]!r} want {ref[i, j]!r} "
            f"S {S[i, j]!r}")


def max_rel(got, ref, S):
    got = np.asarray(got, dtype=np.float64)
    return float(np.max(np.abs(got - ref) / np.where(S > 0, S, 1.0))) if got.size else 0.0


def run(mode, A_dev, B_dev, out=None):
    import dense_gemm_f32_gb300 as dg

    C = dg.matmul(A_dev, B_dev, mode=mode, out=out)
    torch.cuda.synchronize()
    return C


def check_watchdog():
    import dense_gemm_f32_gb300 as dg

    st, where = dg.dgemm_watchdog_status(torch.cuda.current_stream().cuda_stream)
    assert st == dg.OK, f"watchdog tripped at site {where:#x}"


def oracle_full(A, B):
    An, Bn = np_inputs(A, B)
    return oracle.gemm(An, Bn), oracle.abs_gemm(An, Bn)


def oracle_rows(A, B, rows):
    An, Bn = np_inputs(A, B)
    return oracle.gemm_rows(An, Bn, rows)


SENTINEL = float.fromhex("0x1.dead00p+100")


def guarded_output(M, N, ldc, margin=64, device="cuda"):
    """A float32 buffer holding an M x N matrix at row pitch ldc, `margin`
    elements of sentinel before and after it, sentinel in the ldc gap too.
    Returns (buffer, view)."""
    total = margin + (M - 1) * ldc + N + margin if M and N else 2 * margin
    buf = torch.full((total,), SENTINEL, dtype=torch.float32, device=device)
    view = buf.as_strided((M, N), (ldc, 1), margin)
    return buf, view


def assert_guards_intact(buf, M, N, ldc, margin=64):
    h = buf.cpu().numpy()
    mask = np.ones(h.shape, dtype=bool)
    for r in range(M):
        mask[margin + r * ldc: margin + r * ldc + N] = False
    touched = np.argwhere(mask & (h != np.float32(SENTINEL)))
    assert touched.size == 0, f"wrote outside C: first offsets {touched[:5].ravel().tolist()}"


def device_view(buf, view):
    """Copy a host buffer to the GPU and rebuild the same strided window on it
    (keeps the leading dimension and the storage offset, hence the alignment)."""
    dbuf = buf.cuda()
    return dbuf.as_strided(tuple(view.shape), tuple(view.stride()), view.storage_offset())
