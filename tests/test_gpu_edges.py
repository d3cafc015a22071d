"""Edge cases of every GPU path against the CPU oracle.

Boundary sizes around every tile edge (Lesson 8 section 二十六: partial last
tiles are zero-filled on load and masked on store), leading dimensions above
the minimum, operands whose rows are not 16-byte aligned, guard bands around
C (nothing outside the M x N region may change), K = 0, one-row and
one-column shapes, long K loops, more tiles than SMs, determinism, and the
rejection of host pointers.
"""
import numpy as np
import pytest
import torch

import gpu_util as gu
from dense_gemm_f32_gb300 import inputs
import dense_gemm_f32_gb300 as dg

pytestmark = pytest.mark.gpu

EDGE = [1, 2, 3, 7, 8, 15, 16, 17, 31, 33, 63, 65, 127, 129, 255, 257]
# every edge value appears in every dimension, combined with different others
SWEEP = sorted({(EDGE[i], EDGE[(i + 5) % 16], EDGE[(i + 11) % 16]) for i in range(16)}
               | {(EDGE[(i + 3) % 16], EDGE[i], EDGE[(i + 7) % 16]) for i in range(16)}
               | {(EDGE[(i + 9) % 16], EDGE[(i + 2) % 16], EDGE[i]) for i in range(16)})


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    gu.check_watchdog()


def _check(mode, A, B, what, Adev=None, Bdev=None, out=None):
    C = gu.run(mode, A.cuda() if Adev is None else Adev, B.cuda() if Bdev is None else Bdev, out)
    ref, S = gu.oracle_full(A, B)
    gu.assert_close(C.cpu().numpy(), ref, S, gu.TOL[mode], what)
    return C


@pytest.mark.parametrize("mode", gu.ALL_MODES)
def test_boundary_sweep(mode):
    for (M, N, K) in SWEEP:
        A, B = inputs.make_random(M, N, K, seed=M * 1000003 + N * 1009 + K,
                                  dist="normal", dtype=gu.in_dtype(mode))
        _check(mode, A, B, f"{mode} {M}x{N}x{K}")


@pytest.mark.parametrize("mode", gu.ALL_MODES)
def test_degenerate_shapes(mode):
    for (M, N, K) in [(1, 1, 1), (1, 1, 4096), (1, 777, 33), (777, 1, 33), (5, 3, 1),
                      (129, 257, 1), (1, 4096, 1)]:
        A, B = inputs.make_random(M, N, K, seed=17, dist="uniform", dtype=gu.in_dtype(mode))
        _check(mode, A, B, f"{mode} {M}x{N}x{K}")


@pytest.mark.parametrize("mode", gu.ALL_MODES)
def test_long_k_and_many_tiles(mode):
    """K = 5000 (many pipeline wraps, ragged last k-block) and a 4100 x 2100
    output (more tiles than SMs, so the persistent CTAs take several tiles
    and both accumulator buffers)."""
    A, B = inputs.make_random(130, 270, 5000, seed=23, dtype=gu.in_dtype(mode))
    _check(mode, A, B, f"{mode} long K")
    A, B = inputs.make_random(4100, 2100, 100, seed=24, dtype=gu.in_dtype(mode))
    _check(mode, A, B, f"{mode} many tiles")


@pytest.mark.parametrize("mode", gu.ALL_MODES)
def test_k_zero_sets_c_to_zero(mode):
    M, N = 70, 90
    A = torch.zeros((M, 0), dtype=gu.in_dtype(mode), device="cuda")
    B = torch.zeros((0, N), dtype=gu.in_dtype(mode), device="cuda")
    buf, C = gu.guarded_output(M, N, ldc=N + 3)
    gu.run(mode, A, B, out=C)
    assert torch.count_nonzero(C).item() == 0
    gu.assert_guards_intact(buf, M, N, N + 3)


@pytest.mark.parametrize("mode", gu.ALL_MODES)
def test_leading_dimensions_and_guard_bands(mode):
    """A, B, C read/written through leading dimensions above the minimum, with
    NaN in the padding of A and B and a sentinel around and inside C's gaps."""
    M, N, K = 301, 259, 173
    A, B = inputs.make_random(M, N, K, seed=31, dist="normal", dtype=gu.in_dtype(mode))
    for (lda, ldb, ldc) in [(K + 3, N + 5, N + 7), (K + 8, N + 8, N + 8), (2 * K, 2 * N, 3 * N)]:
        Ad = gu.device_view(*inputs.embed(A, lda))
        Bd = gu.device_view(*inputs.embed(B, ldb))
        assert Ad.stride(0) == lda and Bd.stride(0) == ldb
        buf, C = gu.guarded_output(M, N, ldc)
        out = gu.run(mode, Ad, Bd, out=C)
        ref, S = gu.oracle_full(A, B)
        gu.assert_close(out.cpu().numpy(), ref, S, gu.TOL[mode], f"{mode} ld {lda},{ldb},{ldc}")
        gu.assert_guards_intact(buf, M, N, ldc)


@pytest.mark.parametrize("mode", gu.ALL_MODES)
def test_misaligned_bases(mode):
    """Base pointers 1..3 elements past a 16-byte boundary (fp32), 1..7 (16-bit)
    or 1..15 (8-bit): not 16-byte aligned, so no 128-bit or TMA access may
    start there."""
    M, N, K = 190, 150, 90
    es = gu.elem_bytes(mode)
    A, B = inputs.make_random(M, N, K, seed=37, dtype=gu.in_dtype(mode))
    for off in range(1, 16 // es):
        Ad = gu.device_view(*inputs.embed(A, K, offset=off))
        Bd = gu.device_view(*inputs.embed(B, N, offset=(off * 3) % (16 // es)))
        buf = torch.full((1 + M * N + 8,), gu.SENTINEL, dtype=torch.float32, device="cuda")
        C = buf.as_strided((M, N), (N, 1), 1 + (off % 3))
        assert Ad.data_ptr() % 16 != 0 and C.data_ptr() % 16 != 0
        out = gu.run(mode, Ad, Bd, out=C)
        ref, S = gu.oracle_full(A, B)
        gu.assert_close(out.cpu().numpy(), ref, S, gu.TOL[mode], f"{mode} offset {off}")


@pytest.mark.parametrize("mode", gu.ALL_MODES)
def test_deterministic(mode):
    A, B = inputs.make_random(1000, 1100, 900, seed=41, dtype=gu.in_dtype(mode))
    Ad, Bd = A.cuda(), B.cuda()
    C1 = gu.run(mode, Ad, Bd).clone()
    C2 = gu.run(mode, Ad, Bd)
    assert torch.equal(C1, C2)


@pytest.mark.parametrize("mode", gu.ALL_MODES)
def test_host_pointers_rejected(mode):
    """Host memory (pageable or pinned) is refused before any launch."""
    A, B = inputs.make_random(64, 64, 64, seed=43, dtype=gu.in_dtype(mode))
    C = torch.empty((64, 64), dtype=torch.float32, device="cuda")
    call = {"simt": lambda a, b, c: dg.gemm_f32_simt(64, 64, 64, a, 64, b, 64, c, 64, 0),
            "tf32": lambda a, b, c: dg.gemm_f32_tc(dg.TC_TF32, 64, 64, 64, a, 64, b, 64, c, 64, 0),
            "3xtf32": lambda a, b, c: dg.gemm_f32_tc(dg.TC_3XTF32, 64, 64, 64, a, 64, b, 64, c,
                                                     64, 0),
            "bf16": lambda a, b, c: dg.gemm_bf16_tc(64, 64, 64, a, 64, b, 64, c, 64, 0),
            "fp16": lambda a, b, c: dg.gemm_f16_tc(64, 64, 64, a, 64, b, 64, c, 64, 0),
            "e4m3": lambda a, b, c: dg.gemm_f8_tc(dg.F8_E4M3, 64, 64, 64, a, 64, b, 64, c, 64, 0),
            "e5m2": lambda a, b, c: dg.gemm_f8_tc(dg.F8_E5M2, 64, 64, 64, a, 64, b, 64, c, 64,
                                                  0)}[mode]
    Ad, Bd = A.cuda(), B.cuda()
    assert call(A.data_ptr(), Bd.data_ptr(), C.data_ptr()) == dg.ERR_INVALID_POINTER
    Bp = B.pin_memory()
    assert call(Ad.data_ptr(), Bp.data_ptr(), C.data_ptr()) == dg.ERR_INVALID_POINTER
    Ch = torch.empty((64, 64), dtype=torch.float32)
    assert call(Ad.data_ptr(), Bd.data_ptr(), Ch.data_ptr()) == dg.ERR_INVALID_POINTER


def test_streams_are_honoured():
    """Work is enqueued on the given stream and ordered with it."""
    A, B = inputs.make_random(512, 512, 512, seed=47)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        Ad, Bd = A.cuda(non_blocking=False), B.cuda()
        C = dg.matmul(Ad, Bd, mode="tf32", stream=s)
        C2 = dg.matmul(Ad, Bd, mode="simt", stream=s)
    s.synchronize()
    ref, S = gu.oracle_full(A, B)
    gu.assert_close(C.cpu().numpy(), ref, S, gu.TOL["tf32"], "tf32 on side stream")
    gu.assert_close(C2.cpu().numpy(), ref, S, gu.TOL["simt"], "simt on side stream")


def test_simt_tail_split_around_wave_boundaries():
    """The SIMT path splits the tiles of a partial last wave along K and sums
    the parts in a fixed order.  Tile counts at, just above and two waves
    above one full wave of the GPU's SMs (tiles of 128 x 256)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for (rows, K) in [(sms, 777), (sms + 8, 1000), (2 * sms + 3, 520), (5, 4096)]:
        M, N = 128 * rows, 256
        A, B = inputs.make_random(M, N, K, seed=rows + K, dist="normal")
        Ad, Bd = A.cuda(), B.cuda()
        C1 = gu.run("simt", Ad, Bd).clone()
        C2 = gu.run("simt", Ad, Bd)
        assert torch.equal(C1, C2), "split sums must not depend on which part finishes last"
        ref, S = gu.oracle_full(A, B)
        gu.assert_close(C2.cpu().numpy(), ref, S, gu.TOL["simt"], f"simt tail {M}x{N}x{K}")


def test_concurrent_calls_from_host_threads():
    """Four host threads, each on its own stream, call different paths at
    once (re-pitch scratch from the shared pool, cluster K-split, FP8
    transpose, SIMT tail split): every result must match the oracle."""
    import threading

    cases = [("tf32", (1000, 1013, 997)), ("bf16", (1024, 1024, 1024)),
             ("e4m3", (520, 700, 640)), ("simt", (640, 512, 777))]
    data = []
    for mode, (M, N, K) in cases:
        A, B = inputs.make_random(M, N, K, seed=M + K, dist="normal", dtype=gu.in_dtype(mode))
        data.append((mode, A, B, A.cuda(), B.cuda()))
    torch.cuda.synchronize()
    results, errors = [None] * len(data), []

    def work(i):
        try:
            mode, _, _, Ad, Bd = data[i]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(5):
                    C = dg.matmul(Ad, Bd, mode=mode, stream=s)
            s.synchronize()
            results[i] = C.cpu()
        except Exception as e:  # noqa: BLE001 -- reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(data))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    for (mode, A, B, _, _), C in zip(data, results):
        ref, S = gu.oracle_full(A, B)
        gu.assert_close(C.numpy(), ref, S, gu.TOL[mode], f"{mode} from a host thread")


def test_dependent_calls_back_to_back():
    """Calls queued without synchronisation where each reads what the one
    before wrote (read after write) or overwrites what the one before read
    (write after read), across paths and kernels.  Every kernel starts early
    under programmatic dependent launch and must wait for its predecessor
    before touching memory."""
    M = 640
    g = torch.Generator().manual_seed(71)
    X0 = torch.randn(M, M, generator=g) / 8
    W = [torch.randn(M, M, generator=g) / 8 for _ in range(3)]
    Xd, Wd = X0.cuda(), [w.cuda() for w in W]
    Y1 = dg.matmul(Xd, Wd[0], mode="3xtf32")                 # Y1 = X0 W0
    Y2 = dg.matmul(Y1, Wd[1], mode="simt")                   # reads Y1 (RAW)
    dg.matmul(Y2, Wd[2], mode="3xtf32", out=Xd)              # overwrites X0 (WAR with call 1)
    Y4 = dg.matmul(Xd, Y1, mode="simt")                      # reads both again
    torch.cuda.synchronize()
    x0, w0, w1, w2 = (t.double().numpy() for t in (X0, W[0], W[1], W[2]))
    y1 = x0 @ w0
    y2 = y1 @ w1
    x3 = y2 @ w2
    y4 = x3 @ y1
    for got, want, what in [(Y1, y1, "Y1"), (Y2, y2, "Y2"), (Xd, x3, "X overwritten"), (Y4, y4, "Y4")]:
        err = np.abs(got.cpu().double().numpy() - want).max() / np.abs(want).max()
        assert err < 1e-5, f"{what}: relative error {err:.2e}"
