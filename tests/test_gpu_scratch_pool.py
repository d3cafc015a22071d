"""The library's scratch pool gives memory back: after a call that needed far
more scratch than the pool's 32 MiB release threshold (the lo parts of a
3xTF32 product on the CTA-pair kernel, 128 MiB here) and a synchronisation,
device memory is back within that bound of where it was before the call.
"""
import pytest
import torch

import gpu_util as gu
from dense_gemm_f32_gb300 import inputs

pytestmark = pytest.mark.gpu

KEEP = 32 << 20          # the pool's release threshold
SLACK = 4 << 20          # allocation granularity of the driver


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    gu.check_watchdog()


def test_pool_returns_scratch_after_a_sync():
    # load the kernels of the path first (a small problem on the same path,
    # whose lo parts are under 1 MiB), so that only scratch can move the
    # free-memory figure below
    As, Bs = inputs.make_random(1792, 1536, 64, seed=1)
    gu.run("3xtf32", As.cuda(), Bs.cuda())
    M = N = K = 4096
    A, B = inputs.make_random(M, N, K, seed=2)
    Ad, Bd = A.cuda(), B.cuda()
    C = torch.empty((M, N), device="cuda")
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(2):
        gu.run("3xtf32", Ad, Bd, out=C)   # 2 x 64 MiB of lo parts each call
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    held = free_before - free_after
    assert held <= KEEP + SLACK, f"the pool still holds {held / 2**20:.1f} MiB after a sync"
    rows = torch.arange(0, M, 509).numpy()
    ref, S = gu.oracle_rows(A, B, rows)
    gu.assert_close(C.cpu().numpy()[rows], ref, S, gu.TOL["3xtf32"], "3xtf32 4096^3")
