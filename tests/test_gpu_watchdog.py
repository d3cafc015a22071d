"""Failure detection on the GPU without a fault: a bounded wait that runs out.

Every wait of the tensor-core kernels on a shared-memory barrier gives up
after about 2 s; the kernel then records a site code in the device watchdog
word, lets its copies land, frees its tensor memory and returns, and
dgemm_watchdog_status reports DGEMM_ERR_WATCHDOG.  DGEMM_TC_TEST_STALL=1 makes
the MMA thread of the first CTA (or CTA pair) wait on a barrier that nothing
arrives at, so these tests run that path for real: the call must come back
within seconds, the status must name a site of the kernel, and the next call
on the same context must be correct.  DGEMM_SIMT_TEST_STALL=1 does the same
for the SIMT path's TMA ring kernel (warp 0 of its first CTA), whose stages
then stop being refilled, so every other warp's wait runs out too.
"""
import os
import re
import time

import pytest
import torch

import gpu_util as gu
from dense_gemm_f32_gb300 import inputs
import dense_gemm_f32_gb300 as dg

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _site_codes(*files):
    codes = set()
    for f in files or ("tc.cu",):
        src = open(os.path.join(ROOT, "dense_gemm_f32_gb300", "csrc", f), encoding="utf-8").read()
        codes |= {int(c, 16) for c in re.findall(r"kSite\w+ = (0x[0-9a-f]+)", src)}
    return codes


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    gu.check_watchdog()


@pytest.mark.parametrize("pair", ["0", "1"])
@pytest.mark.parametrize("mode", ["tf32", "3xtf32"])
def test_wait_runs_out_and_the_context_survives(mode, pair, monkeypatch):
    monkeypatch.setenv("DGEMM_TC_PAIR", pair)
    A, B = inputs.make_random(1024, 1024, 1024, seed=61, dist="normal")
    Ad, Bd = A.cuda(), B.cuda()
    stream = torch.cuda.current_stream().cuda_stream
    assert dg.dgemm_watchdog_status(stream)[0] == dg.OK

    monkeypatch.setenv("DGEMM_TC_TEST_STALL", "1")
    t0 = time.time()
    gu.run(mode, Ad, Bd)  # synchronises
    elapsed = time.time() - t0
    st, where = dg.dgemm_watchdog_status(stream)
    assert st == dg.ERR_WATCHDOG, dg.dgemm_status_string(st)
    assert where in _site_codes(), hex(where)
    assert elapsed < 30, f"the abort path took {elapsed:.1f} s"
    assert dg.dgemm_watchdog_status(stream)[0] == dg.OK  # reading clears the word

    monkeypatch.delenv("DGEMM_TC_TEST_STALL")
    C = gu.run(mode, Ad, Bd)
    ref, S = gu.oracle_full(A, B)
    gu.assert_close(C.cpu().numpy(), ref, S, gu.TOL[mode], f"{mode} pair={pair} after the abort")
    assert dg.dgemm_watchdog_status(stream)[0] == dg.OK


@pytest.mark.parametrize("ring", ["1", "2"])
@pytest.mark.parametrize("M, N, K", [(1024, 1024, 1024), (4096, 4096, 256)])
def test_simt_ring_wait_runs_out_and_the_context_survives(M, N, K, ring, monkeypatch):
    """1024^3: every tile split over a cluster; 4096 x 4096 x 256: whole tiles
    plus a tail split through scratch."""
    monkeypatch.setenv("DGEMM_SIMT_RING", ring)
    monkeypatch.setenv("DGEMM_SIMT_SMALL", "0")
    A, B = inputs.make_random(M, N, K, seed=62, dist="normal")
    Ad, Bd = A.cuda(), B.cuda()
    stream = torch.cuda.current_stream().cuda_stream
    assert dg.dgemm_watchdog_status(stream)[0] == dg.OK

    monkeypatch.setenv("DGEMM_SIMT_TEST_STALL", "1")
    t0 = time.time()
    gu.run("simt", Ad, Bd)  # synchronises
    elapsed = time.time() - t0
    st, where = dg.dgemm_watchdog_status(stream)
    assert st == dg.ERR_WATCHDOG, dg.dgemm_status_string(st)
    assert where in _site_codes("simt.cu"), hex(where)
    assert elapsed < 30, f"the abort path took {elapsed:.1f} s"
    assert dg.dgemm_watchdog_status(stream)[0] == dg.OK

    monkeypatch.delenv("DGEMM_SIMT_TEST_STALL")
    C = gu.run("simt", Ad, Bd)
    rows = torch.arange(0, M, 97).numpy()
    ref, S = gu.oracle_rows(A, B, rows)
    gu.assert_close(C.cpu().numpy()[rows], ref, S, gu.TOL["simt"], f"simt ring={ring} after the abort")
    assert dg.dgemm_watchdog_status(stream)[0] == dg.OK
