"""A plain C program as a client of the library (tests/c/gemm_from_c.c): it
includes only include/dgemm.h and the CUDA runtime's C header, links
libdgemm.so and libcudart, and calls every entry point.  Without a GPU the
test builds and links it; on a GB300 it runs it, and every path must
reproduce the host product of integer-valued inputs exactly."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _build(tmp_path):
    from dense_gemm_f32_gb300 import build

    lib = build.build()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(lib)
    cudalib = os.path.join(CUDA, "lib64")
    exe = str(tmp_path / "gemm_from_c")
    cmd = [cc, "-std=c99", "-O1", "-Wall", "-Werror", os.path.join(ROOT, "tests", "c", "gemm_from_c.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-L", libdir, "-ldgemm", "-L", cudalib, "-lcudart",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{cudalib}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    return exe


def test_c_client_builds_and_links(tmp_path):
    assert os.path.exists(_build(tmp_path))


@pytest.mark.gpu
def test_c_client_runs_every_path_exactly(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-2000:]
