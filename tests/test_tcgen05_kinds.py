"""Which tcgen05.mma operand kinds the sm_103a toolchain accepts.

The tensor-core formats listed in "第八课：GPU 如何完成矩阵乘法" section 二十二 include
INT8.  On sm_103a this library offers TF32, BF16, FP16 and FP8 but no INT8
path, because the PTX assembler refuses tcgen05.mma's integer kind
(.kind::i8) for that target while it accepts it for sm_100a; the PTX ISA's
target notes for tcgen05.mma restrict .kind::i8 to other targets.  These
tests pin that fact with the installed nvcc, so that the gap is re-examined
if a toolchain ever accepts it.  CPU only: nothing runs on a GPU.
"""
import os
import shutil
import subprocess

import pytest

NVCC = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"

SRC = r"""
#include <cstdint>
__global__ void k(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, int acc) {
  asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
               "tcgen05.mma.cta_group::1.kind::KIND [%0], %1, %2, %3, p;\n}"
               :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
"""


def _compile(tmp_path, kind, arch):
    if not os.path.exists(NVCC):
        pytest.skip("nvcc not available")
    src = tmp_path / f"k_{kind}_{arch}.cu"
    src.write_text(SRC.replace("KIND", kind))
    r = subprocess.run([NVCC, "-gencode", f"arch=compute_{arch},code=sm_{arch}", "-c", str(src),
                        "-o", str(tmp_path / f"k_{kind}_{arch}.o")], capture_output=True, text=True)
    return r.returncode, r.stdout + r.stderr


@pytest.mark.parametrize("kind", ["tf32", "f16", "f8f6f4"])
def test_float_kinds_assemble_for_sm103a(tmp_path, kind):
    rc, out = _compile(tmp_path, kind, "103a")
    assert rc == 0, out


def test_integer_kind_is_refused_for_sm103a(tmp_path):
    rc, out = _compile(tmp_path, "i8", "103a")
    assert rc != 0 and "kind::i8" in out and "sm_103a" in out, out


def test_integer_kind_assembles_for_sm100a(tmp_path):
    """The same instruction is well formed: the refusal is about the target."""
    rc, out = _compile(tmp_path, "i8", "100a")
    assert rc == 0, out
