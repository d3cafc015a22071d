"""Build libdgemm.so (the C-ABI library) in-tree with nvcc for sm_103a.

The translation units compile in parallel; the link keeps only the symbols
declared in include/dgemm.h visible.  ptxas resource usage (-Xptxas -v:
registers, spills, shared memory per kernel) is written to
_build/ptxas_<unit>.log next to the objects.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libdgemm.so")
HEADER = os.path.join(ROOT, "include", "dgemm.h")
# (source, object name, defines): simt.cu and tc.cu are compiled once per
# operand layout so that the four layouts build in parallel.
UNITS = ([("api.cu", "api", []), ("staging.cu", "staging", [])]
         + [("simt.cu", f"simt_{u}", [f"-DDGEMM_SIMT_UNIT={u}"]) for u in range(4)]
         + [("tc.cu", f"tc_{u}", [f"-DDGEMM_TC_UNIT={u}"]) for u in range(4)])
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
EXPORTS = ["gemm_f32_simt", "gemm_f32_tc", "gemm_bf16_tc", "dgemm_status_string",
           "dgemm_last_cuda_error", "dgemm_watchdog_status", "dgemm_version",
           "dgemm_kernel_launches", "gemm_f32_tc_noalloc", "gemm_f16_tc", "dgemm_gemm_ex",
           "gemm_f8_tc"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdgemm.so")


def _sources():
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [HEADER, __file__]
    return [d for d in deps if os.path.isfile(d)]


def _stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(s) > t for s in _sources())


def _compile(nvcc, unit):
    source, name, defines = unit
    src = os.path.join(CSRC, source)
    obj = os.path.join(BUILD, name + ".o")
    cmd = [nvcc, *ARCH, "-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC",
           "-Xptxas", "-v", *defines, "-I", os.path.join(ROOT, "include"), "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    with open(os.path.join(BUILD, f"ptxas_{name}.log"), "w") as f:
        f.write(r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {name}:\n{r.stderr[-6000:]}")
    return obj


def build(force=False, verbose=False):
    """Compile (if stale) and return the path of libdgemm.so."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    with cf.ThreadPoolExecutor(max_workers=min(len(UNITS), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda u: _compile(nvcc, u), UNITS))
    vs = os.path.join(BUILD, "exports.map")
    with open(vs, "w") as f:
        f.write("{\n  global:\n" + "".join(f"    {s};\n" for s in EXPORTS) + "  local: *;\n};\n")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-Xlinker", f"--version-script={vs}", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr[-6000:]}")
    os.replace(tmp, LIB)
    if verbose:
        for _, name, _ in UNITS:
            with open(os.path.join(BUILD, f"ptxas_{name}.log")) as f:
                sys.stdout.write(f.read())
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
