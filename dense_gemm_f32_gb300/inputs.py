"""Seeded synthetic inputs for the GEMM workloads.

This module only draws random numbers and lays them out; it holds none of
the product's arithmetic, and both the CUDA path's tests and the CPU
oracle's checks take their inputs from it.  Everything is generated on the
CPU with torch's CPU generator, so a given (shape, seed) gives the same
values on every machine; callers copy the tensors to the device themselves.

Recipe (the pages fix no distribution or generator, so these are chosen):
  * one torch.Generator('cpu') per workload, seeded with the workload's seed;
    A is drawn first, then B;
  * uniform[-1, 1)      -> 2 * torch.rand(shape) - 1
  * normal N(0, s^2)    -> s * torch.randn(shape)
  * integer copy        -> torch.randint(-4, 5, shape) from a fresh generator
                           with the same seed, stored as float32
  * bf16 / fp16 / fp8   -> the fp32 draws rounded once to bfloat16, float16,
                           float8 e4m3 or e5m2 (round to nearest even, no
                           scaling); the rounded values ARE the inputs.
Shapes follow the pages' workloads: the 1024 x 1024 benchmark of
"4. 矩阵乘法（GEMM）优化" section 4.4, the M = 1000 ragged edge of Lesson 8
section 二十六, the K = 64 = 4 x 16 tile example of Lesson 8 section 九.
"""
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    seed: int
    dist: str          # "uniform" | "normal"
    a_std: float = 1.0  # for "normal"
    b_std: float = 1.0
    bf16: bool = False  # inputs rounded to bfloat16
    fp16: bool = False  # inputs rounded to float16
    fp8: str = ""       # "e4m3" / "e5m2": inputs rounded to that 8-bit float

    @property
    def flops(self):
        return 2 * self.M * self.N * self.K


# The five workloads of the benchmark configuration, by what they are.
SQUARE_64 = Workload("square-64 fp32", 64, 64, 64, 0, "uniform")
SQUARE_1024 = Workload("square-1024 fp32", 1024, 1024, 1024, 1, "uniform")
RAGGED_1000 = Workload("ragged 1000x1013x997 fp32", 1000, 1013, 997, 2, "normal")
SQUARE_8192 = Workload("square-8192 fp32", 8192, 8192, 8192, 3, "uniform")
TRANSFORMER_BF16 = Workload("transformer-layer 16384x14336x4096 bf16", 16384, 14336, 4096, 4,
                            "normal", a_std=1.0, b_std=0.02, bf16=True)
TRANSFORMER_F32 = Workload("transformer-layer 16384x14336x4096 fp32", 16384, 14336, 4096, 4,
                           "normal", a_std=1.0, b_std=0.02, bf16=False)
TRANSFORMER_F16 = Workload("transformer-layer 16384x14336x4096 fp16", 16384, 14336, 4096, 4,
                           "normal", a_std=1.0, b_std=0.02, fp16=True)
TRANSFORMER_E4M3 = Workload("transformer-layer 16384x14336x4096 e4m3", 16384, 14336, 4096, 4,
                            "normal", a_std=1.0, b_std=0.02, fp8="e4m3")
TRANSFORMER_E5M2 = Workload("transformer-layer 16384x14336x4096 e5m2", 16384, 14336, 4096, 4,
                            "normal", a_std=1.0, b_std=0.02, fp8="e5m2")

ALL = [SQUARE_64, SQUARE_1024, RAGGED_1000, SQUARE_8192, TRANSFORMER_BF16, TRANSFORMER_F32,
       TRANSFORMER_F16, TRANSFORMER_E4M3, TRANSFORMER_E5M2]

F8_DTYPES = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


def _draw(gen, shape, dist, std):
    if dist == "uniform":
        return 2.0 * torch.rand(shape, generator=gen, dtype=torch.float32) - 1.0
    if dist == "normal":
        return std * torch.randn(shape, generator=gen, dtype=torch.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def make(w: Workload):
    """(A, B) as CPU tensors: float32, or bfloat16 / float16 / float8 per w."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    A = _draw(g, (w.M, w.K), w.dist, w.a_std)
    B = _draw(g, (w.K, w.N), w.dist, w.b_std)
    if w.bf16:
        A, B = A.to(torch.bfloat16), B.to(torch.bfloat16)
    elif w.fp16:
        A, B = A.to(torch.float16), B.to(torch.float16)
    elif w.fp8:
        A, B = A.to(F8_DTYPES[w.fp8]), B.to(F8_DTYPES[w.fp8])
    return A, B


def make_integer(M, N, K, seed, lo=-4, hi=4):
    """Integer-valued float32 (A, B), entries uniform in {lo..hi}."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    A = torch.randint(lo, hi + 1, (M, K), generator=g).to(torch.float32)
    B = torch.randint(lo, hi + 1, (K, N), generator=g).to(torch.float32)
    return A, B


def make_random(M, N, K, seed, dist="uniform", dtype=torch.float32):
    """Generic seeded (A, B) for sweeps over shapes."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    A = _draw(g, (M, K), dist, 1.0)
    B = _draw(g, (K, N), dist, 1.0)
    if dtype in (torch.bfloat16, torch.float16, torch.float8_e4m3fn, torch.float8_e5m2):
        A, B = A.to(dtype), B.to(dtype)
    return A, B


def embed(X, ld, offset=0, fill=float("nan")):
    """Place matrix X (rows x cols) in a fresh 1-D buffer with leading dimension
    `ld` >= cols, starting `offset` elements in; the rest is `fill`.
    Returns (buffer, view) where view is the strided 2-D window onto X."""
    rows, cols = X.shape
    if ld < cols:
        raise ValueError("ld must be >= the number of columns")
    n = offset + (rows - 1) * ld + cols if rows and cols else offset + 1
    buf = torch.full((max(n, 1),), fill, dtype=X.dtype)
    if rows and cols:
        view = buf.as_strided((rows, cols), (ld, 1), offset)
        view.copy_(X)
    else:
        view = buf.as_strided((rows, cols), (max(ld, 1), 1), offset)
    return buf, view
