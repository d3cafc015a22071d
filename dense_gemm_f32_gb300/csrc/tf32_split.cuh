// tf32_split.cuh -- the 3xTF32 operand split, shared by the GEMM kernels'
// in-kernel split and the split pre-pass.
#pragma once

#include <cstdint>

namespace dg {

// 3xTF32 split of x = hi + lo.  The tensor core reads an fp32 operand at TF32
// precision by dropping its low 13 mantissa bits (truncation; pinned by a GPU
// test), so the raw fp32 tile itself serves as hi = trunc_tf32(x) and only lo
// is written: lo = x - hi, exact in fp32, rounded to TF32 (nearest, ties
// away).  The dropped lo*lo term and the rounding of lo are each below
// 2^-20 |x y| per product.  Infinities and NaNs have no low part (x - x
// would be NaN and turn an infinite result into NaN): their lo is 0 and the
// raw value carries them, as in the plain TF32 product.
__device__ __forceinline__ uint32_t split_lo_tf32(uint32_t xbits) {
  const float r = __uint_as_float(xbits) - __uint_as_float(xbits & 0xFFFFE000u);
  uint32_t l;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(l) : "f"(r));
  return (xbits & 0x7F800000u) == 0x7F800000u ? 0u : l;
}

// The split's fast path: the same lo without the infinity / NaN test, and
// `seen` becomes NaN if any x was infinite or NaN (x - x is NaN then), one
// max.NaN per element; the caller redoes its elements with split_lo_tf32
// in that (rare) case.
__device__ __forceinline__ uint32_t split_lo_tf32_fast(uint32_t xbits, float &seen) {
  const float r = __uint_as_float(xbits) - __uint_as_float(xbits & 0xFFFFE000u);
  asm("max.NaN.f32 %0, %0, %1;" : "+f"(seen) : "f"(r));
  uint32_t l;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(l) : "f"(r));
  return l;
}

}  // namespace dg
