// Scalar arithmetic of the blockwise quantizers, shared by quant.cu and the
// exhaustive division check in tests/cuda/.
#pragma once

#include <cuda_runtime.h>

namespace fp8bw {

// Blockwise rule: s = fl32(max(amax, 1e-12) / 448), IEEE division (the EPS
// floor of PR #4295's scale helpers; 448 = largest finite e4m3).
__device__ __forceinline__ float blockwise_scale(float amax) {
  return __fdiv_rn(fmaxf(amax, 1e-12f), 448.0f);
}

// fl32(x / s) from y = RN(1/s), computed once per block: one correction step
// of Markstein's division -- q = RN(x * y), r = x - q * s (exact through the
// FMA), RN(q + r * y).  With y the correctly rounded reciprocal and q within
// an ulp of x / s, the corrected quotient is the correctly rounded one.  A
// zero quotient keeps its own sign (the correction would turn -0 into +0).
// Identity with IEEE division on every pair the quantizers can meet (s from
// a bf16 amax, x a bf16 value with |x| <= amax) is checked exhaustively at
// the e4m3 level by tests/cuda/division_exhaustive.cu.
__device__ __forceinline__ float div_by_scale(float x, float s, float y) {
  const float q = x * y;
  const float r = fmaf(-q, s, x);
  const float q1 = fmaf(r, y, q);
  return q == 0.0f ? q : q1;
}

}  // namespace fp8bw
