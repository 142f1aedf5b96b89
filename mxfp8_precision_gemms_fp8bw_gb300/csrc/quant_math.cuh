// Scalar arithmetic of the blockwise quantizers, shared by quant.cu and the
// exhaustive division check in tests/cuda/.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace fp8bw {

// Blockwise rule: s = fl32(max(amax, 1e-12) / 448), IEEE division (the EPS
// floor of PR #4295's scale helpers; 448 = largest finite e4m3).
__device__ __forceinline__ float blockwise_scale(float amax) {
  return __fdiv_rn(fmaxf(amax, 1e-12f), 448.0f);
}

// The reciprocal the element divisions work from: ny = RN(1 / -s) = -RN(1 / s).
__device__ __forceinline__ float neg_recip(float s) { return -__frcp_rn(s); }

// fl32(x / -s) = -fl32(x / s) for two values at once (f32x2 FMUL2 / FFMA2),
// from s > 0 and ny = neg_recip(s): one correction step of Markstein's
// division by b = -s -- q = RN(x * ny), r = RN(x - q * b) = RN(x + q * s)
// (exact through the FMA), RN(q + r * ny).  With ny the correctly rounded
// reciprocal of b and q within an ulp of x / b, the corrected quotient is the
// correctly rounded x / b.  Dividing by -s rather than s keeps signed zeros
// right with no select: x = +0 gives -0 and x = -0 gives +0 (the correction
// step adds a zero of q's sign to a zero of the other sign, which rounds to
// +0, and only the negated divisor makes +0 the wanted result).  The
// identity with IEEE division on every pair the quantizers can meet (s from a
// bf16 amax, x a bf16 value with |x| <= amax) is checked exhaustively by
// tests/cuda/division_exhaustive.cu.
__device__ __forceinline__ float2 neg_div_by_scale2(float2 x, float2 s, float2 ny) {
  const float2 q = __fmul2_rn(x, ny);
  const float2 r = __ffma2_rn(q, s, x);
  return __ffma2_rn(r, ny, q);
}

// e4m3 codes of four quotients handed over negated (lo.x, lo.y, hi.x, hi.y in
// byte order): e4m3 rounding and saturation are symmetric in the sign, so the
// code of v is the code of -v with its sign bit flipped.
__device__ __forceinline__ uint32_t e4m3x4_from_neg(float2 lo, float2 hi) {
  return __byte_perm(cvt_e4m3x2(lo.x, lo.y), cvt_e4m3x2(hi.x, hi.y), 0x5410) ^ 0x80808080u;
}

}  // namespace fp8bw
