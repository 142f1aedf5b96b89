// Exhaustive check that the quantizers' division (one Markstein correction
// from a per-block negated reciprocal, two lanes per instruction, codes taken
// from the negated quotients) gives the same e4m3 code as IEEE division on
// every input the blockwise quantizers can meet: s = fl32(max(amax, 1e-12) /
// 448) for every non-negative finite bf16 amax, and every finite bf16 x with
// |x| <= amax.  Prints "checked <pairs> code_mismatches <n> quotient_mismatches <m>".
#include <cstdint>
#include <cstdio>

#include "common.cuh"
#include "quant_math.cuh"

using namespace fp8bw;

__global__ void check(unsigned long long* out) {
  const uint32_t ab = blockIdx.x;  // bf16 bits of amax: 0x0000 .. 0x7F7F
  const float amax = __uint_as_float(ab << 16);
  const float s = blockwise_scale(amax);
  const float ny = neg_recip(s);
  unsigned long long n = 0, bad_code = 0, bad_q = 0;
  for (uint32_t xb = threadIdx.x; xb < 65536u; xb += blockDim.x) {
    const float x = __uint_as_float(xb << 16);
    if (!(fabsf(x) <= amax)) continue;  // NaN, infinities and |x| > amax never occur
    const float2 nq = neg_div_by_scale2(make_float2(x, -x), make_float2(s, s), make_float2(ny, ny));
    const float q_fast = -nq.x;
    const float q_ieee = __fdiv_rn(x, s);
    const uint32_t codes = e4m3x4_from_neg(nq, nq);
    // both lanes of the pair and both halves of the packing must agree
    const uint32_t c_fast = (codes & 0xFFu) | ((codes >> 16) & 0xFFu) << 8 | ((codes >> 8) & 0xFFu) << 16;
    const uint32_t c_neg = cvt_e4m3x2(-q_ieee, 0.0f) & 0xFFu;
    const uint32_t c_ieee = cvt_e4m3x2(q_ieee, 0.0f) & 0xFFu;
    ++n;
    bad_code += (c_fast != (c_ieee | c_ieee << 8 | c_neg << 16));
    bad_q += (__float_as_uint(q_fast) != __float_as_uint(q_ieee));
  }
  atomicAdd(&out[0], n);
  atomicAdd(&out[1], bad_code);
  atomicAdd(&out[2], bad_q);
}

int main() {
  unsigned long long* d = nullptr;
  if (cudaMalloc(&d, 3 * sizeof(unsigned long long)) != cudaSuccess) return 2;
  cudaMemset(d, 0, 3 * sizeof(unsigned long long));
  check<<<0x7F80, 256>>>(d);
  unsigned long long h[3] = {0, 0, 0};
  cudaError_t e = cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost);
  cudaFree(d);
  if (e != cudaSuccess) {
    printf("cuda error %s\n", cudaGetErrorString(e));
    return 3;
  }
  printf("checked %llu code_mismatches %llu quotient_mismatches %llu\n", h[0], h[1], h[2]);
  return h[1] == 0 ? 0 : 1;
}
