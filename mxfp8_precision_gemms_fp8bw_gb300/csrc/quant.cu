// e4m3 quantizers of libfp8bw: 1x128 rowwise / colwise and 128x128 blockwise
// (fp32 scales), and MXFP8 1x32 rowwise / colwise / 3D-colwise (E8M0 scales).
//
// All of them are HBM-bound streaming kernels: each element is read once
// (2 B of bf16) and written once (1 B of e4m3), plus one scale per block.
// Loads are 16-byte vectors; block maxima are reduced with warp shuffles; the
// colwise kernels transpose in registers (each thread owns an 8x8 micro-tile
// and packs e4m3 pairs along the column) so every store is a coalesced
// 8-byte vector.
#include "common.cuh"
#include "launch.h"
#include "quant_math.cuh"

namespace fp8bw {

// ---------------------------------------------------------------- scale rules

// MXFP8 rule: unbiased E8M0 exponent of a block from its amax.
//   RCEIL: smallest E with 448 * 2^E >= amax.  With amax = 1.m * 2^e and
//          448 = 1.75 * 2^8 this is e - 8, plus one when 1.m > 1.75.
//   FLOOR: floor(log2 amax) - 8 = e - 8.
// Clamped to [-127, 127]; zero and subnormal amax give -127.
__device__ __forceinline__ int mx_exponent(float amax, int mode) {
  const uint32_t b = __float_as_uint(amax);
  const int ef = static_cast<int>((b >> 23) & 0xFF);
  if (ef == 0) return -127;
  int E = ef - 127 - 8;
  if (mode == 0 && (b & 0x7FFFFFu) > 0x600000u) E += 1;
  return max(-127, min(127, E));
}

// 2^-E as a float for E in [-127, 127] (exact; 2^-127 is subnormal).
__device__ __forceinline__ float pow2_neg(int E) {
  const int be = 127 - E;  // biased exponent of 2^-E
  return be > 0 ? __uint_as_float(static_cast<uint32_t>(be) << 23) : __uint_as_float(0x00400000u);
}

__device__ __forceinline__ float amax8(const uint4& v) {
  float a = fabsf(bf16lo_to_f32(v.x));
  a = fmaxf(a, fabsf(bf16hi_to_f32(v.x)));
  a = fmaxf(a, fabsf(bf16lo_to_f32(v.y)));
  a = fmaxf(a, fabsf(bf16hi_to_f32(v.y)));
  a = fmaxf(a, fabsf(bf16lo_to_f32(v.z)));
  a = fmaxf(a, fabsf(bf16hi_to_f32(v.z)));
  a = fmaxf(a, fabsf(bf16lo_to_f32(v.w)));
  a = fmaxf(a, fabsf(bf16hi_to_f32(v.w)));
  return a;
}

// Element j (0..7) of 8 packed bf16.
__device__ __forceinline__ float elem8(const uint4& v, int j) {
  const uint32_t w = j < 2 ? v.x : j < 4 ? v.y : j < 6 ? v.z : v.w;
  return (j & 1) ? bf16hi_to_f32(w) : bf16lo_to_f32(w);
}

// Eight e4m3 codes of fl32(x/s) packed little-endian; y = RN(1/s).
__device__ __forceinline__ uint2 quant8_div(const uint4& v, float s, float y) {
  uint2 o;
  o.x = cvt_e4m3x2(div_by_scale(bf16lo_to_f32(v.x), s, y), div_by_scale(bf16hi_to_f32(v.x), s, y)) |
        (cvt_e4m3x2(div_by_scale(bf16lo_to_f32(v.y), s, y), div_by_scale(bf16hi_to_f32(v.y), s, y)) << 16);
  o.y = cvt_e4m3x2(div_by_scale(bf16lo_to_f32(v.z), s, y), div_by_scale(bf16hi_to_f32(v.z), s, y)) |
        (cvt_e4m3x2(div_by_scale(bf16lo_to_f32(v.w), s, y), div_by_scale(bf16hi_to_f32(v.w), s, y)) << 16);
  return o;
}

// Eight e4m3 codes of x * m (MX: m = 2^-E, an exact power of two).
__device__ __forceinline__ uint2 quant8_mul(const uint4& v, float m) {
  uint2 o;
  o.x = cvt_e4m3x2(bf16lo_to_f32(v.x) * m, bf16hi_to_f32(v.x) * m) |
        (cvt_e4m3x2(bf16lo_to_f32(v.y) * m, bf16hi_to_f32(v.y) * m) << 16);
  o.y = cvt_e4m3x2(bf16lo_to_f32(v.z) * m, bf16hi_to_f32(v.z) * m) |
        (cvt_e4m3x2(bf16lo_to_f32(v.w) * m, bf16hi_to_f32(v.w) * m) << 16);
  return o;
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void st_v2(void* p, uint2 v) {
  asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// ---------------------------------------------------------------- 1x128 rowwise

// CTA = 128 rows x one 128-column block.  Warp w owns rows [16w, 16w + 16);
// per step each half-warp takes one row and lane (l & 15) columns
// [8(l & 15), 8(l & 15) + 8).  All eight 16-byte loads are issued first.
__global__ void __launch_bounds__(256) quant_1x128_row_kernel(const uint16_t* __restrict__ x, int64_t R, int64_t C,
                                                              uint8_t* __restrict__ q, float* __restrict__ s) {
  __shared__ float s_tile[128];
  const int kb = blockIdx.x;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = lane >> 4, l16 = lane & 15;
  const int64_t col = static_cast<int64_t>(kb) * 128 + l16 * 8;

  uint4 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t r = r0 + warp * 16 + i * 2 + half;
    v[i] = ld_nc_v4(x + r * C + col);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float a = amax8(v[i]);
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 8));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    const float sc = blockwise_scale(a);
    const int rl = warp * 16 + i * 2 + half;
    st_v2(q + (r0 + rl) * C + col, quant8_div(v[i], sc, __frcp_rn(sc)));
    if (l16 == 0) s_tile[rl] = sc;
  }
  __syncthreads();
  if (threadIdx.x < 128) s[static_cast<int64_t>(kb) * R + r0 + threadIdx.x] = s_tile[threadIdx.x];
}

// ---------------------------------------------------------------- colwise (blockwise and MX)

// CTA = 128 rows x 128 columns.  Thread (warp w, lane l) owns the 8x8
// micro-tile at rows 8*(l & 15) + [0, 8) and columns 8*(2w + (l >> 4)) + [0, 8).
// A column block spans the 16 lanes of a half-warp (blockwise, 128 rows) or 4
// of them (MX, 32 rows); its max is reduced with shuffles inside that group.
// Column j of the micro-tile is quantized into 8 bytes (e4m3 pairs of
// consecutive rows) and stored at qT[col][row0 .. row0 + 8), so the 16 lanes
// of a half-warp write 128 contiguous bytes of one qT row.
template <bool kMX>
__device__ __forceinline__ void colwise_tile(const uint16_t* __restrict__ x, int64_t R, int64_t C, int64_t r0,
                                             int64_t c0, uint8_t* __restrict__ qT, float* __restrict__ s,
                                             uint8_t* __restrict__ e8, int mode) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rg = lane & 15;
  const int64_t row = r0 + rg * 8;
  const int64_t col = c0 + (warp * 2 + (lane >> 4)) * 8;
  const bool row_ok = row < R;  // R % 32 == 0, so a 32-row MX block is all in or all out
  const bool col_ok = col < C;  // C % 8 == 0

  uint4 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[i] = (row_ok && col_ok) ? ld_nc_v4(x + (row + i) * C + col) : make_uint4(0, 0, 0, 0);
  }

  float amax[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(elem8(v[i], j)));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    if (!kMX) {
      a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
      a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 8));
    }
    amax[j] = a;
  }
  if (!(row_ok && col_ok)) return;

#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float qv[8];
    if (kMX) {
      const int E = mx_exponent(amax[j], mode);
      const float m = pow2_neg(E);
#pragma unroll
      for (int i = 0; i < 8; ++i) qv[i] = elem8(v[i], j) * m;
      if ((rg & 3) == 0) e8[(col + j) * (R / 32) + row / 32] = static_cast<uint8_t>(E + 127);
    } else {
      const float sc = blockwise_scale(amax[j]);
      const float y = __frcp_rn(sc);
#pragma unroll
      for (int i = 0; i < 8; ++i) qv[i] = div_by_scale(elem8(v[i], j), sc, y);
      if (rg == j) s[(r0 / 128) * C + col + j] = sc;
    }
    uint2 o;
    o.x = cvt_e4m3x2(qv[0], qv[1]) | (cvt_e4m3x2(qv[2], qv[3]) << 16);
    o.y = cvt_e4m3x2(qv[4], qv[5]) | (cvt_e4m3x2(qv[6], qv[7]) << 16);
    st_v2(qT + (col + j) * R + row, o);
  }
}

__global__ void __launch_bounds__(256) quant_1x128_col_kernel(const uint16_t* __restrict__ x, int64_t R, int64_t C,
                                                              uint8_t* __restrict__ qT, float* __restrict__ s) {
  colwise_tile<false>(x, R, C, static_cast<int64_t>(blockIdx.y) * 128, static_cast<int64_t>(blockIdx.x) * 128, qT, s,
                      nullptr, 0);
}

// grid.z = expert index for the 3D case (per-expert strides passed in).
__global__ void __launch_bounds__(256) mx_quant_col_kernel(const uint16_t* __restrict__ x, int64_t R, int64_t C,
                                                           uint8_t* __restrict__ qT, uint8_t* __restrict__ e8,
                                                           int mode) {
  const int64_t g = blockIdx.z;
  colwise_tile<true>(x + g * R * C, R, C, static_cast<int64_t>(blockIdx.y) * 128,
                     static_cast<int64_t>(blockIdx.x) * 128, qT + g * R * C, nullptr, e8 + g * C * (R / 32), mode);
}

// ---------------------------------------------------------------- 128x128

// Same micro-tile mapping as the colwise kernels; one scale for the whole
// CTA tile.  Writes q row-major and, when requested, qT.
__global__ void __launch_bounds__(256) quant_128x128_kernel(const uint16_t* __restrict__ x, int64_t R, int64_t C,
                                                            uint8_t* __restrict__ q, uint8_t* __restrict__ qT,
                                                            float* __restrict__ s, int64_t s_ld) {
  __shared__ float warp_max[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 128, c0 = static_cast<int64_t>(blockIdx.x) * 128;
  const int64_t row = r0 + (lane & 15) * 8;
  const int64_t col = c0 + (warp * 2 + (lane >> 4)) * 8;

  uint4 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = ld_nc_v4(x + (row + i) * C + col);
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) a = fmaxf(a, amax8(v[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  if (lane == 0) warp_max[warp] = a;
  __syncthreads();
  a = warp_max[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) a = fmaxf(a, warp_max[w]);
  const float sc = blockwise_scale(a);
  const float y = __frcp_rn(sc);
  if (threadIdx.x == 0) s[blockIdx.y * s_ld + blockIdx.x] = sc;

#pragma unroll
  for (int i = 0; i < 8; ++i) st_v2(q + (row + i) * C + col, quant8_div(v[i], sc, y));
  if (qT != nullptr) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float qv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) qv[i] = div_by_scale(elem8(v[i], j), sc, y);
      uint2 o;
      o.x = cvt_e4m3x2(qv[0], qv[1]) | (cvt_e4m3x2(qv[2], qv[3]) << 16);
      o.y = cvt_e4m3x2(qv[4], qv[5]) | (cvt_e4m3x2(qv[6], qv[7]) << 16);
      st_v2(qT + (col + j) * R + row, o);
    }
  }
}

// ---------------------------------------------------------------- MX 1x32 rowwise

// CTA = 32 rows x 256 columns; warp w owns rows r0 + 4w + [0, 4); lane l
// covers columns 8l + [0, 8); a 32-block spans 4 lanes.
__global__ void __launch_bounds__(256) mx_quant_row_kernel(const uint16_t* __restrict__ x, int64_t R, int64_t C,
                                                           uint8_t* __restrict__ q, uint8_t* __restrict__ e8,
                                                           int mode) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t col = static_cast<int64_t>(blockIdx.x) * 256 + lane * 8;
  const int64_t rbase = static_cast<int64_t>(blockIdx.y) * 32 + warp * 4;
  const bool col_ok = col < C;
  uint4 v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t r = rbase + i;
    v[i] = (col_ok && r < R) ? ld_nc_v4(x + r * C + col) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t r = rbase + i;
    float a = amax8(v[i]);
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    if (!col_ok || r >= R) continue;
    const int E = mx_exponent(a, mode);
    st_v2(q + r * C + col, quant8_mul(v[i], pow2_neg(E)));
    if ((lane & 3) == 0) e8[r * (C / 32) + col / 32] = static_cast<uint8_t>(E + 127);
  }
}

// ---------------------------------------------------------------- launchers

static inline cudaError_t finish() { return cudaGetLastError(); }

cudaError_t launch_quant_1x128_row(const uint16_t* x, int64_t R, int64_t C, uint8_t* q, float* s, cudaStream_t st) {
  dim3 grid(static_cast<unsigned>(C / 128), static_cast<unsigned>(R / 128));
  quant_1x128_row_kernel<<<grid, 256, 0, st>>>(x, R, C, q, s);
  return finish();
}

cudaError_t launch_quant_1x128_col(const uint16_t* x, int64_t R, int64_t C, uint8_t* qT, float* s, cudaStream_t st) {
  dim3 grid(static_cast<unsigned>(C / 128), static_cast<unsigned>(R / 128));
  quant_1x128_col_kernel<<<grid, 256, 0, st>>>(x, R, C, qT, s);
  return finish();
}

cudaError_t launch_quant_128x128(const uint16_t* w, int64_t R, int64_t C, uint8_t* q, uint8_t* qT, float* s,
                                 int64_t s_ld, cudaStream_t st) {
  dim3 grid(static_cast<unsigned>(C / 128), static_cast<unsigned>(R / 128));
  quant_128x128_kernel<<<grid, 256, 0, st>>>(w, R, C, q, qT, s, s_ld);
  return finish();
}

cudaError_t launch_mx_quant_row(const uint16_t* x, int64_t R, int64_t C, uint8_t* q, uint8_t* e8, int mode,
                                cudaStream_t st) {
  dim3 grid(static_cast<unsigned>((C + 255) / 256), static_cast<unsigned>((R + 31) / 32));
  mx_quant_row_kernel<<<grid, 256, 0, st>>>(x, R, C, q, e8, mode);
  return finish();
}

cudaError_t launch_mx_quant_col(const uint16_t* x, int64_t G, int64_t R, int64_t C, uint8_t* qT, uint8_t* e8,
                                int mode, cudaStream_t st) {
  dim3 grid(static_cast<unsigned>((C + 127) / 128), static_cast<unsigned>((R + 127) / 128), static_cast<unsigned>(G));
  mx_quant_col_kernel<<<grid, 256, 0, st>>>(x, R, C, qT, e8, mode);
  return finish();
}

}  // namespace fp8bw
