// e4m3 quantizers of libfp8bw: 1x128 rowwise / colwise and 128x128 blockwise
// (fp32 scales), and MXFP8 1x32 rowwise / colwise / 3D-colwise (E8M0 scales).
//
// All of them are HBM-bound streaming kernels: each element is read once
// (2 B of bf16) and written once (1 B of e4m3), plus one scale per block.
// Loads are 16-byte vectors; block maxima are reduced with warp shuffles; the
// colwise kernels stage each 128x128 tile in shared memory (coalesced loads,
// swizzled chunks), then give every thread an 8x8 micro-tile whose columns it
// packs into e4m3 bytes, so every store is a coalesced 8-byte vector.
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

// ---------------------------------------------------------------- staged 128x128 tiles

// A 128-row x 128-column bf16 tile in shared memory (32 KB) whose 16-byte
// chunks are XOR-swizzled by the row's 8-row group: chunk k of row r lives at
// chunk k ^ ((r >> 3) & 15).  Row-major writes (a half-warp per row) and the
// 8x8 micro-tile reads of the colwise path (16 lanes down one column group)
// then both run at the minimum number of shared-memory wavefronts.
struct StagedTile {
  uint4 chunk[128][16];
};

__device__ __forceinline__ int swz(int r, int k) { return k ^ ((r >> 3) & 15); }

// Loads rows [r0, r0 + 128) x columns [c0, c0 + 128) of x[R, C] with
// coalesced 16-byte vectors -- warp w, step i: half-warp h takes row
// 16w + 2i + h, lane (l & 15) chunk (l & 15) -- into `v` and into the staged
// tile.  Rows >= R and columns >= C read as zero (C % 8 == 0).
__device__ __forceinline__ void load_tile(const uint16_t* __restrict__ x, int64_t R, int64_t C, int64_t r0,
                                          int64_t c0, StagedTile& t, uint4 (&v)[8]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = lane >> 4, k = lane & 15;
  const int64_t col = c0 + k * 8;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = warp * 16 + i * 2 + h;
    v[i] = (r0 + r < R && col < C) ? ld_nc_v4(x + (r0 + r) * C + col) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = warp * 16 + i * 2 + h;
    t.chunk[r][swz(r, k)] = v[i];
  }
}

// Thread (warp w, lane l) of the colwise path owns the 8x8 micro-tile at tile
// rows 8 * (l & 15) + [0, 8) and columns 8 * (2w + (l >> 4)) + [0, 8).
__device__ __forceinline__ void read_microtile(const StagedTile& t, uint4 (&v)[8]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rg = lane & 15, cg = warp * 2 + (lane >> 4);
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = t.chunk[rg * 8 + i][cg ^ rg];  // swz(8 rg + i, cg)
}

// Packs column j of the micro-tile (8 consecutive rows, already scaled) into
// 8 e4m3 bytes and stores them at qT[col][row .. row + 8): the 16 lanes of a
// half-warp cover 128 contiguous bytes of one qT row.
__device__ __forceinline__ void store_column8(uint8_t* qT, int64_t R, int64_t col, int64_t row, const float (&qv)[8]) {
  uint2 o;
  o.x = cvt_e4m3x2(qv[0], qv[1]) | (cvt_e4m3x2(qv[2], qv[3]) << 16);
  o.y = cvt_e4m3x2(qv[4], qv[5]) | (cvt_e4m3x2(qv[6], qv[7]) << 16);
  st_v2(qT + col * R + row, o);
}

// Colwise quantization of the staged tile: a column block spans the 16 lanes
// of a half-warp (blockwise, 128 rows) or 4 of them (MX, 32 rows); its max is
// reduced with shuffles inside that group.
template <bool kMX>
__device__ __forceinline__ void colwise_from_tile(const StagedTile& t, int64_t R, int64_t C, int64_t r0, int64_t c0,
                                                  uint8_t* __restrict__ qT, float* __restrict__ s,
                                                  uint8_t* __restrict__ e8, int mode) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rg = lane & 15;
  const int64_t row = r0 + rg * 8;
  const int64_t col = c0 + (warp * 2 + (lane >> 4)) * 8;
  const bool ok = row < R && col < C;  // R % 32 == 0: a 32-row MX block is all in or all out

  uint4 v[8];
  read_microtile(t, v);
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
  if (!ok) return;

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
    store_column8(qT, R, col + j, row, qv);
  }
}

// Rowwise 1x128 quantization of the 8 row chunks a thread loaded in
// load_tile (the half-warp of each row holds its 128 columns).  Writes q and
// leaves each row's scale in s_rows[row of the tile].
__device__ __forceinline__ void rowwise_from_regs(const uint4 (&v)[8], int64_t C, int64_t r0, int64_t c0,
                                                  uint8_t* __restrict__ q, float* s_rows) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = lane >> 4, l16 = lane & 15;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float a = amax8(v[i]);
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 8));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    const float sc = blockwise_scale(a);
    const int rl = warp * 16 + i * 2 + h;
    st_v2(q + (r0 + rl) * C + c0 + l16 * 8, quant8_div(v[i], sc, __frcp_rn(sc)));
    if (l16 == 0) s_rows[rl] = sc;
  }
}

__global__ void __launch_bounds__(256) quant_1x128_col_kernel(const uint16_t* __restrict__ x, int64_t R, int64_t C,
                                                              uint8_t* __restrict__ qT, float* __restrict__ s) {
  __shared__ StagedTile tile;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 128, c0 = static_cast<int64_t>(blockIdx.x) * 128;
  uint4 v[8];
  load_tile(x, R, C, r0, c0, tile, v);
  __syncthreads();
  colwise_from_tile<false>(tile, R, C, r0, c0, qT, s, nullptr, 0);
}

// Both 1x128 quantizations of one tile from a single read of x: rowwise from
// the loaded registers, colwise from the staged tile.
__global__ void __launch_bounds__(256) quant_1x128_rowcol_kernel(const uint16_t* __restrict__ x, int64_t R, int64_t C,
                                                                 uint8_t* __restrict__ q, float* __restrict__ s,
                                                                 uint8_t* __restrict__ qT, float* __restrict__ sT) {
  __shared__ StagedTile tile;
  __shared__ float s_rows[128];
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 128, c0 = static_cast<int64_t>(blockIdx.x) * 128;
  uint4 v[8];
  load_tile(x, R, C, r0, c0, tile, v);
  rowwise_from_regs(v, C, r0, c0, q, s_rows);
  __syncthreads();
  if (threadIdx.x < 128) s[static_cast<int64_t>(blockIdx.x) * R + r0 + threadIdx.x] = s_rows[threadIdx.x];
  colwise_from_tile<false>(tile, R, C, r0, c0, qT, sT, nullptr, 0);
}

// grid.z = expert index for the 3D case (per-expert strides passed in).
__global__ void __launch_bounds__(256) mx_quant_col_kernel(const uint16_t* __restrict__ x, int64_t R, int64_t C,
                                                           uint8_t* __restrict__ qT, uint8_t* __restrict__ e8,
                                                           int mode) {
  __shared__ StagedTile tile;
  const int64_t g = blockIdx.z;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 128, c0 = static_cast<int64_t>(blockIdx.x) * 128;
  uint4 v[8];
  load_tile(x + g * R * C, R, C, r0, c0, tile, v);
  __syncthreads();
  colwise_from_tile<true>(tile, R, C, r0, c0, qT + g * R * C, nullptr, e8 + g * C * (R / 32), mode);
}

// ---------------------------------------------------------------- 128x128

// One scale for the whole tile: the max of the loaded registers reduced over
// the CTA; q is written row-major from registers (a half-warp per 128-byte row
// segment), qT from the staged tile's micro-tiles.
__global__ void __launch_bounds__(256) quant_128x128_kernel(const uint16_t* __restrict__ x, int64_t R, int64_t C,
                                                            uint8_t* __restrict__ q, uint8_t* __restrict__ qT,
                                                            float* __restrict__ s, int64_t s_ld) {
  __shared__ StagedTile tile;
  __shared__ float warp_max[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 128, c0 = static_cast<int64_t>(blockIdx.x) * 128;
  uint4 v[8];
  load_tile(x, R, C, r0, c0, tile, v);
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) a = fmaxf(a, amax8(v[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  if (lane == 0) warp_max[warp] = a;
  __syncthreads();  // also publishes the staged tile
  a = warp_max[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) a = fmaxf(a, warp_max[w]);
  const float sc = blockwise_scale(a);
  const float y = __frcp_rn(sc);
  if (threadIdx.x == 0) s[blockIdx.y * s_ld + blockIdx.x] = sc;

  const int h = lane >> 4, l16 = lane & 15;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t r = r0 + warp * 16 + i * 2 + h;
    st_v2(q + r * C + c0 + l16 * 8, quant8_div(v[i], sc, y));
  }
  if (qT != nullptr) {
    const int rg = lane & 15;
    const int64_t row = r0 + rg * 8;
    const int64_t col = c0 + (warp * 2 + (lane >> 4)) * 8;
    read_microtile(tile, v);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float qv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) qv[i] = div_by_scale(elem8(v[i], j), sc, y);
      store_column8(qT, R, col + j, row, qv);
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

cudaError_t launch_quant_1x128_rowcol(const uint16_t* x, int64_t R, int64_t C, uint8_t* q, float* s, uint8_t* qT,
                                      float* sT, cudaStream_t st) {
  dim3 grid(static_cast<unsigned>(C / 128), static_cast<unsigned>(R / 128));
  quant_1x128_rowcol_kernel<<<grid, 256, 0, st>>>(x, R, C, q, s, qT, sT);
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
