// e4m3 quantizers of libfp8bw: 1x128 rowwise / colwise and 128x128 blockwise
// (fp32 scales), and MXFP8 1x32 rowwise / colwise / 3D-colwise (E8M0 scales).
//
// All of them are HBM-bound streaming kernels: each element is read once
// (2 B of bf16) and written once (1 B of e4m3), plus one scale per block.
// Loads are 16-byte vectors.  Block maxima are taken on packed bf16 pairs
// (max.xorsign.abs.bf16x2, exact) and reduced with warp shuffles; the
// blockwise division runs two elements per instruction (f32x2 FMUL2/FFMA2).
// The colwise-type kernels are persistent: each CTA streams 128x128 tiles
// through a ring of shared-memory buffers filled by cp.async (coalesced row
// loads, swizzled 16-byte chunks) and gives every thread an 8x8 micro-tile
// whose columns it packs into e4m3 bytes, so every store is a coalesced
// 8-byte vector.
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "quant_math.cuh"

namespace fp8bw {

// ---------------------------------------------------------------- scale rules

// MXFP8 rule: unbiased E8M0 exponent E of a block from its amax.
//   RCEIL: smallest E with 448 * 2^E >= amax.  With amax = 1.m * 2^e and
//          448 = 1.75 * 2^8 this is e - 8, plus one when 1.m > 1.75.
//   FLOOR: floor(log2 amax) - 8 = e - 8.
// Clamped to [-127, 127]; zero and subnormal amax give -127.
//
// Every block max here is an exact bf16 value, taken as its magnitude bits
// A = (ef << 7) | m (8-bit biased exponent, 7-bit mantissa).  RCEIL's "plus
// one when 1.m > 1.75" (m > 0x60) is then the carry out of m + 0x1F, so
//   t = (A + round) >> 7,  round = 0x1F (RCEIL) or 0 (FLOOR),
// is E + 135.  The clamp E >= -127 is t >= 8 (it also catches ef = 0); the
// top clamp cannot bind (t <= 256).  The E8M0 byte E + 127 is t - 8 and the
// scale 2^-E has biased exponent 262 - t, in [6, 254]: always a normal bf16
// (and fp32), which the element scaling multiplies in as a bf16 operand.
struct MxScale {
  uint32_t e8;   // the E8M0 code E + 127
  uint16_t mul;  // 2^-E as bf16 bits (biased exponent 262 - t, zero mantissa)
};
__device__ __forceinline__ uint32_t mx_round(int mode) { return mode == 0 ? 0x1Fu : 0u; }
__device__ __forceinline__ MxScale mx_scale(uint32_t A, uint32_t round) {
  const uint32_t t = max((A + round) >> 7, 8u);
  return MxScale{t - 8u, static_cast<uint16_t>((262u - t) << 7)};
}
// Magnitude bits of the larger of the two bf16 values packed in `w` (the
// sign bits may be anything).
__device__ __forceinline__ uint32_t bf16_pair_max_bits(uint32_t w) { return max(w & 0x7FFFu, (w >> 16) & 0x7FFFu); }

// max(|a|, |b|) in each bf16 half (exact); the result's sign bits are
// meaningless (max.xorsign.abs sets them to the XOR of the inputs' signs).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t word(const uint4& v, int k) { return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w; }

// |x| max of 8 packed bf16: even elements in the low half, odd in the high.
__device__ __forceinline__ uint32_t absmax8(const uint4& v) {
  return absmax_bf16x2(absmax_bf16x2(v.x, v.y), absmax_bf16x2(v.z, v.w));
}

// Two such partial maxes (of rows a and b) folded into one word: row a's max
// in the low half, row b's in the high half.
__device__ __forceinline__ uint32_t fold_pair(uint32_t ma, uint32_t mb) {
  return absmax_bf16x2(__byte_perm(ma, mb, 0x5410), __byte_perm(ma, mb, 0x7632));
}

__device__ __forceinline__ uint32_t shfl_absmax(uint32_t m, int lane_mask) {
  return absmax_bf16x2(m, __shfl_xor_sync(0xffffffffu, m, lane_mask));
}

// Value c (0..7) of four packed maxes, as a non-negative fp32 (exact).
__device__ __forceinline__ float unpack_amax(const uint32_t (&m)[4], int c) {
  const uint32_t w = (c & 4) ? ((c & 2) ? m[3] : m[2]) : ((c & 2) ? m[1] : m[0]);
  return __uint_as_float((c & 1) ? (w & 0x7FFF0000u) : (w & 0x7FFFu) << 16);
}
// The same value as bf16 magnitude bits (c a compile-time constant).
__device__ __forceinline__ uint32_t unpack_amax_bits(const uint32_t (&m)[4], int c) {
  const uint32_t w = m[c >> 1];
  return (c & 1) ? (w >> 16) & 0x7FFFu : w & 0x7FFFu;
}

// Element j (0..7) of 8 packed bf16.
__device__ __forceinline__ float elem8(const uint4& v, int j) {
  const uint32_t w = word(v, j >> 1);
  return (j & 1) ? bf16hi_to_f32(w) : bf16lo_to_f32(w);
}

__device__ __forceinline__ float2 pair_of_word(uint32_t w) { return make_float2(bf16lo_to_f32(w), bf16hi_to_f32(w)); }

// Eight e4m3 codes of fl32(x / s) packed little-endian; ny = neg_recip(s).
__device__ __forceinline__ uint2 quant8_div(const uint4& v, float s, float ny) {
  const float2 S = make_float2(s, s), NY = make_float2(ny, ny);
  const float2 a = neg_div_by_scale2(pair_of_word(v.x), S, NY);
  const float2 b = neg_div_by_scale2(pair_of_word(v.y), S, NY);
  const float2 c = neg_div_by_scale2(pair_of_word(v.z), S, NY);
  const float2 d = neg_div_by_scale2(pair_of_word(v.w), S, NY);
  return make_uint2(e4m3x4_from_neg(a, b), e4m3x4_from_neg(c, d));
}

// Eight e4m3 codes of x * m (MX: m = 2^-E, an exact power of two).
// (lo, hi) of a packed bf16 pair times the bf16 power of two m, in fp32:
// the product is exact (or rounds once, where it falls below the fp32
// range, exactly as an fp32 multiply would), and adding -0 keeps the sign
// of a zero product.
__device__ __forceinline__ float2 bf16x2_times(uint32_t w, uint16_t m) {
  float2 r;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "fma.rn.f32.bf16 %0, lo, %3, %4;\n\tfma.rn.f32.bf16 %1, hi, %3, %4;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "r"(w), "h"(m), "f"(-0.0f));
  return r;
}
template <int kHi>
__device__ __forceinline__ float bf16_half_times(uint32_t w, uint16_t m) {
  float r;
  if (kHi)
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tfma.rn.f32.bf16 %0, hi, %2, %3;\n\t}"
        : "=f"(r) : "r"(w), "h"(m), "f"(-0.0f));
  else
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tfma.rn.f32.bf16 %0, lo, %2, %3;\n\t}"
        : "=f"(r) : "r"(w), "h"(m), "f"(-0.0f));
  return r;
}

__device__ __forceinline__ uint2 quant8_mul(const uint4& v, uint16_t m) {
  const float2 a = bf16x2_times(v.x, m), b = bf16x2_times(v.y, m);
  const float2 c = bf16x2_times(v.z, m), d = bf16x2_times(v.w, m);
  return make_uint2(__byte_perm(cvt_e4m3x2(a.x, a.y), cvt_e4m3x2(b.x, b.y), 0x5410),
                    __byte_perm(cvt_e4m3x2(c.x, c.y), cvt_e4m3x2(d.x, d.y), 0x5410));
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

// Rowwise 1x128 quantization of the eight row chunks a thread holds: thread
// (warp w, lane l) has rows r0 + 16w + 2i + (l >> 4), i = 0..7, columns
// c0 + 8 (l & 15) + [0, 8).  The 16 lanes of a row reduce its max (two rows
// per packed word); lane i of each half-warp then derives row i's scale and
// reciprocal once, and shuffles hand them to the other lanes.  Writes q and
// the row scales s[c0 / 128][row].
__device__ __forceinline__ void rowwise_quant(const uint4 (&v)[8], int64_t R, int64_t C, int64_t r0, int64_t c0,
                                              uint8_t* __restrict__ q, float* __restrict__ s) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = lane >> 4, l16 = lane & 15;
  uint32_t m[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) m[p] = fold_pair(absmax8(v[2 * p]), absmax8(v[2 * p + 1]));
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) {
#pragma unroll
    for (int p = 0; p < 4; ++p) m[p] = shfl_absmax(m[p], o);
  }
  const float sc = blockwise_scale(unpack_amax(m, l16 & 7));
  const float ny = neg_recip(sc);
  const int64_t rbase = r0 + warp * 16 + h;
  if (l16 < 8) s[(c0 / 128) * R + rbase + 2 * l16] = sc;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float si = __shfl_sync(0xffffffffu, sc, (lane & 16) | i);
    const float nyi = __shfl_sync(0xffffffffu, ny, (lane & 16) | i);
    st_v2(q + (rbase + 2 * i) * C + c0 + l16 * 8, quant8_div(v[i], si, nyi));
  }
}

// CTA = 128 rows x one 128-column block, all eight 16-byte loads per thread
// issued up front.
__global__ void __launch_bounds__(256) quant_1x128_row_kernel(const uint16_t* __restrict__ x, int64_t R, int64_t C,
                                                              uint8_t* __restrict__ q, float* __restrict__ s) {
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 128, r0 = static_cast<int64_t>(blockIdx.y) * 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t col = c0 + (lane & 15) * 8;
  uint4 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = ld_nc_v4(x + (r0 + warp * 16 + i * 2 + (lane >> 4)) * C + col);
  rowwise_quant(v, R, C, r0, c0, q, s);
}

// ---------------------------------------------------------------- staged 128x128 tiles

// A 128-row x 128-column bf16 tile in shared memory (32 KB) whose 16-byte
// chunks are XOR-swizzled by the row's 8-row group: chunk k of row r lives at
// chunk k ^ ((r >> 3) & 15).  Row-major accesses (a half-warp per row) and the
// 8x8 micro-tile reads of the colwise path (16 lanes down one column group)
// then both run at the minimum number of shared-memory wavefronts.
struct StagedTile {
  uint4 chunk[128][16];
};

__device__ __forceinline__ int swz(int r, int k) { return k ^ ((r >> 3) & 15); }

// The colwise-type quantizers are persistent: each CTA walks tiles
// blockIdx.x, blockIdx.x + gridDim.x, ... through a ring of kQuantStages
// staged tiles filled by cp.async, so the loads of the next tiles are in
// flight while the current one is quantized and stored.
#ifndef FP8BW_QSTAGES
#define FP8BW_QSTAGES 3
#endif
#ifndef FP8BW_QCTAS
#define FP8BW_QCTAS 2
#endif
constexpr int kQuantStages = FP8BW_QSTAGES;
constexpr int kQuantCtasPerSm = FP8BW_QCTAS;
constexpr size_t kQuantSmem = kQuantStages * sizeof(StagedTile);

__device__ __forceinline__ void cp_async_16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Issues the copy of rows [r0, r0 + 128) x columns [c0, c0 + 128) of x[R, C]
// into `t`: warp w, step i, half-warp h takes row 16w + 2i + h, lane (l & 15)
// chunk (l & 15) -- two 256-byte row segments per warp instruction.  Rows >= R
// and columns >= C are zero-filled (C % 8 == 0), reading nothing.
__device__ __forceinline__ void fetch_tile(const uint16_t* __restrict__ x, int64_t R, int64_t C, int64_t r0,
                                           int64_t c0, StagedTile& t) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = lane >> 4, k = lane & 15;
  const int64_t col = c0 + k * 8;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = warp * 16 + i * 2 + h;
    const bool ok = r0 + r < R && col < C;
    cp_async_16(&t.chunk[r][swz(r, k)], ok ? x + (r0 + r) * C + col : x, ok ? 16u : 0u);
  }
}

// The thread's 8 row chunks of the staged tile, in the mapping of fetch_tile.
__device__ __forceinline__ void read_rows(const StagedTile& t, uint4 (&v)[8]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = lane >> 4, k = lane & 15;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = warp * 16 + i * 2 + h;
    v[i] = t.chunk[r][swz(r, k)];
  }
}

// Tiles of a stack of G matrices [R, C]: tile t -> matrix g, row band rb,
// column block cb (column blocks fastest).
struct TileSpace {
  int64_t R, C;
  int tiles_c, tiles_r, G;
};

struct TileCursor {
  int g, rb, cb;
};

// A stride of whole tiles split into column blocks, row bands and matrices.
struct TileStep {
  int dcb, drb, dg;
};

__device__ __forceinline__ TileCursor cursor_at(const TileSpace& ts, int64_t t) {
  const int64_t per_matrix = static_cast<int64_t>(ts.tiles_c) * ts.tiles_r;
  TileCursor c;
  c.g = static_cast<int>(t / per_matrix);
  const int64_t u = t - c.g * per_matrix;
  c.rb = static_cast<int>(u / ts.tiles_c);
  c.cb = static_cast<int>(u - static_cast<int64_t>(c.rb) * ts.tiles_c);
  return c;
}

__device__ __forceinline__ TileStep step_of(const TileSpace& ts, int stride) {
  const int rest = stride / ts.tiles_c;
  return TileStep{stride % ts.tiles_c, rest % ts.tiles_r, rest / ts.tiles_r};
}

// Moves the cursor `d` tiles on with carries instead of divisions.
__device__ __forceinline__ void advance(TileCursor& c, const TileSpace& ts, const TileStep& d) {
  c.cb += d.dcb;
  int carry = c.cb >= ts.tiles_c;
  if (carry) c.cb -= ts.tiles_c;
  c.rb += d.drb + carry;
  carry = c.rb >= ts.tiles_r;
  if (carry) c.rb -= ts.tiles_r;
  c.g += d.dg + carry;
}

// Runs body(tile, g, r0, c0) on the tiles blockIdx.x, blockIdx.x + gridDim.x,
// ..., kQuantStages - 1 tiles ahead of the loads.  Each iteration waits for
// its own tile's copies (cp.async.wait_group), then a CTA barrier makes them
// visible to all threads and guarantees that everyone has left the previous
// tile, whose buffer the next prefetch overwrites.
template <typename Body>
__device__ __forceinline__ void for_each_staged_tile(const uint16_t* __restrict__ x, const TileSpace& ts,
                                                     StagedTile* ring, Body&& body) {
  const TileStep d = step_of(ts, gridDim.x);
  TileCursor pre = cursor_at(ts, blockIdx.x);
  TileCursor cur = pre;
  const int64_t matrix = ts.R * ts.C;
#pragma unroll
  for (int s = 0; s < kQuantStages - 1; ++s) {
    if (pre.g < ts.G) fetch_tile(x + pre.g * matrix, ts.R, ts.C, pre.rb * 128ll, pre.cb * 128ll, ring[s]);
    cp_async_commit();
    advance(pre, ts, d);
  }
  int stage = 0;
  while (cur.g < ts.G) {
    cp_async_wait<kQuantStages - 2>();
    __syncthreads();
    const int ahead = stage == 0 ? kQuantStages - 1 : stage - 1;
    if (pre.g < ts.G) fetch_tile(x + pre.g * matrix, ts.R, ts.C, pre.rb * 128ll, pre.cb * 128ll, ring[ahead]);
    cp_async_commit();
    advance(pre, ts, d);
    body(ring[stage], static_cast<int64_t>(cur.g), cur.rb * 128ll, cur.cb * 128ll);
    advance(cur, ts, d);
    stage = stage + 1 == kQuantStages ? 0 : stage + 1;
  }
  cp_async_wait<0>();
}

// Thread (warp w, lane l) of the colwise path owns the 8x8 micro-tile at tile
// rows 8 * (l & 15) + [0, 8) and columns 8 * (2w + (l >> 4)) + [0, 8).
__device__ __forceinline__ void read_microtile(const StagedTile& t, uint4 (&v)[8]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rg = lane & 15, cg = warp * 2 + (lane >> 4);
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = t.chunk[rg * 8 + i][cg ^ rg];  // swz(8 rg + i, cg)
}

// Column j of the micro-tile (8 consecutive rows) as 8 e4m3 codes of
// fl32(x / s), or of x * m for MX.
__device__ __forceinline__ uint2 column8_div(const uint4 (&v)[8], int j, float s, float ny) {
  const float2 S = make_float2(s, s), NY = make_float2(ny, ny);
  const float2 a = neg_div_by_scale2(make_float2(elem8(v[0], j), elem8(v[1], j)), S, NY);
  const float2 b = neg_div_by_scale2(make_float2(elem8(v[2], j), elem8(v[3], j)), S, NY);
  const float2 c = neg_div_by_scale2(make_float2(elem8(v[4], j), elem8(v[5], j)), S, NY);
  const float2 d = neg_div_by_scale2(make_float2(elem8(v[6], j), elem8(v[7], j)), S, NY);
  return make_uint2(e4m3x4_from_neg(a, b), e4m3x4_from_neg(c, d));
}

template <int kJ>
__device__ __forceinline__ float elem8_times(const uint4& v, uint16_t m) {
  return bf16_half_times<kJ & 1>(word(v, kJ >> 1), m);
}
template <int kJ>
__device__ __forceinline__ uint2 column8_mul(const uint4 (&v)[8], uint16_t m) {
  const float2 a = make_float2(elem8_times<kJ>(v[0], m), elem8_times<kJ>(v[1], m));
  const float2 b = make_float2(elem8_times<kJ>(v[2], m), elem8_times<kJ>(v[3], m));
  const float2 c = make_float2(elem8_times<kJ>(v[4], m), elem8_times<kJ>(v[5], m));
  const float2 d = make_float2(elem8_times<kJ>(v[6], m), elem8_times<kJ>(v[7], m));
  return make_uint2(__byte_perm(cvt_e4m3x2(a.x, a.y), cvt_e4m3x2(b.x, b.y), 0x5410),
                    __byte_perm(cvt_e4m3x2(c.x, c.y), cvt_e4m3x2(d.x, d.y), 0x5410));
}

// Packed |x| maxes of the micro-tile's column pairs (2k, 2k + 1) over its
// 8 rows.
__device__ __forceinline__ void column_pair_maxes(const uint4 (&v)[8], uint32_t (&m)[4]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    m[k] = word(v[0], k);
#pragma unroll
    for (int i = 1; i < 8; ++i) m[k] = absmax_bf16x2(m[k], word(v[i], k));
  }
}

// Colwise quantization of the staged tile.  A column block spans the 16
// lanes of a half-warp (blockwise, 128 rows) or 4 of them (MX, 32 rows); its
// max is reduced with shuffles inside that group, two columns per packed
// word.  Each column of the micro-tile is stored as 8 bytes at
// qT[col][row .. row + 8): the 16 lanes of a half-warp cover 128 contiguous
// bytes of one qT row.
template <bool kMX>
__device__ __forceinline__ void colwise_from_tile(const StagedTile& t, int64_t R, int64_t C, int64_t r0, int64_t c0,
                                                  uint8_t* __restrict__ qT, float* __restrict__ s,
                                                  uint8_t* __restrict__ e8, int mode) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rg = lane & 15;
  const int64_t row = r0 + rg * 8;
  const int64_t col = c0 + (warp * 2 + (lane >> 4)) * 8;

  uint4 v[8];
  read_microtile(t, v);
  uint32_t m[4];
  column_pair_maxes(v, m);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    m[k] = shfl_absmax(m[k], 1);
    m[k] = shfl_absmax(m[k], 2);
    if (!kMX) {
      m[k] = shfl_absmax(m[k], 4);
      m[k] = shfl_absmax(m[k], 8);
    }
  }
  if (kMX) {
    if (!(row < R && col < C)) return;  // R % 32 == 0: a 32-row MX block is all in or all out
    const uint32_t round = mx_round(mode);
    uint8_t* qcol = qT + col * R + row;
    uint8_t* ecol = e8 + col * (R / 32) + row / 32;
    auto column = [&](auto J) {
      constexpr int j = decltype(J)::value;
      const MxScale sc = mx_scale(unpack_amax_bits(m, j), round);
      if ((rg & 3) == 0) ecol[j * (R / 32)] = static_cast<uint8_t>(sc.e8);
      st_v2(qcol + j * R, column8_mul<j>(v, sc.mul));
    };
    column(std::integral_constant<int, 0>{});
    column(std::integral_constant<int, 1>{});
    column(std::integral_constant<int, 2>{});
    column(std::integral_constant<int, 3>{});
    column(std::integral_constant<int, 4>{});
    column(std::integral_constant<int, 5>{});
    column(std::integral_constant<int, 6>{});
    column(std::integral_constant<int, 7>{});
  } else {
    // Blockwise tiles are whole (R, C multiples of 128).  Lane j of each
    // half-warp derives column j's scale; shuffles hand it to the others.
    const float sc = blockwise_scale(unpack_amax(m, rg & 7));
    const float ny = neg_recip(sc);
    if (rg < 8) s[(r0 / 128) * C + col + rg] = sc;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float sj = __shfl_sync(0xffffffffu, sc, (lane & 16) | j);
      const float nyj = __shfl_sync(0xffffffffu, ny, (lane & 16) | j);
      st_v2(qT + (col + j) * R + row, column8_div(v, j, sj, nyj));
    }
  }
}

// Rowwise 1x128 quantization of the staged tile's rows.
__device__ __forceinline__ void rowwise_from_tile(const StagedTile& t, int64_t R, int64_t C, int64_t r0, int64_t c0,
                                                  uint8_t* __restrict__ q, float* __restrict__ s) {
  uint4 v[8];
  read_rows(t, v);
  rowwise_quant(v, R, C, r0, c0, q, s);
}

__device__ __forceinline__ TileSpace tile_space(int64_t G, int64_t R, int64_t C) {
  return TileSpace{R, C, static_cast<int>((C + 127) / 128), static_cast<int>((R + 127) / 128), static_cast<int>(G)};
}

__global__ void __launch_bounds__(256, kQuantCtasPerSm)
    quant_1x128_col_kernel(const uint16_t* __restrict__ x, int64_t R, int64_t C, uint8_t* __restrict__ qT,
                           float* __restrict__ s) {
  extern __shared__ __align__(128) uint8_t quant_smem[];
  StagedTile* ring = reinterpret_cast<StagedTile*>(quant_smem);
  for_each_staged_tile(x, tile_space(1, R, C), ring, [&](const StagedTile& t, int64_t, int64_t r0, int64_t c0) {
    colwise_from_tile<false>(t, R, C, r0, c0, qT, s, nullptr, 0);
  });
}

// Both 1x128 quantizations of one tile from a single read of x.
__global__ void __launch_bounds__(256, kQuantCtasPerSm)
    quant_1x128_rowcol_kernel(const uint16_t* __restrict__ x, int64_t R, int64_t C, uint8_t* __restrict__ q,
                              float* __restrict__ s, uint8_t* __restrict__ qT, float* __restrict__ sT) {
  extern __shared__ __align__(128) uint8_t quant_smem[];
  StagedTile* ring = reinterpret_cast<StagedTile*>(quant_smem);
  for_each_staged_tile(x, tile_space(1, R, C), ring, [&](const StagedTile& t, int64_t, int64_t r0, int64_t c0) {
    rowwise_from_tile(t, R, C, r0, c0, q, s);
    colwise_from_tile<false>(t, R, C, r0, c0, qT, sT, nullptr, 0);
  });
}

// Rowwise MX (1x32 along the columns) of the staged tile's rows, in the
// mapping of read_rows: a 32-column block spans the 4 lanes that hold its
// chunks, which reduce its max with two shuffles.  Same arithmetic as
// mx_quant_row_kernel.
__device__ __forceinline__ void rowwise_mx_from_tile(const StagedTile& t, int64_t R, int64_t C, int64_t r0, int64_t c0,
                                                     uint8_t* __restrict__ q, uint8_t* __restrict__ e8, int mode) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = lane >> 4, l16 = lane & 15;
  const int64_t col = c0 + l16 * 8;
  const int64_t rfirst = r0 + warp * 16 + h;  // rows rfirst + 2i
  const uint32_t round = mx_round(mode);
  uint8_t* qrow = q + rfirst * C + col;
  uint8_t* erow = e8 + rfirst * (C / 32) + col / 32;
  uint4 v[8];
  read_rows(t, v);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t mm = shfl_absmax(shfl_absmax(absmax8(v[i]), 1), 2);
    if (rfirst + 2 * i >= R || col >= C) continue;  // C % 32 == 0: a 32-column block is all in or all out
    const MxScale sc = mx_scale(bf16_pair_max_bits(mm), round);
    st_v2(qrow + 2 * i * C, quant8_mul(v[i], sc.mul));
    if ((l16 & 3) == 0) erow[2 * i * (C / 32)] = static_cast<uint8_t>(sc.e8);
  }
}

// Both MX quantizations of G stacked matrices [R, C] from one read: rowwise
// (1x32 along C) into q [G*R, C], e8 [G*R][C/32] and colwise (32 along R)
// into qT [G, C, R], e8T [G][C][R/32].
__global__ void __launch_bounds__(256, kQuantCtasPerSm)
    mx_quant_rowcol_kernel(const uint16_t* __restrict__ x, int64_t G, int64_t R, int64_t C, uint8_t* __restrict__ q,
                           uint8_t* __restrict__ e8, uint8_t* __restrict__ qT, uint8_t* __restrict__ e8T, int mode) {
  extern __shared__ __align__(128) uint8_t quant_smem[];
  StagedTile* ring = reinterpret_cast<StagedTile*>(quant_smem);
  for_each_staged_tile(x, tile_space(G, R, C), ring, [&](const StagedTile& t, int64_t g, int64_t r0, int64_t c0) {
    rowwise_mx_from_tile(t, R, C, r0, c0, q + g * R * C, e8 + g * R * (C / 32), mode);
    colwise_from_tile<true>(t, R, C, r0, c0, qT + g * R * C, nullptr, e8T + g * C * (R / 32), mode);
  });
}

// G stacked matrices (the 3D expert case; G = 1 for a plain 2D operand).
__global__ void __launch_bounds__(256, kQuantCtasPerSm)
    mx_quant_col_kernel(const uint16_t* __restrict__ x, int64_t G, int64_t R, int64_t C, uint8_t* __restrict__ qT,
                        uint8_t* __restrict__ e8, int mode) {
  extern __shared__ __align__(128) uint8_t quant_smem[];
  StagedTile* ring = reinterpret_cast<StagedTile*>(quant_smem);
  for_each_staged_tile(x, tile_space(G, R, C), ring, [&](const StagedTile& t, int64_t g, int64_t r0, int64_t c0) {
    colwise_from_tile<true>(t, R, C, r0, c0, qT + g * R * C, nullptr, e8 + g * C * (R / 32), mode);
  });
}

// ---------------------------------------------------------------- 128x128

// One scale for the whole tile: the max of the rows reduced over the CTA; q
// is written row-major (a half-warp per 128-byte row segment), qT from the
// micro-tiles.
__global__ void __launch_bounds__(256, kQuantCtasPerSm)
    quant_128x128_kernel(const uint16_t* __restrict__ x, int64_t R, int64_t C, uint8_t* __restrict__ q,
                         uint8_t* __restrict__ qT, float* __restrict__ s, int64_t s_ld) {
  extern __shared__ __align__(128) uint8_t quant_smem[];
  StagedTile* ring = reinterpret_cast<StagedTile*>(quant_smem);
  __shared__ float warp_max[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for_each_staged_tile(x, tile_space(1, R, C), ring, [&](const StagedTile& t, int64_t, int64_t r0, int64_t c0) {
    uint4 v[8];
    read_rows(t, v);
    uint32_t m = absmax8(v[0]);
#pragma unroll
    for (int i = 1; i < 8; ++i) m = absmax_bf16x2(m, absmax8(v[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = shfl_absmax(m, o);
    // warp_max is rewritten only after the next tile's leading barrier, which
    // every thread reaches after its reads below.
    if (lane == 0) warp_max[warp] = fmaxf(__uint_as_float((m & 0x7FFFu) << 16), __uint_as_float(m & 0x7FFF0000u));
    __syncthreads();
    float a = warp_max[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) a = fmaxf(a, warp_max[w]);
    const float sc = blockwise_scale(a);
    const float ny = neg_recip(sc);
    if (threadIdx.x == 0) s[(r0 / 128) * s_ld + c0 / 128] = sc;

    const int h = lane >> 4, l16 = lane & 15;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int64_t r = r0 + warp * 16 + i * 2 + h;
      st_v2(q + r * C + c0 + l16 * 8, quant8_div(v[i], sc, ny));
    }
    if (qT != nullptr) {
      const int64_t row = r0 + (lane & 15) * 8;
      const int64_t col = c0 + (warp * 2 + (lane >> 4)) * 8;
      read_microtile(t, v);
#pragma unroll
      for (int j = 0; j < 8; ++j) st_v2(qT + (col + j) * R + row, column8_div(v, j, sc, ny));
    }
  });
}

// 128x128 without the transposed copy: one CTA per tile, the tile loaded
// straight into registers (thread (warp w, lane l) holds 16-byte chunk l % 16
// of rows 16w + 2i + l / 16, i < 8: each half-warp reads one 256-byte row
// segment), so the loads of every resident CTA are in flight at once and the
// hardware balances tiles across SMs; the CTA's max is reduced through
// shared memory.  Same arithmetic as quant_128x128_kernel.
__global__ void __launch_bounds__(256) quant_128x128_direct_kernel(const uint16_t* __restrict__ x, int64_t C,
                                                                   uint8_t* __restrict__ q, float* __restrict__ s,
                                                                   int64_t s_ld) {
  __shared__ float warp_max[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = lane >> 4, l16 = lane & 15;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 128 + warp * 16 + h;
  const int64_t c = static_cast<int64_t>(blockIdx.x) * 128 + l16 * 8;
  uint4 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = ld_nc_v4(x + (r0 + 2 * i) * C + c);
  uint32_t m = absmax8(v[0]);
#pragma unroll
  for (int i = 1; i < 8; ++i) m = absmax_bf16x2(m, absmax8(v[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = shfl_absmax(m, o);
  if (lane == 0) warp_max[warp] = fmaxf(__uint_as_float((m & 0x7FFFu) << 16), __uint_as_float(m & 0x7FFF0000u));
  __syncthreads();
  float a = warp_max[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) a = fmaxf(a, warp_max[w]);
  const float sc = blockwise_scale(a);
  const float ny = neg_recip(sc);
  if (threadIdx.x == 0) s[static_cast<int64_t>(blockIdx.y) * s_ld + blockIdx.x] = sc;
#pragma unroll
  for (int i = 0; i < 8; ++i) st_v2(q + (r0 + 2 * i) * C + c, quant8_div(v[i], sc, ny));
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
  const uint32_t round = mx_round(mode);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t r = rbase + i;
    const uint32_t mm = shfl_absmax(shfl_absmax(absmax8(v[i]), 1), 2);
    if (!col_ok || r >= R) continue;
    const MxScale sc = mx_scale(bf16_pair_max_bits(mm), round);
    st_v2(q + r * C + col, quant8_mul(v[i], sc.mul));
    if ((lane & 3) == 0) e8[r * (C / 32) + col / 32] = static_cast<uint8_t>(sc.e8);
  }
}

// ---------------------------------------------------------------- launchers

static inline cudaError_t finish() { return cudaGetLastError(); }

// Per device, once: the staged-tile kernels' dynamic shared memory limit and
// the SM count that sizes their persistent grids.
static int staged_grid_cap() {
  static std::mutex mu;
  static int sms[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 0;
    const int smem = static_cast<int>(kQuantSmem);
    if (cudaFuncSetAttribute(quant_1x128_col_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) ||
        cudaFuncSetAttribute(quant_1x128_rowcol_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) ||
        cudaFuncSetAttribute(mx_quant_col_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) ||
        cudaFuncSetAttribute(mx_quant_rowcol_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) ||
        cudaFuncSetAttribute(quant_128x128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem))
      return 0;
    sms[dev] = n;
  }
  return sms[dev] * kQuantCtasPerSm;
}

static inline bool staged_grid(int64_t tiles, dim3& grid) {
  const int cap = staged_grid_cap();
  if (cap <= 0) return false;
  grid = dim3(static_cast<unsigned>(tiles < cap ? tiles : cap));
  return true;
}

cudaError_t launch_quant_1x128_row(const uint16_t* x, int64_t R, int64_t C, uint8_t* q, float* s, cudaStream_t st) {
  dim3 grid(static_cast<unsigned>(C / 128), static_cast<unsigned>(R / 128));
  quant_1x128_row_kernel<<<grid, 256, 0, st>>>(x, R, C, q, s);
  return finish();
}

cudaError_t launch_quant_1x128_col(const uint16_t* x, int64_t R, int64_t C, uint8_t* qT, float* s, cudaStream_t st) {
  dim3 grid;
  if (!staged_grid((R / 128) * (C / 128), grid)) return cudaErrorInvalidConfiguration;
  quant_1x128_col_kernel<<<grid, 256, kQuantSmem, st>>>(x, R, C, qT, s);
  return finish();
}

cudaError_t launch_quant_1x128_rowcol(const uint16_t* x, int64_t R, int64_t C, uint8_t* q, float* s, uint8_t* qT,
                                      float* sT, cudaStream_t st) {
  dim3 grid;
  if (!staged_grid((R / 128) * (C / 128), grid)) return cudaErrorInvalidConfiguration;
  quant_1x128_rowcol_kernel<<<grid, 256, kQuantSmem, st>>>(x, R, C, q, s, qT, sT);
  return finish();
}

cudaError_t launch_quant_128x128(const uint16_t* w, int64_t R, int64_t C, uint8_t* q, uint8_t* qT, float* s,
                                 int64_t s_ld, cudaStream_t st) {
  if (qT == nullptr) {
    quant_128x128_direct_kernel<<<dim3(static_cast<unsigned>(C / 128), static_cast<unsigned>(R / 128)), 256, 0, st>>>(
        w, C, q, s, s_ld);
    return finish();
  }
  dim3 grid;
  if (!staged_grid((R / 128) * (C / 128), grid)) return cudaErrorInvalidConfiguration;
  quant_128x128_kernel<<<grid, 256, kQuantSmem, st>>>(w, R, C, q, qT, s, s_ld);
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
  dim3 grid;
  if (!staged_grid(G * ((R + 127) / 128) * ((C + 127) / 128), grid)) return cudaErrorInvalidConfiguration;
  mx_quant_col_kernel<<<grid, 256, kQuantSmem, st>>>(x, G, R, C, qT, e8, mode);
  return finish();
}

cudaError_t launch_mx_quant_rowcol(const uint16_t* x, int64_t G, int64_t R, int64_t C, uint8_t* q, uint8_t* e8,
                                   uint8_t* qT, uint8_t* e8T, int mode, cudaStream_t st) {
  dim3 grid;
  if (!staged_grid(G * ((R + 127) / 128) * ((C + 127) / 128), grid)) return cudaErrorInvalidConfiguration;
  mx_quant_rowcol_kernel<<<grid, 256, kQuantSmem, st>>>(x, G, R, C, q, e8, qT, e8T, mode);
  return finish();
}

}  // namespace fp8bw
