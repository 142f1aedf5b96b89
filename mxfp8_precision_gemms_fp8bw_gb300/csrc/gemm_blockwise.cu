// Blockwise-scaled e4m3 GEMM on the 5th-generation tensor cores (tcgen05),
// the three GEMMs of Float8BlockwiseLinear (PR #2386 description; PR #4295
// Summary):
//
//   out[i, j] = sum_kb  sa[kb][i] * sb(kb, j) * P_kb[i, j],
//   P_kb[i, j] = sum_{k in block kb} dec(A[i, k]) * dec(B[j, k])
//
// where kb runs over 128-deep contraction blocks.  The per-block scales are
// arbitrary fp32 values (amax / 448), so they cannot ride on the tensor
// core's power-of-two block scaling; instead each P_kb is accumulated by the
// tensor core into tensor memory (TMEM) and "promoted" by CUDA cores into
// fp32 register accumulators: acc += P_kb * sa * sb.
//
// Kernel structure (one persistent CTA per SM, 384 threads):
//   warp 0      TMA producer: A tile 128x128 and B tile 256x128 (e4m3,
//               128-byte swizzle) per contraction block into a ring of 3
//               stages (one B scale per block) or 4 (per-column B scale).
//   warps 1-2   warp 1 allocates / frees the 512 TMEM columns; one thread
//               of each issues 4 tcgen05.mma (K = 32 each) per block, warp 1
//               for the even blocks into TMEM partial buffer 0, warp 2 for
//               the odd ones into buffer 1 (128x256 fp32 each), then commits
//               to the smem ring's "empty" barrier and to the buffer's "full"
//               barrier.
//   warp 3      idle (it completes warpgroup 0, which gives its registers
//               to the promotion warpgroups).
//   warps 4-11  promotion + epilogue: warp w reads TMEM lanes 32*(w%4)...,
//               warps 4-7 columns 0-127 and warps 8-11 columns 128-255 of the
//               partial, multiply-add it into 128 fp32 accumulators per
//               thread, release the buffer, and after the last block write
//               their part of the bf16 output tile.  With one B scale per
//               128x128 block (fwd, dgrad) a thread owns one row (32x32b
//               TMEM loads) and the warp's 32 x 128 output slice leaves
//               through its shared staging area by two TMA stores that
//               complete while the warp promotes the next tile; with one B
//               scale per column (wgrad) a thread owns 4 rows x 32 columns
//               (16x128b loads), which divides the broadcast reads of the
//               column scales by four.
// The MMA of block kb+1 runs while block kb is being promoted.
//
// Every wait is bounded (see mbar_wait): a lost arrival makes the kernel
// record a timeout in the device error word and unwind, freeing its TMEM.

#include "common.cuh"
#include "launch.h"
#include "quant_math.cuh"

namespace fp8bw {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;
constexpr int A_BYTES = BM * BK;
constexpr int B_BYTES = BN * BK;
constexpr int NUM_THREADS = 384;
constexpr int EPI_WARP0 = 4;
constexpr int NUM_EPI_WARPS = 8;
constexpr uint32_t TMEM_COLS = 512;  // two BN-column fp32 partial buffers
// Tile raster: group_m() row-blocks share a column sweep (one B scale per
// block: 32; per-column B scale: 16, each measured fastest).
template <int kBScale>
__host__ __device__ constexpr int group_m() {
  return kBScale == 0 ? 32 : 16;
}
constexpr int SB_STRIDE = 36;        // floats per lane-quarter row of the staged column scales
constexpr int EPI_BOX_ROWS = 16;     // output staging box: 16 rows x 64 bf16 columns (128 B rows)
constexpr int EPI_BOX_COLS = 64;
constexpr int EPI_BOX_BYTES = EPI_BOX_ROWS * EPI_BOX_COLS * 2;
// Register split.  Each SM sub-partition holds one warp of every warpgroup and
// 16384 registers, so a 384-thread CTA launches with 168 per thread; warpgroup
// 0 (producer, MMA, TMEM owner) then gives up registers to warpgroups 1-2
// (promotion): 88 + 2 * 208 = 56 + 2 * 224 = 3 * 168.
// The per-column-scale variant holds four more live values per column pair,
// so it takes a larger share.
template <int kBScale>
struct RegSplit {
  static constexpr uint32_t ctrl = kBScale == 0 ? 88 : 56;
  static constexpr uint32_t epi = kBScale == 0 ? 208 : 224;
  static_assert(ctrl + 2 * epi <= 3 * 168, "register split exceeds the launch budget");
};

template <int kBScale>
struct SharedStorageT {
  // fwd/dgrad: 3 stages and an 8 KB output staging area per promotion warp
  // (its 32 rows x 128 columns as two 32 x 64 boxes for TMA stores);
  // wgrad: 4 stages and one 16 x 64 box (2 KB) per warp.
  static constexpr int S = kBScale == 0 ? 3 : 4;
  static constexpr int EPI = kBScale == 0 ? 8192 : EPI_BOX_BYTES;
  uint8_t a[S][A_BYTES];  // each stage 1024-byte aligned (swizzle atom)
  uint8_t b[S][B_BYTES];
  uint8_t epi[NUM_EPI_WARPS][EPI];
  // Per-column B scales of the current and next block (per-column-scale
  // kernel only), private to each promotion warp: [warp][buffer][SB_STRIDE * q + i]
  // holds column 4 * i + q of the warp's 128 (q = lane % 4), so a thread's 32
  // scales are contiguous and the four lane classes' 16-byte loads hit
  // distinct banks.
  float sb_vec[NUM_EPI_WARPS][2][4 * SB_STRIDE];
  uint64_t full[S];
  uint64_t empty[S];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t mma_drain[2];       // used only when unwinding after a timeout
  // Output quantization in the epilogue (one-scale-per-block kernel): per
  // tile half, the four warps have staged their bf16 rows / have finished
  // reading the other warps' rows.
  uint64_t epi_staged[2];
  uint64_t epi_read[2];
  uint32_t tmem_base;
  int abort_flag;
};

template <int kBScale>
constexpr size_t smem_bytes() {
  return sizeof(SharedStorageT<kBScale>) + 1024;
}

// TMA bulk tensor store of a box from shared memory (128-byte swizzle) and
// the bulk async-group bookkeeping around it.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t c0, int32_t c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(map), "r"(src),
               "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void sts_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

template <int kGroupM>
__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int& mb, int& nb) {
  const int group_size = kGroupM * num_n;
  const int g = tile / group_size;
  const int first_m = g * kGroupM;
  const int gm = min(num_m - first_m, kGroupM);
  const int t = tile - g * group_size;
  mb = first_m + t % gm;
  nb = t / gm;
}

// Explicit shared-memory accesses (a generic pointer into the dynamic
// shared block would compile to generic loads with global-memory latency).
__device__ __forceinline__ float4 lds_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts_f32(uint32_t addr, float a) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(a) : "memory");
}

// Byte offset of 16-byte chunk k (0..7) of row r in a box of 128-byte rows
// written for a 128-byte-swizzled TMA map: chunk k of row r sits at chunk
// k ^ (r % 8), which also spreads a warp's writes over all banks.
__device__ __forceinline__ uint32_t sw128_offset(int r, int k) {
  return static_cast<uint32_t>(r * 128 + ((k ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// Writes a staged 16-row x 64-column bf16 box (rows of 128 bytes, chunk k of
// row r at chunk k ^ (r % 8)) to out[row0 + r][col0 + c]: each warp store
// covers four whole 128-byte row segments.
__device__ __forceinline__ void store_box(uint32_t stage, uint16_t* __restrict__ out, int64_t ld, int64_t row0,
                                          int64_t col0, int lane) {
  const int k = lane & 7;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 4 * i + (lane >> 3);
    const uint4 v = lds_v4(stage + sw128_offset(r, k));
    uint16_t* p = out + (row0 + r) * ld + col0 + 8 * k;
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
  }
}

__device__ __forceinline__ void sts_u16(uint32_t addr, uint16_t a) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(a) : "memory");
}
__device__ __forceinline__ uint16_t bf16_bits(float x) { return static_cast<uint16_t>(pack_bf16x2(x, 0.0f) & 0xFFFFu); }
// Contraction split of the last round of wgrad tiles.  The first full_units
// work units are whole tiles; the remaining tiles (when the tile count is not
// a multiple of the grid) are each cut into k contraction ranges, so the last
// rounds keep every SM busy.  The part of a split tile that finishes last
// (per promotion warp, counted in cnt) sums the k fp32 partials in part order
// from the caller's workspace and writes the output.  k = 1: no split.
struct SplitK {
  int full_units;
  int k;
  float2* ws;  // [tail tile][part][64][256] float2, thread-major: element j of thread t at j * 256 + t
  int* cnt;    // [tail tile][8 promotion warps], zero before the launch, back to zero after it
};

struct Unit {
  int tile, kb0, kb1;
  int part;    // -1 for a whole tile
  int t_idx;   // tail-tile index of a split unit
};

__device__ __forceinline__ Unit unit_of(int u, const SplitK& sp, int num_k) {
  Unit U;
  if (u < sp.full_units) {
    U.tile = u;
    U.kb0 = 0;
    U.kb1 = num_k;
    U.part = -1;
    U.t_idx = 0;
  } else {
    const int t = u - sp.full_units;
    U.t_idx = t / sp.k;
    U.part = t - U.t_idx * sp.k;
    U.tile = sp.full_units + U.t_idx;
    U.kb0 = U.part * num_k / sp.k;
    U.kb1 = (U.part + 1) * num_k / sp.k;
  }
  return U;
}

// Promotion with a per-column B scale (wgrad: both operands in 1x128 blocks
// along the contraction), out[i, j] = sum_kb sa[kb][i] * sb[kb][j] * P_kb[i, j].
// Every column of a block has its own scale, which every row needs.  Reading
// the partial with the 16x128b TMEM shape gives each thread 4 rows x 32
// columns (one column of every 4), so it needs 32 of the 128 column scales,
// staged per warp so that a thread's 32 are contiguous (8 conflict-free
// 16-byte shared loads per thread per block).  The two rows of a load that
// share a column are folded in as one packed pair.
template <bool kSplit>
__device__ __forceinline__ void promote_per_column(SharedStorageT<1>& sm, uint32_t tmem, int ew, int half, int quarter,
                                                   int lane, int num_units, int num_m, int num_n, int num_k,
                                                   const float* __restrict__ sa, int64_t sa_ld,
                                                   const float* __restrict__ sb, int64_t sb_ld_kb,
                                                   uint16_t* __restrict__ out, float* __restrict__ out_acc, int No,
                                                   const SplitK& sp, int* status, AbortFlag ab) {
  const int q4 = lane & 3, r8 = lane >> 2;
  int buf = 0;
  uint32_t tphase = 0;
  bool alive = true;
  for (int u = blockIdx.x; u < num_units && alive; u += gridDim.x) {
    const Unit U = kSplit ? unit_of(u, sp, num_k) : Unit{u, 0, num_k, -1, 0};
    int mb, nb;
    tile_coords<group_m<1>()>(U.tile, num_m, num_n, mb, nb);
    const int64_t rbase = static_cast<int64_t>(mb) * BM + quarter * 32 + r8;  // rows rbase + 16h + 8e
    const int64_t col0 = static_cast<int64_t>(nb) * BN + half * 128;
    float2 acc[64];  // column 32cq + 4j + q4, rows 16h + r8 (x) and 16h + r8 + 8 (y): acc[(h * 4 + cq) * 8 + j]
#pragma unroll
    for (int j = 0; j < 64; ++j) acc[j] = make_float2(0.0f, 0.0f);

    // Scales of the next block are fetched one block ahead; each lane fetches
    // four consecutive column scales of the warp's 128 (one coalesced 512-byte
    // row per warp) and stages them in the warp's own shared buffer, and the
    // A scale of one of the warp's 32 rows, which shuffles hand to the four
    // threads holding that row (one global load per lane instead of four).
    float sa_lane = __ldg(sa + static_cast<int64_t>(U.kb0) * sa_ld + (rbase - r8) + lane);
    float4 sb4_next = __ldg(reinterpret_cast<const float4*>(sb + static_cast<int64_t>(U.kb0) * sb_ld_kb + col0) + lane);
    for (int kb = U.kb0; kb < U.kb1; ++kb) {
      float sa_cur[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) sa_cur[i] = __shfl_sync(0xffffffffu, sa_lane, r8 + 16 * (i >> 1) + 8 * (i & 1));
      {
        // Lane L holds columns 4L .. 4L + 3 = 32cq + 4j + e with cq * 8 + j = L.
        // The buffer written now was last read two blocks ago; every lane
        // finished those reads before the previous block's __syncwarp.
        const uint32_t dst = smem_u32(sm.sb_vec[ew][kb & 1] + lane);
        sts_f32(dst, sb4_next.x);
        sts_f32(dst + 4 * SB_STRIDE, sb4_next.y);
        sts_f32(dst + 8 * SB_STRIDE, sb4_next.z);
        sts_f32(dst + 12 * SB_STRIDE, sb4_next.w);
      }
      __syncwarp();
      if (kb + 1 < U.kb1) {
        const float* sak = sa + static_cast<int64_t>(kb + 1) * sa_ld;
        sa_lane = __ldg(sak + (rbase - r8) + lane);
        sb4_next = __ldg(reinterpret_cast<const float4*>(sb + static_cast<int64_t>(kb + 1) * sb_ld_kb + col0) + lane);
      }
      if (!mbar_wait(&sm.tmem_full[buf], tphase, ab, status)) {
        alive = false;
        break;
      }
      tc_fence_after();
      const uint32_t t_col = tmem + static_cast<uint32_t>(buf * BN + half * 128);
      const uint32_t sbv = smem_u32(sm.sb_vec[ew][kb & 1] + q4 * SB_STRIDE);
      const float2 fa[2] = {make_float2(sa_cur[0], sa_cur[1]), make_float2(sa_cur[2], sa_cur[3])};
      // One load/wait round per column quarter cq (columns 32cq .. 32cq + 31)
      // for both 16-lane halves h of the warp's 32 TMEM lanes; the quarter's
      // scales serve both halves.  Wider rounds, or the next round's loads
      // issued before this round's products, measured no faster: the
      // partial's TMEM reads, which share TMEM with the MMAs, set the pace.
#pragma unroll
      for (int cq = 0; cq < 4; ++cq) {
        const float4 s0 = lds_f32x4(sbv + 32 * cq);
        const float4 s1 = lds_f32x4(sbv + 32 * cq + 16);
        const float sc[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
        uint32_t r[2][16];
#pragma unroll
        for (int h = 0; h < 2; ++h)
          tmem_ld_16x128b_x8(t_col + (static_cast<uint32_t>(quarter * 32 + 16 * h) << 16) + cq * 32, r[h]);
        tmem_ld_wait();
        if (cq == 3) {
          // The whole partial is in registers: the buffer goes back to the MMA warp.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.tmem_empty[buf]);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float2 p = make_float2(__uint_as_float(r[h][2 * j]), __uint_as_float(r[h][2 * j + 1]));
            float2& a = acc[(h * 4 + cq) * 8 + j];
            a = __ffma2_rn(__fmul2_rn(p, make_float2(sc[j], sc[j])), fa[h], a);
          }
        }
      }
      if (++buf == 2) {
        buf = 0;
        tphase ^= 1u;
      }
    }
    if (!alive) break;
    if (kSplit && U.part >= 0) {
      // A split tile: hand this part's fp32 partial over through the
      // workspace; the warp whose part arrives last for its 32 x 128 region
      // sums all k partials in part order (the same bits whichever part is
      // last) and stores the region.
      const int t = ew * 32 + lane;
      float2* slot = sp.ws + static_cast<int64_t>(U.t_idx * sp.k + U.part) * (64 * 256) + t;
#pragma unroll
      for (int j = 0; j < 64; ++j) slot[j * 256] = acc[j];
      __threadfence();
      __syncwarp();
      int arrived = 0;
      if (lane == 0) arrived = atomicAdd(&sp.cnt[U.t_idx * NUM_EPI_WARPS + ew], 1);
      arrived = __shfl_sync(0xffffffffu, arrived, 0);
      if (arrived != sp.k - 1) continue;
      __threadfence();
      const float2* first = sp.ws + static_cast<int64_t>(U.t_idx * sp.k) * (64 * 256) + t;
#pragma unroll
      for (int j = 0; j < 64; ++j) acc[j] = __ldcg(first + j * 256);
      for (int p = 1; p < sp.k; ++p) {
        const float2* part = first + static_cast<int64_t>(p) * (64 * 256);
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const float2 v = __ldcg(part + j * 256);
          acc[j] = make_float2(acc[j].x + v.x, acc[j].y + v.y);
        }
      }
      if (lane == 0) sp.cnt[U.t_idx * NUM_EPI_WARPS + ew] = 0;  // ready for the next call
      __syncwarp();
    }
    if (out_acc != nullptr) {
      // Gradient accumulation: add the tile to the caller's fp32 dW.
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float* row0 = out_acc + (rbase + 16 * h) * No + col0 + q4;
        float* row1 = row0 + 8 * static_cast<int64_t>(No);
#pragma unroll
        for (int cq = 0; cq < 4; ++cq) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float2 v = acc[(h * 4 + cq) * 8 + j];
            row0[32 * cq + 4 * j] += v.x;
            row1[32 * cq + 4 * j] += v.y;
          }
        }
      }
    } else {
      // Four 16-row x 64-column boxes per warp (lane half h, column half cc),
      // staged through the warp's swizzled buffer for whole-line stores.
      const uint32_t stage = smem_u32(sm.epi[ew]);
      const int64_t row0 = static_cast<int64_t>(mb) * BM + quarter * 32;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float2 v = acc[(h * 4 + 2 * cc + c2) * 8 + j];
              const int k8 = 4 * c2 + (j >> 1);
              const uint32_t off = 2 * (4 * (j & 1) + q4);
              sts_u16(stage + sw128_offset(r8, k8) + off, bf16_bits(v.x));
              sts_u16(stage + sw128_offset(r8 + 8, k8) + off, bf16_bits(v.y));
            }
          }
          __syncwarp();
          store_box(stage, out, No, row0 + h * 16, col0 + cc * EPI_BOX_COLS, lane);
          __syncwarp();
        }
      }
    }
  }
}

// Quantized copies of the bf16 output written by the epilogue (see
// BlockwiseGemmArgs::q_out).
struct QuantOut {
  uint8_t* q;
  float* s;
  uint8_t* qT;
  float* sT;
};

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
// 32 bytes as two 16-byte stores (the caller's arrays are only guaranteed
// 16-byte alignment).
__device__ __forceinline__ void stg_2x16(void* p, const uint32_t (&w)[8]) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
               : "memory");
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(static_cast<uint8_t*>(p) + 16), "r"(w[4]),
               "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// kQuantOut (one-scale-per-block kernel only): 0 = bf16 output alone; 1 = also
// its 1x128 rowwise quantization; 2 = rowwise and colwise.  Both are the
// blockwise rule applied to the bf16-rounded output, bit-identical to running
// the stand-alone quantizers on it.
// kBmn (one-scale-per-block kernel only): 1 = operand B is given MN-major,
// b[k][n] over [Kc, No] (the dgrad weight read from its row-major codes),
// loaded as two 128-column boxes and fed to the MMA with "transpose B".
// kSplit (per-column-scale kernel only): the work-unit loop with the
// contraction split of the last round (SplitK); without it the loops run over
// whole tiles, as compiled before the split existed (the unit loop costs a few
// per cent even when nothing is split).
template <int kBScale, int kQuantOut, int kBmn, bool kSplit = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    blockwise_gemm_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                          const __grid_constant__ CUtensorMap tma_out,
                          const float* __restrict__ sa, int64_t sa_ld, const float* __restrict__ sb, int64_t sb_ld_nb,
                          int64_t sb_ld_kb, uint16_t* __restrict__ out, float* __restrict__ out_acc, QuantOut qo,
                          SplitK sp, int Mo, int No, int Kc, int* status) {
  static_assert(kQuantOut == 0 || kBScale == 0, "output quantization is implemented for the fwd/dgrad kernel");
  static_assert(kBmn == 0 || kBScale == 0, "an MN-major B is implemented for the fwd/dgrad kernel");
  extern __shared__ uint8_t smem_raw[];
  using Storage = SharedStorageT<kBScale>;
  constexpr int STAGES = Storage::S;
  Storage& sm =
      *reinterpret_cast<Storage*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_m = Mo / BM, num_n = No / BN, num_k = Kc / BK;
  const int num_tiles = num_m * num_n;
  // Work units: whole tiles, then the contraction parts of the split tail
  // (the per-column-scale kernel only; sp.k = 1 leaves num_units = num_tiles).
  static_assert(!kSplit || kBScale == 1, "the contraction split is implemented for the wgrad kernel");
  const int num_units = kSplit ? sp.full_units + (num_tiles - sp.full_units) * sp.k : num_tiles;
  const AbortFlag ab{&sm.abort_flag};

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.tmem_full[b], 1);
      mbar_init(&sm.tmem_empty[b], NUM_EPI_WARPS);
    }
    mbar_init(&sm.mma_drain[0], 1);
    mbar_init(&sm.mma_drain[1], 1);
    for (int h = 0; h < 2; ++h) {
      mbar_init(&sm.epi_staged[h], 4);
      mbar_init(&sm.epi_read[h], 4);
    }
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tma_a);
    tma_prefetch_desc(&tma_b);
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp < EPI_WARP0) {
    regs_dec<RegSplit<kBScale>::ctrl>();
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;  // loads issued so far
      bool alive = true;
      for (int u = blockIdx.x; u < num_units && alive; u += gridDim.x) {
        const Unit U = kSplit ? unit_of(u, sp, num_k) : Unit{u, 0, num_k, -1, 0};
        int mb, nb;
        tile_coords<group_m<kBScale>()>(U.tile, num_m, num_n, mb, nb);
        for (int kb = U.kb0; kb < U.kb1; ++kb) {
          if (!mbar_wait(&sm.empty[stage], phase ^ 1u, ab, status)) {
            alive = false;
            break;
          }
          mbar_arrive_expect_tx(&sm.full[stage], A_BYTES + B_BYTES);
          tma_load_2d(sm.a[stage], &tma_a, &sm.full[stage], kb * BK, mb * BM);
          if constexpr (kBmn) {
            // B[k][n]: two boxes of 128 contraction rows x 128 columns.
            tma_load_2d(sm.b[stage], &tma_b, &sm.full[stage], nb * BN, kb * BK);
            tma_load_2d(sm.b[stage] + B_BYTES / 2, &tma_b, &sm.full[stage], nb * BN + 128, kb * BK);
          } else {
            tma_load_2d(sm.b[stage], &tma_b, &sm.full[stage], kb * BK, nb * BN);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!alive) {
        // Unwinding: only the last STAGES loads can still be in flight (each
        // earlier one was consumed before its stage was refilled).  Let them
        // land before the CTA's shared memory is released.
        uint32_t n = issued < STAGES ? issued : STAGES;
        int s = stage;
        uint32_t p = phase;
        for (uint32_t i = 0; i < n; ++i) {
          if (--s < 0) {
            s = STAGES - 1;
            p ^= 1u;
          }
          int dummy = 0;
          mbar_wait(&sm.full[s], p, AbortFlag{&dummy}, status, 1000000ull);
        }
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // Two issuing threads: warp 1 issues the even contraction blocks (into
    // TMEM buffer 0), warp 2 the odd ones (buffer 1), so the MMAs of block
    // g + 2 go out as soon as the promotion hands buffer g % 2 back, even
    // while the other issuer is still feeding block g + 1 to the tensor core.
    if (lane == 0) {
      constexpr uint32_t idesc = kBmn ? idesc_e4m3_f32_bmn(BM, BN) : idesc_e4m3_f32(BM, BN);
      // Start-address step of one 32-deep MMA along B: 32 bytes K-major, 32
      // rows of 128 bytes MN-major (16-byte units).
      constexpr uint64_t kBStep = kBmn ? (32 * 128) >> 4 : 32 >> 4;
      const int me = warp - 1;
      const uint32_t d_tmem = tmem + static_cast<uint32_t>(me * BN);
      // Descriptors of stage 0; stage s and the 32-byte K step k are plain
      // adds to the start-address field (in 16-byte units).
      const uint64_t a_desc0 = sdesc_kmajor_sw128(smem_u32(sm.a[0]));
      const uint64_t b_desc0 = kBmn ? sdesc_mnmajor_sw128(smem_u32(sm.b[0]), B_BYTES / 2)
                                    : sdesc_kmajor_sw128(smem_u32(sm.b[0]));
      bool alive = true;
      uint32_t g = 0;  // running block index over this CTA's tiles
      for (int u = blockIdx.x; u < num_units && alive; u += gridDim.x) {
        const Unit U = kSplit ? unit_of(u, sp, num_k) : Unit{u, 0, num_k, -1, 0};
        for (int kb = U.kb0; kb < U.kb1; ++kb, ++g) {
          if ((g & 1u) != static_cast<uint32_t>(me)) continue;
          const int stage = static_cast<int>(g % STAGES);
          const uint32_t phase = (g / STAGES) & 1u;
          const uint32_t tphase = (g >> 1) & 1u;
          if (!mbar_wait(&sm.tmem_empty[me], tphase ^ 1u, ab, status) ||
              !mbar_wait(&sm.full[stage], phase, ab, status)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = a_desc0 + static_cast<uint64_t>(stage * (A_BYTES >> 4));
          const uint64_t bd = b_desc0 + static_cast<uint64_t>(stage * (B_BYTES >> 4));
          mma_e4m3_k<false>(d_tmem, ad, bd, idesc);
          mma_e4m3_k<true>(d_tmem, ad + 2, bd + kBStep, idesc);
          mma_e4m3_k<true>(d_tmem, ad + 4, bd + 2 * kBStep, idesc);
          mma_e4m3_k<true>(d_tmem, ad + 6, bd + 3 * kBStep, idesc);
          mma_commit(&sm.empty[stage]);
          mma_commit(&sm.tmem_full[me]);
        }
      }
      if (!alive) {
        // Unwinding: wait for this thread's MMAs already issued before TMEM is freed.
        mma_commit(&sm.mma_drain[me]);
        int dummy = 0;
        mbar_wait(&sm.mma_drain[me], 0, AbortFlag{&dummy}, status, 1000000ull);
      }
    }
  }
  } else {
    regs_inc<RegSplit<kBScale>::epi>();
    // ------------------------------------------------------------ promotion + epilogue
    const int ew = warp - EPI_WARP0;
    const int half = ew >> 2;                  // column half of the tile
    const int quarter = warp & 3;              // TMEM lane quarter this warp may access
    if constexpr (kBScale == 1) {
      promote_per_column<kSplit>(sm, tmem, ew, half, quarter, lane, num_units, num_m, num_n, num_k, sa, sa_ld, sb, sb_ld_kb,
                         out, out_acc, No, sp, status, ab);
    } else {
      const int row = quarter * 32 + lane;       // row of the tile this thread owns
      const uint32_t t_lane = static_cast<uint32_t>(quarter * 32) << 16;
      uint32_t tile_i = 0;                       // tiles finished by this warp (epilogue barrier phases)
      int buf = 0;
      uint32_t tphase = 0;
      bool alive = true;
      for (int tile = blockIdx.x; tile < num_tiles && alive; tile += gridDim.x) {
        int mb, nb;
        tile_coords<group_m<kBScale>()>(tile, num_m, num_n, mb, nb);
        const int64_t m = static_cast<int64_t>(mb) * BM + row;
        const int64_t col0 = static_cast<int64_t>(nb) * BN + half * 128;
        float2 acc[64];
#pragma unroll
        for (int j = 0; j < 64; ++j) acc[j] = make_float2(0.0f, 0.0f);

        // Scales of the next block are fetched one block ahead: the row's A
        // scale and the tile half's B block scale.
        float sa_next = __ldg(sa + m);
        float sb_next = __ldg(sb + (col0 / 128) * sb_ld_nb);
        for (int kb = 0; kb < num_k; ++kb) {
          const float sa_cur = sa_next;
          const float sb_cur = sb_next;
          if (kb + 1 < num_k) {
            sa_next = __ldg(sa + static_cast<int64_t>(kb + 1) * sa_ld + m);
            sb_next = __ldg(sb + (col0 / 128) * sb_ld_nb + static_cast<int64_t>(kb + 1) * sb_ld_kb);
          }
          if (!mbar_wait(&sm.tmem_full[buf], tphase, ab, status)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint32_t t_base = tmem + t_lane + static_cast<uint32_t>(buf * BN + half * 128);
          // 16-column TMEM loads, one per wait (eight load/wait rounds per
          // block measured fastest: with 2 or 4 loads per wait the promotion
          // warps take more of the TMEM read bandwidth the MMAs share and all
          // three GEMMs slow down by a fifth).  The buffer goes back to the
          // MMA warp as soon as the last load has landed in registers.
          constexpr int NC = 1;
          constexpr int NG = 8 / NC;
          const float2 f2 = make_float2(sa_cur * sb_cur, sa_cur * sb_cur);
#pragma unroll
          for (int g = 0; g < NG; ++g) {
            uint32_t r[NC][16];
#pragma unroll
            for (int c = 0; c < NC; ++c) tmem_ld_32x32b_x16(t_base + (g * NC + c) * 16, r[c]);
            tmem_ld_wait();
            if (g == NG - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&sm.tmem_empty[buf]);
            }
#pragma unroll
            for (int c = 0; c < NC; ++c) {
              const int col = (g * NC + c) * 16;
#pragma unroll
              for (int j = 0; j < 8; j += 2) {
                const float2 p0 = make_float2(__uint_as_float(r[c][2 * j]), __uint_as_float(r[c][2 * j + 1]));
                const float2 p1 = make_float2(__uint_as_float(r[c][2 * j + 2]), __uint_as_float(r[c][2 * j + 3]));
                float2& a0 = acc[(col >> 1) + j];
                float2& a1 = acc[(col >> 1) + j + 1];
                a0 = __ffma2_rn(p0, f2, a0);
                a1 = __ffma2_rn(p1, f2, a1);
              }
            }
          }
          if (++buf == 2) {
            buf = 0;
            tphase ^= 1u;
          }
        }
        if (!alive) break;
        // Output: the warp's 32 rows x 128 columns go through its staging
        // area (two 32 x 64 boxes, 128-byte swizzle) to two TMA stores, which
        // complete while the warp promotes the next tile.
        const uint32_t stage = smem_u32(sm.epi[ew]);
        if constexpr (kQuantOut == 2) {
          // The other three warps of this half have read the previous tile's rows.
          if (tile_i > 0 && !mbar_wait(&sm.epi_read[half], (tile_i - 1) & 1u, ab, status)) break;
        }
        if (lane == 0) bulk_wait_read_all();  // the previous tile's stores have read the area
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int j = 4 * c;
          sts_v4(stage + (c >> 3) * 4096 + sw128_offset(lane, c & 7), pack_bf16x2(acc[j].x, acc[j].y),
                 pack_bf16x2(acc[j + 1].x, acc[j + 1].y), pack_bf16x2(acc[j + 2].x, acc[j + 2].y),
                 pack_bf16x2(acc[j + 3].x, acc[j + 3].y));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int32_t r0 = mb * BM + quarter * 32;
          tma_store_2d(&tma_out, stage, static_cast<int32_t>(col0), r0);
          tma_store_2d(&tma_out, stage + 4096, static_cast<int32_t>(col0) + 64, r0);
          bulk_commit();
        }
        if constexpr (kQuantOut >= 1) {
          if constexpr (kQuantOut == 2) {
            if (lane == 0) mbar_arrive(&sm.epi_staged[half]);  // this warp's rows are staged
          }
          // 1x128 rowwise: the thread's row holds the whole block (the warp's
          // 128 columns of this tile half), in registers.
          float amax = 0.0f;
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const uint32_t pk = pack_bf16x2(acc[j].x, acc[j].y);
            amax = fmaxf(amax, fmaxf(fabsf(bf16lo_to_f32(pk)), fabsf(bf16hi_to_f32(pk))));
          }
          const float sc = blockwise_scale(amax);
          const float2 s2 = make_float2(sc, sc), ny2 = make_float2(neg_recip(sc), neg_recip(sc));
          uint8_t* qrow = qo.q + m * No + col0;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int j = c * 16 + i * 2;  // columns 4 (c * 8 + i) .. + 3
              const uint32_t p0 = pack_bf16x2(acc[j].x, acc[j].y), p1 = pack_bf16x2(acc[j + 1].x, acc[j + 1].y);
              w[i] = e4m3x4_from_neg(
                  neg_div_by_scale2(make_float2(bf16lo_to_f32(p0), bf16hi_to_f32(p0)), s2, ny2),
                  neg_div_by_scale2(make_float2(bf16lo_to_f32(p1), bf16hi_to_f32(p1)), s2, ny2));
            }
            stg_2x16(qrow + 32 * c, w);
          }
          qo.s[(col0 / 128) * Mo + m] = sc;
        }
        if constexpr (kQuantOut == 2) {
          // 1x128 colwise: the tile's 128 rows are one block of every column.
          // Thread (quarter q, lane l) takes column 32q + l of this half and
          // reads its 128 staged values from the four warps' areas (a warp's
          // 32 lanes read one 64-byte run of a staged row: conflict-free).
          if (!mbar_wait(&sm.epi_staged[half], tile_i & 1u, ab, status)) break;
          const int cc = quarter * 32 + lane;
          const uint32_t col_off = static_cast<uint32_t>((cc >> 6) * 4096 + (cc & 7) * 2);
          uint32_t v[64];  // rows 2i, 2i + 1 as a bf16 pair
          float amax = 0.0f;
#pragma unroll
          for (int rq = 0; rq < 4; ++rq) {
            const uint32_t base = smem_u32(sm.epi[half * 4 + rq]) + col_off;
#pragma unroll
            for (int r = 0; r < 32; r += 2) {
              const uint32_t lo = lds_u16(base + sw128_offset(r, (cc & 63) >> 3));
              const uint32_t hi = lds_u16(base + sw128_offset(r + 1, (cc & 63) >> 3));
              v[rq * 16 + r / 2] = lo | (hi << 16);
              amax = fmaxf(amax, fmaxf(fabsf(bf16lo_to_f32(lo)), fabsf(bf16lo_to_f32(hi))));
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.epi_read[half]);  // done with the other warps' rows
          const float sc = blockwise_scale(amax);
          const float2 s2 = make_float2(sc, sc), ny2 = make_float2(neg_recip(sc), neg_recip(sc));
          const int64_t col = col0 + cc;
          uint8_t* qcol = qo.qT + col * Mo + static_cast<int64_t>(mb) * BM;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int j = c * 16 + i * 2;  // rows 4 (c * 8 + i) .. + 3
              w[i] = e4m3x4_from_neg(
                  neg_div_by_scale2(make_float2(bf16lo_to_f32(v[j]), bf16hi_to_f32(v[j])), s2, ny2),
                  neg_div_by_scale2(make_float2(bf16lo_to_f32(v[j + 1]), bf16hi_to_f32(v[j + 1])), s2, ny2));
            }
            stg_2x16(qcol + 32 * c, w);
          }
          qo.sT[static_cast<int64_t>(mb) * No + col] = sc;
        }
        ++tile_i;
      }
      if (lane == 0) bulk_wait_all();  // this warp's stores are done before the CTA ends
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// 2D map over a row-major [rows, cols] uint8 matrix, box = box_rows x 128
// bytes, 128-byte swizzle.
bool encode_kmajor_u8(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, uint32_t box_rows) {
  auto fn = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
  cuuint32_t box[2] = {128u, box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// 2D map over the row-major [rows, cols] bf16 output, box 32 rows x 64
// columns (128 bytes), 128-byte swizzle.
bool encode_out_bf16(CUtensorMap* map, const void* base, int64_t rows, int64_t cols) {
  auto fn = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {64u, 32u};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The split is chosen by a cost model in units of one 128-deep block's time:
// the tail's rounds of parts, each part costing its blocks plus about kIo
// block-times of writing its 128 KB fp32 partial, and the last part reading
// the others'.  k is capped at 16 (the workspace grows with it).
WgradSplitPlan wgrad_split_plan(int64_t Mo, int64_t No, int64_t Kc, int num_sms) {
  const int num_tiles = static_cast<int>((Mo / BM) * (No / BN)), num_k = static_cast<int>(Kc / BK);
  WgradSplitPlan best{num_tiles, 0, 1, 0};
  if (num_sms <= 0 || num_tiles <= 0) return best;
  const int rounds = num_tiles / num_sms, tail = num_tiles - rounds * num_sms;
  if (tail == 0 || num_k < 2) return best;
  constexpr long kIo = 6;
  // The split kernel's work-unit loop runs a few per cent slower per block
  // than the whole-tile one, so a split must save more than that (3 %
  // charged: on the 16384-token dense shape a two-part split of the 64 tail
  // tiles, predicted 4.5 % faster without the charge, measured 1.4 %).
  const long whole = static_cast<long>(rounds + 1) * num_k;
  long best_cost = whole;
  for (int k = 2; k <= 16 && k <= num_k; ++k) {
    const long sub_rounds = (static_cast<long>(tail) * k + num_sms - 1) / num_sms;
    const long part = (num_k + k - 1) / k;
    const long cost = (static_cast<long>(rounds) * num_k + sub_rounds * (part + kIo) + kIo * (k - 1)) * 103 / 100;
    if (cost < best_cost) {
      best_cost = cost;
      best.k = k;
    }
  }
  if (best.k == 1) return best;
  best.full_units = rounds * num_sms;
  best.tail = tail;
  const size_t partials = static_cast<size_t>(tail) * best.k * BM * BN * sizeof(float);
  best.bytes = partials + static_cast<size_t>(tail) * NUM_EPI_WARPS * sizeof(int);
  return best;
}

cudaError_t launch_blockwise_gemm(const BlockwiseGemmArgs& g, cudaStream_t st) {
  CUtensorMap ta, tb, to;
  // B K-major: [No, Kc], boxes of BN rows x 128 bytes; MN-major: [Kc, No]
  // (row length No), boxes of 128 rows x 128 bytes.
  const bool b_ok = g.b_mn_major ? encode_kmajor_u8(&tb, g.b, g.Kc, g.No, 128)
                                 : encode_kmajor_u8(&tb, g.b, g.No, g.Kc, BN);
  if (!encode_kmajor_u8(&ta, g.a, g.Mo, g.Kc, BM) || !b_ok) return cudaErrorInvalidValue;
  if (g.b_scale == BScale::kBlock128x128 && !encode_out_bf16(&to, g.out, g.Mo, g.No)) return cudaErrorInvalidValue;
  if (g.b_scale != BScale::kBlock128x128) to = ta;  // unused by the per-column kernel
  const int num_tiles = static_cast<int>((g.Mo / BM) * (g.No / BN));
  int grid = num_tiles < g.num_sms ? num_tiles : g.num_sms;
  SplitK sp{num_tiles, 1, nullptr, nullptr};
  if (g.b_scale == BScale::kPerRow && g.out_acc == nullptr && g.split_ws != nullptr) {
    const WgradSplitPlan pl = wgrad_split_plan(g.Mo, g.No, g.Kc, g.num_sms);
    if (pl.k > 1) {
      if (g.split_ws_bytes < pl.bytes) return cudaErrorInvalidValue;
      uint8_t* ws = static_cast<uint8_t*>(g.split_ws);
      sp = SplitK{pl.full_units, pl.k, reinterpret_cast<float2*>(ws),
                  reinterpret_cast<int*>(ws + (pl.bytes - static_cast<size_t>(pl.tail) * NUM_EPI_WARPS * sizeof(int)))};
      const cudaError_t e = cudaMemsetAsync(sp.cnt, 0, static_cast<size_t>(pl.tail) * NUM_EPI_WARPS * sizeof(int), st);
      if (e != cudaSuccess) return e;
      const int units = pl.full_units + pl.tail * pl.k;
      grid = units < g.num_sms ? units : g.num_sms;
    }
  }
  const QuantOut qo{g.q_out, g.s_out, g.qT_out, g.sT_out};
  const int Mo = static_cast<int>(g.Mo), No = static_cast<int>(g.No), Kc = static_cast<int>(g.Kc);
  auto launch = [&](auto kernel, size_t smem) -> cudaError_t {
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    kernel<<<grid, NUM_THREADS, smem, st>>>(ta, tb, to, g.sa, g.sa_ld, g.sb, g.sb_ld_nb, g.sb_ld_kb, g.out, g.out_acc,
                                            qo, sp, Mo, No, Kc, g.status);
    return cudaGetLastError();
  };
  if (g.b_scale != BScale::kBlock128x128) {
    if (sp.k > 1) return launch(blockwise_gemm_kernel<1, 0, 0, true>, smem_bytes<1>());
    return launch(blockwise_gemm_kernel<1, 0, 0>, smem_bytes<1>());
  }
  if (g.b_mn_major) return launch(blockwise_gemm_kernel<0, 0, 1>, smem_bytes<0>());
  if (g.q_out == nullptr) return launch(blockwise_gemm_kernel<0, 0, 0>, smem_bytes<0>());
  if (g.qT_out == nullptr) return launch(blockwise_gemm_kernel<0, 1, 0>, smem_bytes<0>());
  return launch(blockwise_gemm_kernel<0, 2, 0>, smem_bytes<0>());
}

// ---------------------------------------------------------------- bounded-wait self-test

namespace {
__global__ void selftest_wait_kernel(uint64_t limit_ns, int* status) {
  __shared__ uint64_t bar;
  __shared__ int flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, AbortFlag{&flag}, status, limit_ns);  // nothing ever arrives
}
}  // namespace

cudaError_t launch_selftest_bounded_wait(uint32_t timeout_us, int* status, cudaStream_t st) {
  selftest_wait_kernel<<<1, 32, 0, st>>>(static_cast<uint64_t>(timeout_us) * 1000ull, status);
  return cudaGetLastError();
}

}  // namespace fp8bw
