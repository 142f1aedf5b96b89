// MXFP8 grouped GEMM for MoE (PR #3037, "[mxfp8 moe training] use new 3d
// colwise quantization kernel": Summary and Microbenchmarks table -- grouped
// mm forward and backward with MoEScalingType.MXFP8).
//
// Operands are e4m3 with one E8M0 scale per 32 contraction elements.  Those
// scales are exact powers of two, so the tensor core applies them itself:
// tcgen05.mma kind::mxf8f6f4.block_scale reads A/B tiles from shared memory
// and their scale factors from tensor memory, and accumulates the whole
// contraction in a 128x256 fp32 TMEM tile -- no promotion on CUDA cores.
//
// Kinds (dims of the MoE linear: M tokens in G groups, K in, N out features):
//   FWD   : out[M, N]  rows of group g = A_g[., K] * W_g^T      (2D x 3D)
//   DGRAD : out[M, K]  rows of group g = dY_g[., N] * W_g        (2D x 3D)
//   WGRAD : out[G, N, K] = dY_g^T X_g over the tokens of group g (2D x 2D)
// FWD/DGRAD tiles are 128-token slices of one group; rows past the group's
// end are computed with the wrong expert and never stored.  WGRAD tiles
// contract over the group's token range in 128-wide steps, issuing only the
// 32-wide MMAs that lie inside the group (group sizes are multiples of 32).
//
// CTA (persistent, 384 threads):
//   warp 0      TMA producer (A 128x128, B 256x128 e4m3 per stage)
//   warp 1      TMEM owner and MMA issuer: per stage, tcgen05.cp of the
//               stage's scale factors into TMEM, then up to 4 block-scaled
//               MMAs (K = 32 each, scale byte j of each row's word selected
//               by the instruction descriptor)
//   warp 2      scale-factor gatherer: per stage, each operand row's 4 E8M0
//               bytes into the 32-row x 16-byte interleaved layout tcgen05.cp
//               consumes (row r -> 32-bit word (r % 32) * 4 + r / 32 of its
//               128-row chunk)
//   warp 3      idle
//   warps 4-11  epilogue: drain the accumulator (warp w: lanes 32*(w%4).., one
//               128-column half), release it, write bf16 rows.
#include "common.cuh"
#include "launch.h"

namespace fp8bw {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK;
constexpr int B_BYTES = BN * BK;
constexpr int NUM_THREADS = 384;
constexpr int EPI_WARP0 = 4;
constexpr int NUM_EPI_WARPS = 8;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COL = 0;        // accumulator: columns [0, 256)
constexpr uint32_t SF_COL0 = 256;      // per stage: SFA 4 columns, SFB 8 columns, in 16-column slots
constexpr int GROUP_M = 16;
constexpr int MAX_GROUPS = 1024;

struct SharedStorage {
  uint8_t a[STAGES][A_BYTES];
  uint8_t b[STAGES][B_BYTES];
  uint32_t sfa[STAGES][BM];
  uint32_t sfb[STAGES][BN];
  int32_t g_start[MAX_GROUPS + 1];   // token start of each group (clamped)
  int32_t g_tile0[MAX_GROUPS + 1];   // FWD/DGRAD: first 128-row tile of each group
  uint64_t full[STAGES];
  uint64_t sf_full[STAGES];
  uint64_t empty[STAGES];
  uint64_t acc_full;
  uint64_t acc_empty;
  uint64_t mma_drain;
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t kSmemBytes = sizeof(SharedStorage) + 1024;

struct Tile {
  int g;          // group
  int a_row0;     // first row of A
  int b_row0;     // first row of B
  int k_begin;    // contraction range
  int k_end;
  int out_row0;   // first output row (FWD/DGRAD: token; WGRAD: row within dW_g)
  int row_limit;  // output rows >= row_limit are not stored (FWD/DGRAD)
  int out_col0;
};

struct Problem {
  int kind, G, M, N, K;
  int n_out;      // output columns
  int kc;         // FWD/DGRAD contraction length
  int num_mt;     // FWD/DGRAD: 128-row tiles over all groups
  int num_nt;     // output column tiles (256 wide)
  int num_tiles;
};

__device__ __forceinline__ void raster(int t, int num_m, int num_n, int& mt, int& nt) {
  const int group_size = GROUP_M * num_n;
  const int gi = t / group_size;
  const int first = gi * GROUP_M;
  const int gm = min(num_m - first, GROUP_M);
  const int r = t - gi * group_size;
  mt = first + r % gm;
  nt = r / gm;
}

__device__ __forceinline__ Tile decode(const SharedStorage& sm, const Problem& p, int t) {
  Tile T;
  if (p.kind != 2) {
    int mt, nt;
    raster(t, p.num_mt, p.num_nt, mt, nt);
    int g = 0;
    while (g + 1 < p.G && sm.g_tile0[g + 1] <= mt) ++g;
    const int m0 = sm.g_start[g] + (mt - sm.g_tile0[g]) * BM;
    T.g = g;
    T.a_row0 = m0;
    T.b_row0 = g * p.n_out + nt * BN;
    T.k_begin = 0;
    T.k_end = p.kc;
    T.out_row0 = m0;
    T.row_limit = sm.g_start[g + 1];
    T.out_col0 = nt * BN;
  } else {
    const int per_group = (p.N / BM) * p.num_nt;
    const int g = t / per_group;
    int mt, nt;
    raster(t - g * per_group, p.N / BM, p.num_nt, mt, nt);
    T.g = g;
    T.a_row0 = mt * BM;
    T.b_row0 = nt * BN;
    T.k_begin = sm.g_start[g];
    T.k_end = sm.g_start[g + 1];
    T.out_row0 = mt * BM;
    T.row_limit = p.N;
    T.out_col0 = nt * BN;
  }
  return T;
}

__device__ __forceinline__ int num_kb(const Tile& T) { return (T.k_end - T.k_begin + BK - 1) / BK; }

__device__ __forceinline__ uint32_t ld_u32(const uint8_t* p) {
  return __ldg(reinterpret_cast<const unsigned int*>(p));
}

// The 4 scale bytes of one operand row for contraction elements [k0, k0+128):
// byte j = scale of chunk j; chunks at or past k_end read as 0.
__device__ __forceinline__ uint32_t row_sf(const uint8_t* e8, int64_t row, int64_t row_bytes, int k0, int k_end,
                                           bool aligned) {
  const uint8_t* p = e8 + row * row_bytes + k0 / 32;
  if (aligned && k0 + BK <= k_end) return ld_u32(p);
  uint32_t w = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (k0 + 32 * j < k_end) w |= static_cast<uint32_t>(__ldg(p + j)) << (8 * j);
  return w;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    mx_grouped_gemm_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                           const uint8_t* __restrict__ a_e8, const uint8_t* __restrict__ b_e8,
                           const int32_t* __restrict__ group_end, uint16_t* __restrict__ out, Problem p,
                           int64_t a_rows, int64_t b_rows, int* status) {
  extern __shared__ uint8_t smem_raw[];
  SharedStorage& sm =
      *reinterpret_cast<SharedStorage*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const AbortFlag ab{&sm.abort_flag};

  if (threadIdx.x == 0) {
    // Group table: clamp every range into [0, M] and round each end down to
    // a multiple of 32 (so every TMA coordinate along tokens stays 32-byte
    // aligned whatever group_end holds); flag sizes that are not multiples
    // of 32, decreasing ends, or a last end other than M.
    int prev = 0, tile0 = 0;
    bool bad = false;
    for (int g = 0; g < p.G; ++g) {
      int e = group_end[g];
      if (e < prev || e > p.M || ((e - prev) & 31) != 0) bad = true;
      e = min(max(e, prev), p.M) & ~31;
      e = max(e, prev);
      sm.g_start[g] = prev;
      sm.g_tile0[g] = tile0;
      tile0 += (e - prev + BM - 1) / BM;
      prev = e;
    }
    if (prev != p.M) bad = true;
    sm.g_start[p.G] = prev;
    sm.g_tile0[p.G] = tile0;
    if (bad && blockIdx.x == 0) atomicExch(status, kStatusShape);
    p.num_mt = tile0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.sf_full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    mbar_init(&sm.acc_full, 1);
    mbar_init(&sm.acc_empty, NUM_EPI_WARPS);
    mbar_init(&sm.mma_drain, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
    sm.g_tile0[MAX_GROUPS] = tile0;  // total 128-row tiles, read back by every thread below
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
  if (p.kind != 2) {
    p.num_mt = sm.g_tile0[MAX_GROUPS];
    p.num_tiles = p.num_mt * p.num_nt;
  }
  const bool sf_aligned = p.kind != 2;  // FWD/DGRAD blocks start at multiples of 128

  if (warp < EPI_WARP0) {
    regs_dec<88>();
    if (warp == 0) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        int stage = 0;
        uint32_t phase = 0, issued = 0;
        bool alive = true;
        for (int t = blockIdx.x; t < p.num_tiles && alive; t += gridDim.x) {
          const Tile T = decode(sm, p, t);
          const int nkb = num_kb(T);
          for (int kb = 0; kb < nkb; ++kb) {
            if (!mbar_wait(&sm.empty[stage], phase ^ 1u, ab, status)) {
              alive = false;
              break;
            }
            const int k0 = T.k_begin + kb * BK;
            mbar_arrive_expect_tx(&sm.full[stage], A_BYTES + B_BYTES);
            tma_load_2d(sm.a[stage], &tma_a, &sm.full[stage], k0, T.a_row0);
            tma_load_2d(sm.b[stage], &tma_b, &sm.full[stage], k0, T.b_row0);
            ++issued;
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (!alive) {
          uint32_t n = issued < STAGES ? issued : STAGES;
          int s = stage;
          uint32_t ph = phase;
          for (uint32_t i = 0; i < n; ++i) {
            if (--s < 0) {
              s = STAGES - 1;
              ph ^= 1u;
            }
            int dummy = 0;
            mbar_wait(&sm.full[s], ph, AbortFlag{&dummy}, status, 1000000ull);
          }
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        int stage = 0;
        uint32_t phase = 0, aphase = 0;
        bool alive = true;
        for (int t = blockIdx.x; t < p.num_tiles && alive; t += gridDim.x) {
          const Tile T = decode(sm, p, t);
          const int nkb = num_kb(T);
          if (nkb == 0) continue;  // empty WGRAD group: the epilogue writes zeros
          if (!mbar_wait(&sm.acc_empty, aphase ^ 1u, ab, status)) {
            alive = false;
            break;
          }
          tc_fence_after();
          for (int kb = 0; kb < nkb; ++kb) {
            if (!mbar_wait(&sm.full[stage], phase, ab, status) || !mbar_wait(&sm.sf_full[stage], phase, ab, status)) {
              alive = false;
              break;
            }
            tc_fence_after();
            const uint32_t sf_col = tmem + SF_COL0 + static_cast<uint32_t>(stage) * 16;
            tmem_cp_32x128b_warpx4(sf_col, sdesc_plain_128b_rows(smem_u32(sm.sfa[stage])));
            tmem_cp_32x128b_warpx4(sf_col + 4, sdesc_plain_128b_rows(smem_u32(sm.sfb[stage])));
            tmem_cp_32x128b_warpx4(sf_col + 8, sdesc_plain_128b_rows(smem_u32(sm.sfb[stage] + 128)));
            const int k0 = T.k_begin + kb * BK;
            const int chunks = min(4, (T.k_end - k0) / 32);
            const uint32_t a_addr = smem_u32(sm.a[stage]);
            const uint32_t b_addr = smem_u32(sm.b[stage]);
            for (int j = 0; j < chunks; ++j) {
              mma_mx_e4m3(tmem + ACC_COL, sdesc_kmajor_sw128(a_addr + j * 32), sdesc_kmajor_sw128(b_addr + j * 32),
                          idesc_mx_e4m3(BM, BN, static_cast<uint32_t>(j), static_cast<uint32_t>(j)), sf_col,
                          sf_col + 4, (kb > 0 || j > 0) ? 1u : 0u);
            }
            mma_commit(&sm.empty[stage]);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!alive) break;
          mma_commit(&sm.acc_full);
          aphase ^= 1u;
        }
        if (!alive) {
          mma_commit(&sm.mma_drain);
          int dummy = 0;
          mbar_wait(&sm.mma_drain, 0, AbortFlag{&dummy}, status, 1000000ull);
        }
      }
    } else if (warp == 2) {
      // ------------------------------------------------------------ scale-factor gatherer
      int stage = 0;
      uint32_t phase = 0;
      bool alive = true;
      const int64_t a_row_bytes = (p.kind == 2 ? p.M : p.kc) / 32;
      for (int t = blockIdx.x; t < p.num_tiles && alive; t += gridDim.x) {
        const Tile T = decode(sm, p, t);
        const int nkb = num_kb(T);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&sm.empty[stage], phase ^ 1u, ab, status)) {
            alive = false;
            break;
          }
          const int k0 = T.k_begin + kb * BK;
#pragma unroll
          for (int i = 0; i < BM / 32; ++i) {
            const int r = i * 32 + lane;
            const int64_t row = T.a_row0 + r;
            const uint32_t w = row < a_rows ? row_sf(a_e8, row, a_row_bytes, k0, T.k_end, sf_aligned) : 0u;
            sm.sfa[stage][(r & 31) * 4 + (r >> 5)] = w;
          }
#pragma unroll
          for (int i = 0; i < BN / 32; ++i) {
            const int r = i * 32 + lane;
            const int64_t row = T.b_row0 + r;
            const uint32_t w = row < b_rows ? row_sf(b_e8, row, a_row_bytes, k0, T.k_end, sf_aligned) : 0u;
            sm.sfb[stage][(r >> 7) * 128 + (r & 31) * 4 + ((r >> 5) & 3)] = w;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.sf_full[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else {
    regs_inc<208>();
    // ------------------------------------------------------------ epilogue
    const int ew = warp - EPI_WARP0;
    const int half = ew >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t t_lane = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t aphase = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      const Tile T = decode(sm, p, t);
      const int nkb = num_kb(T);
      const int out_row = T.out_row0 + row;
      const bool store = out_row < T.row_limit;
      uint16_t* orow = out;
      if (p.kind == 2) {
        orow += (static_cast<int64_t>(T.g) * p.N + out_row) * p.n_out + T.out_col0 + half * 128;
      } else {
        orow += static_cast<int64_t>(out_row) * p.n_out + T.out_col0 + half * 128;
      }
      uint32_t v[64];  // 128 bf16 values of this thread's row, packed in pairs
      if (nkb == 0) {
#pragma unroll
        for (int i = 0; i < 64; ++i) v[i] = 0u;
      } else {
        if (!mbar_wait(&sm.acc_full, aphase, ab, status)) break;
        aphase ^= 1u;
        tc_fence_after();
        const uint32_t t_base = tmem + t_lane + ACC_COL + static_cast<uint32_t>(half * 128);
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          uint32_t r[4][16];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x16(t_base + (g * 4 + c) * 16, r[c]);
          tmem_ld_wait();
          if (g == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.acc_empty);
          }
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int j = 0; j < 8; ++j)
              v[(g * 4 + c) * 8 + j] = pack_bf16x2(__uint_as_float(r[c][2 * j]), __uint_as_float(r[c][2 * j + 1]));
        }
      }
      if (store) {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(orow + c * 8), "r"(v[4 * c]),
                       "r"(v[4 * c + 1]), "r"(v[4 * c + 2]), "r"(v[4 * c + 3])
                       : "memory");
        }
      }
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

cudaError_t launch_mx_grouped_gemm(const MxGroupedGemmArgs& g, cudaStream_t st) {
  Problem p{};
  p.kind = g.kind;
  p.G = static_cast<int>(g.G);
  p.M = static_cast<int>(g.M);
  p.N = static_cast<int>(g.N);
  p.K = static_cast<int>(g.K);
  int64_t a_rows, a_cols, b_rows, b_cols;
  if (g.kind == 0) {          // FWD: A = x [M, K], B = W [G*N, K]
    p.n_out = p.N;
    p.kc = p.K;
    a_rows = g.M, a_cols = g.K, b_rows = g.G * g.N, b_cols = g.K;
  } else if (g.kind == 1) {   // DGRAD: A = dy [M, N], B = W^T [G*K, N]
    p.n_out = p.K;
    p.kc = p.N;
    a_rows = g.M, a_cols = g.N, b_rows = g.G * g.K, b_cols = g.N;
  } else {                    // WGRAD: A = dy^T [N, M], B = x^T [K, M]
    p.n_out = p.K;
    p.kc = p.M;
    a_rows = g.N, a_cols = g.M, b_rows = g.K, b_cols = g.M;
  }
  p.num_nt = p.n_out / BN;
  // FWD/DGRAD: at most M/128 + G row tiles; the kernel computes the exact
  // count from group_end and skips the tiles past it.
  const int max_mt = p.M / BM + p.G;
  p.num_mt = max_mt;
  p.num_tiles = g.kind == 2 ? p.G * (p.N / BM) * p.num_nt : max_mt * p.num_nt;
  CUtensorMap ta, tb;
  if (!encode_kmajor_u8(&ta, g.a, a_rows, a_cols, BM) || !encode_kmajor_u8(&tb, g.b, b_rows, b_cols, BN))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(mx_grouped_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  const int grid = p.num_tiles < g.num_sms ? p.num_tiles : g.num_sms;
  mx_grouped_gemm_kernel<<<grid, NUM_THREADS, kSmemBytes, st>>>(ta, tb, g.a_e8, g.b_e8, g.group_end, g.out, p, a_rows,
                                                                b_rows, g.status);
  return cudaGetLastError();
}

}  // namespace fp8bw
