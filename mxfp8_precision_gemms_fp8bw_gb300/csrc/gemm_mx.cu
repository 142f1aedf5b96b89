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
// contract over the group's token range in 128-wide windows, issuing only the
// 32-wide MMAs that lie inside the group (group sizes are multiples of 32).
//
// Scale factors reach shared memory by TMA, like the operands.  A pack kernel
// launched just before the GEMM rewrites the row-major E8M0 bytes into
// 512-byte chunks, one per 128 operand rows per 128-wide contraction window,
// already in the 32-row x 16-byte interleaved layout tcgen05.cp consumes (row
// r of the chunk -> 32-bit word (r % 32) * 4 + r / 32; byte j of the word =
// scale of the window's j-th 32-element chunk).  The chunks live in a
// caller-provided workspace, B's two 128-row chunks of a stage side by side:
//   FWD/DGRAD  A: [Kc/128][M/128 + G][512 B]   (row tiles start at group starts)
//              B: [Kc/128][G*Nout/128][512 B]
//   WGRAD      A: [M/128 + G windows][N/128][512 B]
//              B: [M/128 + G windows][K/128][512 B]
// (windows: the 128-token steps of each group, numbered group after group).
//
// GEMM CTA (persistent, 384 threads), run in clusters of two CTAs whose
// tiles share B (consecutive 128-token tiles of one group for FWD/DGRAD,
// consecutive dW row tiles of one group for WGRAD; a WGRAD with an odd
// N / 128 runs unpaired):
//   warp 0      TMA producer: per stage the CTA's A 128x128 tile, one
//               128-row half of the shared B 256x128 tile, which the TMA
//               multicast writes into both CTAs (each SM fetches 32 KB of
//               operands per stage instead of 48 KB), and the 512 B + 1 KB
//               scale chunks (bulk copies); a stage is refilled once the
//               MMAs of both CTAs have read it
//   warp 1      TMEM owner and MMA issuer: up to 4 block-scaled MMAs per
//               stage (K = 32 each; the instruction descriptor selects scale
//               byte j)
//   warp 2      scale copier: once a stage has landed, tcgen05.cp of its scale
//               chunks into that stage's TMEM slot, committed to the stage's
//               sf_ready barrier, which the MMA issuer waits on instead of the
//               load barrier (the copies stay off the issuing thread, where
//               every instruction delays the next MMA)
//   warp 3      idle
//   warps 4-11  epilogue: drain the accumulator (warp w: lanes 32*(w%4).., one
//               128-column half), release it, write bf16 rows.
#include <mutex>

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
constexpr int SFA_BYTES = BM * 4;
constexpr int SFB_BYTES = BN * 4;
constexpr int NUM_THREADS = 384;
constexpr int EPI_WARP0 = 4;
constexpr int NUM_EPI_WARPS = 8;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COL = 0;    // accumulator: columns [0, 256)
constexpr uint32_t SF_COL0 = 256;  // per stage: SFA 4 columns, SFB 8 columns, in 16-column slots
constexpr int GROUP_M = 16;
constexpr int MAX_GROUPS = 1024;

struct Problem {
  int kind, G, M, N, K;
  int n_out;    // output columns
  int kc;       // FWD/DGRAD contraction length
  int mt_max;   // FWD/DGRAD row tiles / WGRAD windows bound: M/128 + G
  int rb_b;     // FWD/DGRAD: 128-row chunks of B (G * n_out / 128)
  int num_nt;   // output column tiles (256 wide)
  int num_tiles;
};

struct GroupTable {
  int32_t start[MAX_GROUPS + 1];  // token start of each group (sanitized), start[G] = end
  int32_t tile0[MAX_GROUPS + 1];  // first 128-token tile / window of each group; tile0[G] = total
  int32_t pair0[MAX_GROUPS + 1];  // FWD/DGRAD, CTA pairs: first pair of 128-token tiles of each group
};

// Clamps every group range into [0, M] and rounds each end down to a multiple
// of 32 (so every token coordinate stays 32-byte aligned for TMA whatever
// group_end holds).  Returns true when group_end broke the rules (a size that
// is not a multiple of 32, a decreasing end, or a last end other than M).
__device__ bool build_group_table(const int32_t* group_end, int G, int M, GroupTable& t) {
  int prev = 0, tile0 = 0, pair0 = 0;
  bool bad = false;
  for (int g = 0; g < G; ++g) {
    int e = group_end[g];
    if (e < prev || e > M || ((e - prev) & 31) != 0) bad = true;
    e = max(min(max(e, prev), M) & ~31, prev);
    t.start[g] = prev;
    t.tile0[g] = tile0;
    t.pair0[g] = pair0;
    const int tiles = (e - prev + BM - 1) / BM;
    tile0 += tiles;
    pair0 += (tiles + 1) / 2;
    prev = e;
  }
  if (prev != M) bad = true;
  t.start[G] = prev;
  t.tile0[G] = tile0;
  t.pair0[G] = pair0;
  return bad;
}

// The group owning 128-token tile (or window) i: the last g with tile0[g] <= i
// (empty groups own no tile and are skipped).
__device__ __forceinline__ int group_of_in(const int32_t* first, int G, int i) {
  int lo = 0, hi = G;  // invariant: first[lo] <= i < first[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (first[mid] <= i) lo = mid;
    else hi = mid;
  }
  return lo;
}
__device__ __forceinline__ int group_of(const GroupTable& t, int G, int i) { return group_of_in(t.tile0, G, i); }

struct SharedStorage {
  uint8_t a[STAGES][A_BYTES];
  uint8_t b[STAGES][B_BYTES];
  uint32_t sfa[STAGES][BM];
  uint32_t sfb[STAGES][BN];
  GroupTable groups;
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t sf_ready[STAGES];  // the stage's scale factors are in TMEM (and its tiles in smem)
  uint64_t acc_full;
  uint64_t acc_empty;
  uint64_t mma_drain;
  uint64_t cp_drain;
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t kSmemBytes = sizeof(SharedStorage) + 1024;

struct Tile {
  int g;
  int a_row0, b_row0;           // first rows of A and B
  int k_begin, k_end;           // contraction range
  int out_row0, row_limit;      // first output row; rows >= row_limit are not stored
  int out_col0;
  int64_t sfa_chunk0, sfa_step;  // scale chunks of A: chunk0 + kb * step
  int64_t sfb_chunk0, sfb_step;  // of B (two adjacent chunks per stage)
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

__device__ __forceinline__ Tile decode(const GroupTable& gt, const Problem& p, int t) {
  Tile T;
  if (p.kind != 2) {
    int mt, nt;
    raster(t, gt.tile0[p.G], p.num_nt, mt, nt);
    const int g = group_of(gt, p.G, mt);
    const int m0 = gt.start[g] + (mt - gt.tile0[g]) * BM;
    T.g = g;
    T.a_row0 = m0;
    T.b_row0 = g * p.n_out + nt * BN;
    T.k_begin = 0;
    T.k_end = p.kc;
    T.out_row0 = m0;
    T.row_limit = gt.start[g + 1];
    T.out_col0 = nt * BN;
    T.sfa_chunk0 = mt;
    T.sfa_step = p.mt_max;
    T.sfb_chunk0 = T.b_row0 / BM;
    T.sfb_step = p.rb_b;
  } else {
    const int rb_a = p.N / BM, rb_b = p.K / BM;
    const int per_group = rb_a * p.num_nt;
    const int g = t / per_group;
    int mt, nt;
    raster(t - g * per_group, rb_a, p.num_nt, mt, nt);
    T.g = g;
    T.a_row0 = mt * BM;
    T.b_row0 = nt * BN;
    T.k_begin = gt.start[g];
    T.k_end = gt.start[g + 1];
    T.out_row0 = mt * BM;
    T.row_limit = p.N;
    T.out_col0 = nt * BN;
    T.sfa_chunk0 = static_cast<int64_t>(gt.tile0[g]) * rb_a + mt;
    T.sfa_step = rb_a;
    T.sfb_chunk0 = static_cast<int64_t>(gt.tile0[g]) * rb_b + T.b_row0 / BM;
    T.sfb_step = rb_b;
  }
  return T;
}

// The tile of CTA `rank` (0 or 1) of a cluster for pair-tile `pt`: the two
// CTAs take two 128-row tiles that share one 256-row B tile -- consecutive
// token tiles of one group (FWD/DGRAD; a group with an odd tile count gets a
// second tile whose rows all lie past the group's end, computed and never
// stored) or consecutive dW row tiles of one group (WGRAD).
__device__ __forceinline__ Tile decode_pair(const GroupTable& gt, const Problem& p, int pt, int rank) {
  Tile T;
  if (p.kind != 2) {
    int pm, nt;
    raster(pt, gt.pair0[p.G], p.num_nt, pm, nt);
    const int g = group_of_in(gt.pair0, p.G, pm);
    const int local = 2 * (pm - gt.pair0[g]) + rank;
    const int tiles = gt.tile0[g + 1] - gt.tile0[g];
    const int m0 = gt.start[g] + local * BM;
    T.g = g;
    T.a_row0 = m0;
    T.b_row0 = g * p.n_out + nt * BN;
    T.k_begin = 0;
    T.k_end = p.kc;
    T.out_row0 = m0;
    T.row_limit = gt.start[g + 1];
    T.out_col0 = nt * BN;
    // A tile past the group's end reads any valid scale chunk of the group.
    T.sfa_chunk0 = gt.tile0[g] + min(local, tiles - 1);
    T.sfa_step = p.mt_max;
    T.sfb_chunk0 = T.b_row0 / BM;
    T.sfb_step = p.rb_b;
  } else {
    const int rb_a = p.N / BM, rb_b = p.K / BM;
    const int per_group = (rb_a / 2) * p.num_nt;
    const int g = pt / per_group;
    int pm, nt;
    raster(pt - g * per_group, rb_a / 2, p.num_nt, pm, nt);
    const int mt = 2 * pm + rank;
    T.g = g;
    T.a_row0 = mt * BM;
    T.b_row0 = nt * BN;
    T.k_begin = gt.start[g];
    T.k_end = gt.start[g + 1];
    T.out_row0 = mt * BM;
    T.row_limit = p.N;
    T.out_col0 = nt * BN;
    T.sfa_chunk0 = static_cast<int64_t>(gt.tile0[g]) * rb_a + mt;
    T.sfa_step = rb_a;
    T.sfb_chunk0 = static_cast<int64_t>(gt.tile0[g]) * rb_b + T.b_row0 / BM;
    T.sfb_step = rb_b;
  }
  return T;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// 2D tiled load delivered to the same shared-memory offset (data and
// mbarrier) of every CTA of the cluster in `mask`.
__device__ __forceinline__ void tma_load_2d_multicast(void* dst, const CUtensorMap* map, uint64_t* bar, int32_t c0,
                                                      int32_t c1, uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "h"(mask)
      : "memory");
}
// tcgen05.commit arriving on the mbarrier at `bar`'s offset in every CTA of `mask`.
__device__ __forceinline__ void mma_commit_multicast(uint64_t* bar, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "h"(mask)
               : "memory");
}

__device__ __forceinline__ int num_kb(const Tile& T) { return (T.k_end - T.k_begin + BK - 1) / BK; }

// 1D bulk copy global -> shared completing `bytes` on `bar` (16-byte aligned).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// ---------------------------------------------------------------- scale packing

// Words of the packed scale regions (see the file comment).
__host__ __device__ inline int64_t packed_words_a(const Problem& p) {
  return p.kind != 2 ? static_cast<int64_t>(p.kc / BK) * p.mt_max * BM
                     : static_cast<int64_t>(p.mt_max) * (p.N / BM) * BM;
}
__host__ __device__ inline int64_t packed_words_b(const Problem& p) {
  return p.kind != 2 ? static_cast<int64_t>(p.kc / BK) * p.rb_b * BM
                     : static_cast<int64_t>(p.mt_max) * (p.K / BM) * BM;
}

// One thread per packed 32-bit word: gathers the four E8M0 bytes of one
// operand row for one 128-wide contraction window.
__global__ void __launch_bounds__(256) mx_pack_scales_kernel(const uint8_t* __restrict__ a_e8,
                                                             const uint8_t* __restrict__ b_e8,
                                                             const int32_t* __restrict__ group_end, Problem p,
                                                             uint32_t* __restrict__ ws_a, uint32_t* __restrict__ ws_b) {
  __shared__ GroupTable gt;
  if (threadIdx.x == 0) build_group_table(group_end, p.G, p.M, gt);
  __syncthreads();
  const int64_t words_a = packed_words_a(p), total = words_a + packed_words_b(p);
  const int64_t e8_row_bytes = (p.kind == 2 ? p.M : p.kc) / 32;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const bool is_a = i < words_a;
    const int64_t w = is_a ? i : i - words_a;
    const int slot = static_cast<int>(w & 127);
    const int64_t chunk = w >> 7;
    const int r = (slot & 3) * 32 + (slot >> 2);  // row of the 128-row chunk held by this word
    const uint8_t* e8 = is_a ? a_e8 : b_e8;
    uint32_t word = 0;
    if (p.kind != 2) {
      // chunk = kb * rows_chunks + row_chunk
      const int rows_chunks = is_a ? p.mt_max : p.rb_b;
      const int kb = static_cast<int>(chunk / rows_chunks);
      const int rc = static_cast<int>(chunk - static_cast<int64_t>(kb) * rows_chunks);
      int64_t row = -1;
      if (is_a) {
        if (rc < gt.tile0[p.G]) {
          const int g = group_of(gt, p.G, rc);
          row = gt.start[g] + static_cast<int64_t>(rc - gt.tile0[g]) * BM + r;
          if (row >= p.M) row = -1;
        }
      } else {
        row = static_cast<int64_t>(rc) * BM + r;
      }
      if (row >= 0) word = __ldg(reinterpret_cast<const unsigned int*>(e8 + row * e8_row_bytes + kb * 4));
    } else {
      // chunk = window * row_chunks + row_chunk
      const int rows_chunks = (is_a ? p.N : p.K) / BM;
      const int win = static_cast<int>(chunk / rows_chunks);
      const int rc = static_cast<int>(chunk - static_cast<int64_t>(win) * rows_chunks);
      if (win < gt.tile0[p.G]) {
        const int g = group_of(gt, p.G, win);
        const int k0 = gt.start[g] + (win - gt.tile0[g]) * BK;
        const int k_end = gt.start[g + 1];
        const uint8_t* src = e8 + (static_cast<int64_t>(rc) * BM + r) * e8_row_bytes + k0 / 32;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (k0 + 32 * j < k_end) word |= static_cast<uint32_t>(__ldg(src + j)) << (8 * j);
      }
    }
    (is_a ? ws_a : ws_b)[w] = word;
  }
}

// ---------------------------------------------------------------- GEMM

// kPair: the kernel runs in clusters of two CTAs that share each stage's B
// tile; each CTA loads half of it (128 rows) and the TMA multicast delivers
// both halves to both CTAs, so each SM fetches 32 KB instead of 48 KB per
// stage.  Each CTA still issues its own M128 N256 MMAs on its own A tile.
template <bool kPair>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    mx_grouped_gemm_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                           const uint32_t* __restrict__ ws_a, const uint32_t* __restrict__ ws_b,
                           const int32_t* __restrict__ group_end, uint16_t* __restrict__ out, Problem p,
                           int* status) {
  extern __shared__ uint8_t smem_raw[];
  SharedStorage& sm =
      *reinterpret_cast<SharedStorage*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const AbortFlag ab{&sm.abort_flag};

  if (threadIdx.x == 0) {
    if (build_group_table(group_end, p.G, p.M, sm.groups) && blockIdx.x == 0) atomicExch(status, kStatusShape);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sm.full[s], 1);
      // A stage is free once the MMAs of every CTA that received its B half have read it.
      mbar_init(&sm.empty[s], kPair ? 2 : 1);
      mbar_init(&sm.sf_ready[s], 1);
    }
    mbar_init(&sm.acc_full, 1);
    mbar_init(&sm.acc_empty, NUM_EPI_WARPS);
    mbar_init(&sm.mma_drain, 1);
    mbar_init(&sm.cp_drain, 1);
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
  // The peer's multicast loads and commits target this CTA's barriers.
  if constexpr (kPair) cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const GroupTable& gt = sm.groups;
  // Work items: tiles, or for CTA pairs pair-tiles walked by clusters.
  const int rank = kPair ? static_cast<int>(cluster_rank()) : 0;
  const int first = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int stride = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  if (kPair) {
    p.num_tiles = p.kind != 2 ? gt.pair0[p.G] * p.num_nt : p.G * (p.N / BM / 2) * p.num_nt;
  } else if (p.kind != 2) {
    p.num_tiles = gt.tile0[p.G] * p.num_nt;
  }
  auto tile_of = [&](int t) { return kPair ? decode_pair(gt, p, t, rank) : decode(gt, p, t); };

  if (warp < EPI_WARP0) {
    regs_dec<88>();
    if (warp == 0) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        int stage = 0;
        uint32_t phase = 0, issued = 0;
        bool alive = true;
        for (int t = first; t < p.num_tiles && alive; t += stride) {
          const Tile T = tile_of(t);
          const int nkb = num_kb(T);
          for (int kb = 0; kb < nkb; ++kb) {
            if (!mbar_wait(&sm.empty[stage], phase ^ 1u, ab, status)) {
              alive = false;
              break;
            }
            const int k0 = T.k_begin + kb * BK;
            mbar_arrive_expect_tx(&sm.full[stage], A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES);
            tma_load_2d(sm.a[stage], &tma_a, &sm.full[stage], k0, T.a_row0);
            if constexpr (kPair) {
              tma_load_2d_multicast(sm.b[stage] + rank * (B_BYTES / 2), &tma_b, &sm.full[stage], k0,
                                    T.b_row0 + rank * (BN / 2), 0x3);
            } else {
              tma_load_2d(sm.b[stage], &tma_b, &sm.full[stage], k0, T.b_row0);
            }
            bulk_load(sm.sfa[stage], ws_a + (T.sfa_chunk0 + kb * T.sfa_step) * BM, SFA_BYTES, &sm.full[stage]);
            bulk_load(sm.sfb[stage], ws_b + (T.sfb_chunk0 + kb * T.sfb_step) * BM, SFB_BYTES, &sm.full[stage]);
            ++issued;
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (kPair && alive) {
          // The peer's last commits arrive on this CTA's empty barriers: wait
          // for every stage's final release before the CTA may exit.
          for (int i = 0; i < STAGES; ++i) {
            if (!mbar_wait(&sm.empty[stage], phase ^ 1u, ab, status)) break;
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (!alive) {
          // Unwinding: only the last STAGES loads can still be in flight.
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
        // Descriptors of stage 0; stage s and the 32-byte K step j are plain
        // adds to the start-address field (in 16-byte units).
        const uint64_t a_desc0 = sdesc_kmajor_sw128(smem_u32(sm.a[0]));
        const uint64_t b_desc0 = sdesc_kmajor_sw128(smem_u32(sm.b[0]));
        const uint32_t acc = tmem + ACC_COL;
        for (int t = first; t < p.num_tiles && alive; t += stride) {
          const Tile T = tile_of(t);
          const int nkb = num_kb(T);
          if (nkb == 0) continue;  // empty WGRAD group: the epilogue writes zeros
          if (!mbar_wait(&sm.acc_empty, aphase ^ 1u, ab, status)) {
            alive = false;
            break;
          }
          tc_fence_after();
          for (int kb = 0; kb < nkb; ++kb) {
            // Waited after the previous stage's last MMA, not before it: the
            // scale copies that complete sf_ready pass through the tensor
            // pipe behind the queued MMAs, so an earlier wait stalls the pipe.
            if (!mbar_wait(&sm.sf_ready[stage], phase, ab, status)) {
              alive = false;
              break;
            }
            tc_fence_after();
            const uint32_t sf_col = tmem + SF_COL0 + static_cast<uint32_t>(stage) * 16;
            const int k0 = T.k_begin + kb * BK;
            const int chunks = min(4, (T.k_end - k0) / 32);
            const uint64_t ad = a_desc0 + static_cast<uint64_t>(stage * (A_BYTES >> 4));
            const uint64_t bd = b_desc0 + static_cast<uint64_t>(stage * (B_BYTES >> 4));
            if (chunks == 4) {
              // A whole 128-deep window: four MMAs, scale byte j for the j-th.
              if (kb == 0) mma_mx_e4m3_k<false>(acc, ad, bd, idesc_mx_e4m3(BM, BN, 0, 0), sf_col, sf_col + 4);
              else mma_mx_e4m3_k<true>(acc, ad, bd, idesc_mx_e4m3(BM, BN, 0, 0), sf_col, sf_col + 4);
              mma_mx_e4m3_k<true>(acc, ad + 2, bd + 2, idesc_mx_e4m3(BM, BN, 1, 1), sf_col, sf_col + 4);
              mma_mx_e4m3_k<true>(acc, ad + 4, bd + 4, idesc_mx_e4m3(BM, BN, 2, 2), sf_col, sf_col + 4);
              mma_mx_e4m3_k<true>(acc, ad + 6, bd + 6, idesc_mx_e4m3(BM, BN, 3, 3), sf_col, sf_col + 4);
            } else {
              // The last window of a group whose size is not a multiple of 128.
              for (int j = 0; j < chunks; ++j) {
                mma_mx_e4m3(acc, ad + 2 * j, bd + 2 * j,
                            idesc_mx_e4m3(BM, BN, static_cast<uint32_t>(j), static_cast<uint32_t>(j)), sf_col,
                            sf_col + 4, (kb > 0 || j > 0) ? 1u : 0u);
              }
            }
            if constexpr (kPair) mma_commit_multicast(&sm.empty[stage], 0x3);
            else mma_commit(&sm.empty[stage]);
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
      // ------------------------------------------------------------ scale copier
      if (lane == 0) {
        int stage = 0;
        uint32_t phase = 0;
        bool alive = true;
        const uint64_t sfa_desc0 = sdesc_plain_128b_rows(smem_u32(sm.sfa[0]));
        const uint64_t sfb_desc0 = sdesc_plain_128b_rows(smem_u32(sm.sfb[0]));
        for (int t = first; t < p.num_tiles && alive; t += stride) {
          const int nkb = num_kb(tile_of(t));
          for (int kb = 0; kb < nkb; ++kb) {
            // Stage `stage` of this round has landed; its TMEM slot was last
            // read by the MMAs of the previous round, which completed before
            // the producer could refill the stage.
            if (!mbar_wait(&sm.full[stage], phase, ab, status)) {
              alive = false;
              break;
            }
            tc_fence_after();
            const uint32_t sf_col = tmem + SF_COL0 + static_cast<uint32_t>(stage) * 16;
            const uint64_t sfa_d = sfa_desc0 + static_cast<uint64_t>(stage * (SFA_BYTES >> 4));
            const uint64_t sfb_d = sfb_desc0 + static_cast<uint64_t>(stage * (SFB_BYTES >> 4));
            tmem_cp_32x128b_warpx4(sf_col, sfa_d);
            tmem_cp_32x128b_warpx4(sf_col + 4, sfb_d);
            tmem_cp_32x128b_warpx4(sf_col + 8, sfb_d + ((BM * 4) >> 4));  // B's second 128-row chunk, 512 B on
            mma_commit(&sm.sf_ready[stage]);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (!alive) {
          // Unwinding: wait for this thread's copies already issued before TMEM is freed.
          mma_commit(&sm.cp_drain);
          int dummy = 0;
          mbar_wait(&sm.cp_drain, 0, AbortFlag{&dummy}, status, 1000000ull);
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
    const bool out32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
    uint32_t aphase = 0;
    for (int t = first; t < p.num_tiles; t += stride) {
      const Tile T = tile_of(t);
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
      if (store && out32) {
        // Eight 32-byte stores: each lane writes whole sectors of its row
        // (out is 32-byte aligned and every row segment starts a multiple of
        // 256 bytes into its row).
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(orow + c * 16),
                       "r"(v[8 * c]), "r"(v[8 * c + 1]), "r"(v[8 * c + 2]), "r"(v[8 * c + 3]), "r"(v[8 * c + 4]),
                       "r"(v[8 * c + 5]), "r"(v[8 * c + 6]), "r"(v[8 * c + 7])
                       : "memory");
        }
      } else if (store) {
        // out only 16-byte aligned: the same bytes as 16-byte stores.
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(orow + c * 8), "r"(v[4 * c]),
                       "r"(v[4 * c + 1]), "r"(v[4 * c + 2]), "r"(v[4 * c + 3])
                       : "memory");
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // Neither CTA of a pair leaves while the other may still signal it.
  if constexpr (kPair) cluster_sync_all();
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

Problem make_problem(int kind, int64_t G, int64_t M, int64_t N, int64_t K) {
  Problem p{};
  p.kind = kind;
  p.G = static_cast<int>(G);
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.n_out = kind == 0 ? p.N : p.K;
  p.kc = kind == 0 ? p.K : (kind == 1 ? p.N : p.M);
  p.mt_max = p.M / BM + p.G;
  p.rb_b = kind == 2 ? 0 : p.G * p.n_out / BM;
  p.num_nt = p.n_out / BN;
  // FWD/DGRAD: the kernel takes the exact count from group_end; this is its bound.
  p.num_tiles = kind == 2 ? p.G * (p.N / BM) * p.num_nt : p.mt_max * p.num_nt;
  return p;
}

constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

}  // namespace

// Scratch of mxfp8_grouped_gemm_noalloc: a fixed array in the library's own
// device image, so that entry point never allocates.  Every GPU that loads
// the library holds it until the process exits.  In host code this name is a
// host-side stand-in, never a device address: launches get the address from
// static_scratch_address().
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch on the current device, resolved once per
// device (host code may not use the symbol itself as a device pointer).
cudaError_t static_scratch_address(void** out) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

// Clusters of two CTAs of the pair kernel that fit on the current device at
// once, resolved on a device's first call (the query is not a stream
// operation, so later calls can be captured in a CUDA graph).
static cudaError_t pair_clusters(cudaLaunchConfig_t* cfg, int* out) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static int clusters[kMaxDevices] = {};
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (clusters[dev] == 0) {
    e = cudaFuncSetAttribute(mx_grouped_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    const dim3 grid = cfg->gridDim;
    cfg->gridDim = dim3(2);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, mx_grouped_gemm_kernel<true>, cfg);
    cfg->gridDim = grid;
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    clusters[dev] = n;
  }
  *out = clusters[dev];
  return cudaSuccess;
}

size_t mx_grouped_gemm_workspace_bytes(int kind, int64_t G, int64_t M, int64_t N, int64_t K) {
  const Problem p = make_problem(kind, G, M, N, K);
  return align_up(static_cast<size_t>(packed_words_a(p)) * 4) + align_up(static_cast<size_t>(packed_words_b(p)) * 4);
}

cudaError_t launch_mx_grouped_gemm(const MxGroupedGemmArgs& g, cudaStream_t st) {
  const Problem p = make_problem(g.kind, g.G, g.M, g.N, g.K);
  int64_t a_rows, a_cols, b_rows, b_cols;
  if (g.kind == 0) {          // FWD: A = x [M, K], B = W [G*N, K]
    a_rows = g.M, a_cols = g.K, b_rows = g.G * g.N, b_cols = g.K;
  } else if (g.kind == 1) {   // DGRAD: A = dy [M, N], B = W^T [G*K, N]
    a_rows = g.M, a_cols = g.N, b_rows = g.G * g.K, b_cols = g.N;
  } else {                    // WGRAD: A = dy^T [N, M], B = x^T [K, M]
    a_rows = g.N, a_cols = g.M, b_rows = g.K, b_cols = g.M;
  }
  if (g.workspace_bytes < mx_grouped_gemm_workspace_bytes(g.kind, g.G, g.M, g.N, g.K)) return cudaErrorInvalidValue;
  uint32_t* ws_a = static_cast<uint32_t*>(g.workspace);
  uint32_t* ws_b = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(g.workspace) +
                                               align_up(static_cast<size_t>(packed_words_a(p)) * 4));
  // CTA pairs sharing B: WGRAD pairs dW row tiles, so N / 128 must be even.
  const bool pair = g.kind != 2 || (g.N / BM) % 2 == 0;
  CUtensorMap ta, tb;
  if (!encode_kmajor_u8(&ta, g.a, a_rows, a_cols, BM) ||
      !encode_kmajor_u8(&tb, g.b, b_rows, b_cols, pair ? BN / 2 : BN))
    return cudaErrorInvalidValue;

  const int64_t words = packed_words_a(p) + packed_words_b(p);
  const int64_t pack_blocks = (words + 255) / 256;
  const int pack_grid = static_cast<int>(pack_blocks < 8LL * g.num_sms ? pack_blocks : 8LL * g.num_sms);
  mx_pack_scales_kernel<<<pack_grid, 256, 0, st>>>(g.a_e8, g.b_e8, g.group_end, p, ws_a, ws_b);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  if (!pair) {
    e = cudaFuncSetAttribute(mx_grouped_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    const int grid = p.num_tiles < g.num_sms ? p.num_tiles : g.num_sms;
    mx_grouped_gemm_kernel<false><<<grid, NUM_THREADS, kSmemBytes, st>>>(ta, tb, ws_a, ws_b, g.group_end, g.out, p,
                                                                          g.status);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  e = pair_clusters(&cfg, &clusters);
  if (e != cudaSuccess) return e;
  // Pair-tiles: the kernel takes the exact count from group_end; this bounds it.
  const int64_t pairs = g.kind == 2 ? p.G * (p.N / BM / 2) * p.num_nt : (p.mt_max / 2 + p.G) * p.num_nt;
  const int64_t c = pairs < clusters ? pairs : clusters;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * (c > 0 ? c : 1)));
  e = cudaLaunchKernelEx(&cfg, mx_grouped_gemm_kernel<true>, ta, tb, static_cast<const uint32_t*>(ws_a),
                         static_cast<const uint32_t*>(ws_b), g.group_end, g.out, p, g.status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace fp8bw
