// Internal launchers of libfp8bw: one per kernel family.  The C ABI in
// api.cu validates every argument, then calls these; they only configure and
// enqueue kernels and return the launch status.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace fp8bw {

cudaError_t launch_quant_1x128_row(const uint16_t* x, int64_t R, int64_t C, uint8_t* q, float* s, cudaStream_t st);
cudaError_t launch_quant_1x128_col(const uint16_t* x, int64_t R, int64_t C, uint8_t* qT, float* s, cudaStream_t st);
cudaError_t launch_quant_1x128_rowcol(const uint16_t* x, int64_t R, int64_t C, uint8_t* q, float* s, uint8_t* qT,
                                      float* sT, cudaStream_t st);
cudaError_t launch_quant_128x128(const uint16_t* w, int64_t R, int64_t C, uint8_t* q, uint8_t* qT, float* s,
                                 int64_t s_ld, cudaStream_t st);
cudaError_t launch_mx_quant_row(const uint16_t* x, int64_t R, int64_t C, uint8_t* q, uint8_t* e8, int mode,
                                cudaStream_t st);
cudaError_t launch_mx_quant_col(const uint16_t* x, int64_t G, int64_t R, int64_t C, uint8_t* qT, uint8_t* e8,
                                int mode, cudaStream_t st);
cudaError_t launch_mx_quant_rowcol(const uint16_t* x, int64_t G, int64_t R, int64_t C, uint8_t* q, uint8_t* e8,
                                   uint8_t* qT, uint8_t* e8T, int mode, cudaStream_t st);

// Which operand-B scale structure a blockwise GEMM applies (see gemm_blockwise.cu).
enum class BScale : int {
  kBlock128x128 = 0,   // one scale per 128x128 block of B: sb[nb * ld_nb + kb * ld_kb]
  kPerRow = 1          // one scale per B row per contraction block: sb[kb * ld_kb + n]
};

struct BlockwiseGemmArgs {
  const uint8_t* a;   // [Mo, Kc] e4m3, K-major
  const uint8_t* b;   // [No, Kc] e4m3, K-major, or [Kc, No] when b_mn_major
  bool b_mn_major;    // kBlock128x128 only, without output quantization
  const float* sa;    // sa[kb * sa_ld + m]
  int64_t sa_ld;
  const float* sb;
  int64_t sb_ld_nb;   // kBlock128x128: stride between 128-row blocks of B
  int64_t sb_ld_kb;   // stride between contraction blocks
  BScale b_scale;
  uint16_t* out;      // [Mo, No] bf16 (unused when out_acc is set)
  float* out_acc;     // kPerRow only, may be null: out_acc[Mo, No] += result in fp32
  // kBlock128x128 only, may be null: the 1x128 rowwise quantization of the
  // bf16 output (q_out [Mo, No], s_out [No/128][Mo]) and, with qT_out set
  // too, its colwise one (qT_out [No, Mo], sT_out [Mo/128][No]).
  uint8_t* q_out;
  float* s_out;
  uint8_t* qT_out;
  float* sT_out;
  // kPerRow with out_acc null, may be null: workspace for the contraction
  // split of the last round of tiles (wgrad_split_plan(...).bytes).
  void* split_ws;
  size_t split_ws_bytes;
  int64_t Mo, No, Kc;
  int* status;
  int num_sms;
};
cudaError_t launch_blockwise_gemm(const BlockwiseGemmArgs& args, cudaStream_t st);

// How the per-column-scale (wgrad) kernel splits its last round of tiles on
// num_sms SMs: full_units whole tiles, then each of the `tail` remaining tiles
// in k contraction parts (k = 1: no split); bytes of workspace it needs.
struct WgradSplitPlan {
  int full_units, tail, k;
  size_t bytes;
};
WgradSplitPlan wgrad_split_plan(int64_t Mo, int64_t No, int64_t Kc, int num_sms);

struct MxGroupedGemmArgs {
  int kind;                   // 0 fwd, 1 dgrad, 2 wgrad
  const uint8_t* a;
  const uint8_t* a_e8;
  const uint8_t* b;
  const uint8_t* b_e8;
  const int32_t* group_end;
  int64_t G, M, N, K;
  uint16_t* out;
  void* workspace;            // packed scale factors (mx_grouped_gemm_workspace_bytes)
  size_t workspace_bytes;
  int* status;
  int num_sms;
};
size_t mx_grouped_gemm_workspace_bytes(int kind, int64_t G, int64_t M, int64_t N, int64_t K);

// Size of the fixed scratch array behind mxfp8_grouped_gemm_noalloc (16 MiB).
constexpr size_t kStaticScratchBytes = size_t{16} << 20;
// Its device address on the current device (resolved once per device).
cudaError_t static_scratch_address(void** out);
cudaError_t launch_mx_grouped_gemm(const MxGroupedGemmArgs& args, cudaStream_t st);

cudaError_t launch_selftest_bounded_wait(uint32_t timeout_us, int* status, cudaStream_t st);

// cuTensorMapEncodeTiled, resolved once through the runtime's driver entry
// point query (no link-time dependency on libcuda).
void* tensor_map_encoder();

}  // namespace fp8bw
