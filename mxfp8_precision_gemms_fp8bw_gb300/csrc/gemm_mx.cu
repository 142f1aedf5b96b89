// MXFP8 grouped GEMM (placeholder until the block-scaled kernel lands).
#include "common.cuh"
#include "launch.h"

namespace fp8bw {
cudaError_t launch_mx_grouped_gemm(const MxGroupedGemmArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace fp8bw
