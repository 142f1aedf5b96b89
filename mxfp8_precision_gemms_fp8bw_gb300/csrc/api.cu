// C ABI of libfp8bw (declared in include/fp8bw.h): argument validation, the
// per-device error word, and dispatch to the kernel launchers.  Nothing here
// computes on the host; every call ends in a kernel launch or an error code.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "fp8bw.h"
#include "launch.h"

#define FP8BW_API extern "C" __attribute__((visibility("default")))

namespace {

thread_local char g_msg[512];

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  g_msg[0] = '\0';
  return FP8BW_OK;
}

// The device error word: set by kernels when a bounded wait expires or a
// device-side argument check fails; read and cleared by fp8bw_sync_status.
__device__ int g_error_word;

struct DeviceState {
  bool probed = false;
  bool supported = false;
  int num_sms = 0;
  int* error_word = nullptr;
  char why[160] = {0};
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Checks (once per device) that the current device is compute capability
// 10.3 and resolves the address of its error word.
int current_device(DeviceState** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return fail(FP8BW_ERR_UNSUPPORTED, "no usable CUDA device (%s)", cudaGetErrorString(e));
  }
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.probed) {
    d.probed = true;
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (major != 10 || minor != 3) {
      snprintf(d.why, sizeof(d.why), "device %d has compute capability %d.%d; the kernels are built for sm_103a", dev,
               major, minor);
    } else {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_error_word);
      if (e != cudaSuccess) {
        snprintf(d.why, sizeof(d.why), "cannot resolve the error word: %s", cudaGetErrorString(e));
        cudaGetLastError();
      } else {
        d.error_word = static_cast<int*>(p);
        d.supported = true;
      }
    }
  }
  if (!d.supported) return fail(FP8BW_ERR_UNSUPPORTED, "%s", d.why);
  *out = &d;
  return FP8BW_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1;

bool dim_ok(int64_t d, int64_t mult) { return d > 0 && d <= kMaxDim && d % mult == 0; }

bool overlaps(const void* a, int64_t abytes, const void* b, int64_t bbytes) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + static_cast<uintptr_t>(bbytes) && b0 < a0 + static_cast<uintptr_t>(abytes);
}

int launched(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return fail(FP8BW_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
  return ok();
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

}  // namespace

namespace fp8bw {

void* tensor_map_encoder() {
  static void* fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = p;
    cudaGetLastError();
  });
  return fn;
}

}  // namespace fp8bw

// ============================================================ quantizers

FP8BW_API int fp8bw_quant_1x128_row(const fp8bw_bf16* x, int64_t R, int64_t C, uint8_t* q, float* s, void* stream) {
  if (!x || !q || !s) return fail(FP8BW_ERR_NULL, "fp8bw_quant_1x128_row: x, q and s must be non-NULL");
  if (!dim_ok(R, 128) || !dim_ok(C, 128) || R / 128 > 65535)
    return fail(FP8BW_ERR_SHAPE, "fp8bw_quant_1x128_row: R=%lld and C=%lld must be positive multiples of 128",
                (long long)R, (long long)C);
  if (!aligned16(x) || !aligned16(q) || !aligned16(s))
    return fail(FP8BW_ERR_ALIGN, "fp8bw_quant_1x128_row: pointers must be 16-byte aligned");
  if (overlaps(x, R * C * 2, q, R * C) || overlaps(x, R * C * 2, s, C / 128 * R * 4))
    return fail(FP8BW_ERR_LAYOUT, "fp8bw_quant_1x128_row: outputs overlap the input");
  DeviceState* d;
  if (int rc = current_device(&d)) return rc;
  return launched(fp8bw::launch_quant_1x128_row(x, R, C, q, s, as_stream(stream)), "fp8bw_quant_1x128_row");
}

FP8BW_API int fp8bw_quant_1x128_col(const fp8bw_bf16* x, int64_t R, int64_t C, uint8_t* qT, float* s, void* stream) {
  if (!x || !qT || !s) return fail(FP8BW_ERR_NULL, "fp8bw_quant_1x128_col: x, qT and s must be non-NULL");
  if (!dim_ok(R, 128) || !dim_ok(C, 128) || R / 128 > 65535)
    return fail(FP8BW_ERR_SHAPE, "fp8bw_quant_1x128_col: R=%lld and C=%lld must be positive multiples of 128",
                (long long)R, (long long)C);
  if (!aligned16(x) || !aligned16(qT) || !aligned16(s))
    return fail(FP8BW_ERR_ALIGN, "fp8bw_quant_1x128_col: pointers must be 16-byte aligned");
  if (overlaps(x, R * C * 2, qT, R * C) || overlaps(x, R * C * 2, s, R / 128 * C * 4))
    return fail(FP8BW_ERR_LAYOUT, "fp8bw_quant_1x128_col: outputs overlap the input");
  DeviceState* d;
  if (int rc = current_device(&d)) return rc;
  return launched(fp8bw::launch_quant_1x128_col(x, R, C, qT, s, as_stream(stream)), "fp8bw_quant_1x128_col");
}

FP8BW_API int fp8bw_quant_1x128_rowcol(const fp8bw_bf16* x, int64_t R, int64_t C, uint8_t* q, float* s,
                                       uint8_t* qT, float* sT, void* stream) {
  const char* name = "fp8bw_quant_1x128_rowcol";
  if (!x || !q || !s || !qT || !sT) return fail(FP8BW_ERR_NULL, "%s: x, q, s, qT and sT must be non-NULL", name);
  if (!dim_ok(R, 128) || !dim_ok(C, 128) || R / 128 > 65535)
    return fail(FP8BW_ERR_SHAPE, "%s: R=%lld and C=%lld must be positive multiples of 128", name, (long long)R,
                (long long)C);
  if (!aligned16(x) || !aligned16(q) || !aligned16(s) || !aligned16(qT) || !aligned16(sT))
    return fail(FP8BW_ERR_ALIGN, "%s: pointers must be 16-byte aligned", name);
  const int64_t n = R * C;
  if (overlaps(x, n * 2, q, n) || overlaps(x, n * 2, qT, n) || overlaps(q, n, qT, n) ||
      overlaps(x, n * 2, s, n / 32) || overlaps(x, n * 2, sT, n / 32) || overlaps(s, n / 32, sT, n / 32))
    return fail(FP8BW_ERR_LAYOUT, "%s: outputs overlap the input or each other", name);
  DeviceState* d;
  if (int rc = current_device(&d)) return rc;
  return launched(fp8bw::launch_quant_1x128_rowcol(x, R, C, q, s, qT, sT, as_stream(stream)), name);
}

FP8BW_API int fp8bw_quant_128x128(const fp8bw_bf16* w, int64_t R, int64_t C, uint8_t* q, uint8_t* qT, float* s,
                                  void* stream) {
  if (!w || !q || !s) return fail(FP8BW_ERR_NULL, "fp8bw_quant_128x128: w, q and s must be non-NULL");
  if (!dim_ok(R, 128) || !dim_ok(C, 128) || R / 128 > 65535)
    return fail(FP8BW_ERR_SHAPE, "fp8bw_quant_128x128: R=%lld and C=%lld must be positive multiples of 128",
                (long long)R, (long long)C);
  if (!aligned16(w) || !aligned16(q) || !aligned16(s) || (qT && !aligned16(qT)))
    return fail(FP8BW_ERR_ALIGN, "fp8bw_quant_128x128: pointers must be 16-byte aligned");
  const int64_t ld = FP8BW_SCALE_LD_128X128(C);
  if (overlaps(w, R * C * 2, q, R * C) || (qT && overlaps(w, R * C * 2, qT, R * C)) ||
      overlaps(w, R * C * 2, s, R / 128 * ld * 4) || (qT && overlaps(q, R * C, qT, R * C)))
    return fail(FP8BW_ERR_LAYOUT, "fp8bw_quant_128x128: outputs overlap the input or each other");
  DeviceState* d;
  if (int rc = current_device(&d)) return rc;
  return launched(fp8bw::launch_quant_128x128(w, R, C, q, qT, s, ld, as_stream(stream)), "fp8bw_quant_128x128");
}

FP8BW_API int mxfp8_quant_1x32_row(const fp8bw_bf16* x, int64_t R, int64_t C, uint8_t* q, uint8_t* e8, int mode,
                                   void* stream) {
  if (!x || !q || !e8) return fail(FP8BW_ERR_NULL, "mxfp8_quant_1x32_row: x, q and e8 must be non-NULL");
  if (!dim_ok(R, 1) || !dim_ok(C, 32) || (R + 31) / 32 > 65535)
    return fail(FP8BW_ERR_SHAPE, "mxfp8_quant_1x32_row: R=%lld must be positive, C=%lld a positive multiple of 32",
                (long long)R, (long long)C);
  if (!aligned16(x) || !aligned16(q) || !aligned16(e8))
    return fail(FP8BW_ERR_ALIGN, "mxfp8_quant_1x32_row: pointers must be 16-byte aligned");
  if (mode != FP8BW_MX_RCEIL && mode != FP8BW_MX_FLOOR)
    return fail(FP8BW_ERR_ARG, "mxfp8_quant_1x32_row: mode %d is neither RCEIL (0) nor FLOOR (1)", mode);
  if (overlaps(x, R * C * 2, q, R * C) || overlaps(x, R * C * 2, e8, R * C / 32))
    return fail(FP8BW_ERR_LAYOUT, "mxfp8_quant_1x32_row: outputs overlap the input");
  DeviceState* d;
  if (int rc = current_device(&d)) return rc;
  return launched(fp8bw::launch_mx_quant_row(x, R, C, q, e8, mode, as_stream(stream)), "mxfp8_quant_1x32_row");
}

static int mx_col_common(const char* name, const fp8bw_bf16* x, int64_t G, int64_t R, int64_t C, uint8_t* qT,
                         uint8_t* e8, int mode, void* stream) {
  if (!x || !qT || !e8) return fail(FP8BW_ERR_NULL, "%s: input, qT and e8 must be non-NULL", name);
  if (!dim_ok(G, 1) || G > 65535 || !dim_ok(R, 32) || !dim_ok(C, 8) || (R + 127) / 128 > 65535)
    return fail(FP8BW_ERR_SHAPE, "%s: the blocked dim (%lld) must be a positive multiple of 32, the other (%lld) of 8",
                name, (long long)R, (long long)C);
  if (!aligned16(x) || !aligned16(qT) || !aligned16(e8))
    return fail(FP8BW_ERR_ALIGN, "%s: pointers must be 16-byte aligned", name);
  if (mode != FP8BW_MX_RCEIL && mode != FP8BW_MX_FLOOR)
    return fail(FP8BW_ERR_ARG, "%s: mode %d is neither RCEIL (0) nor FLOOR (1)", name, mode);
  const int64_t n = G * R * C;
  if (overlaps(x, n * 2, qT, n) || overlaps(x, n * 2, e8, n / 32))
    return fail(FP8BW_ERR_LAYOUT, "%s: outputs overlap the input", name);
  DeviceState* d;
  if (int rc = current_device(&d)) return rc;
  return launched(fp8bw::launch_mx_quant_col(x, G, R, C, qT, e8, mode, as_stream(stream)), name);
}

FP8BW_API int mxfp8_quant_1x32_col(const fp8bw_bf16* x, int64_t R, int64_t C, uint8_t* qT, uint8_t* e8, int mode,
                                   void* stream) {
  return mx_col_common("mxfp8_quant_1x32_col", x, 1, R, C, qT, e8, mode, stream);
}

FP8BW_API int mxfp8_quant_3d_col(const fp8bw_bf16* w, int64_t G, int64_t N, int64_t K, uint8_t* qT, uint8_t* e8,
                                 int mode, void* stream) {
  return mx_col_common("mxfp8_quant_3d_col", w, G, N, K, qT, e8, mode, stream);
}

FP8BW_API int mxfp8_quant_1x32_rowcol(const fp8bw_bf16* x, int64_t G, int64_t R, int64_t C, uint8_t* q, uint8_t* e8,
                                      uint8_t* qT, uint8_t* e8T, int mode, void* stream) {
  const char* name = "mxfp8_quant_1x32_rowcol";
  if (!x || !q || !e8 || !qT || !e8T) return fail(FP8BW_ERR_NULL, "%s: x, q, e8, qT and e8T must be non-NULL", name);
  if (!dim_ok(G, 1) || G > 65535 || !dim_ok(R, 32) || !dim_ok(C, 32) || (R + 127) / 128 > 65535)
    return fail(FP8BW_ERR_SHAPE, "%s: G=%lld must be positive, R=%lld and C=%lld positive multiples of 32", name,
                (long long)G, (long long)R, (long long)C);
  if (!aligned16(x) || !aligned16(q) || !aligned16(e8) || !aligned16(qT) || !aligned16(e8T))
    return fail(FP8BW_ERR_ALIGN, "%s: pointers must be 16-byte aligned", name);
  if (mode != FP8BW_MX_RCEIL && mode != FP8BW_MX_FLOOR)
    return fail(FP8BW_ERR_ARG, "%s: mode %d is neither RCEIL (0) nor FLOOR (1)", name, mode);
  const int64_t n = G * R * C;
  if (overlaps(x, n * 2, q, n) || overlaps(x, n * 2, qT, n) || overlaps(q, n, qT, n) || overlaps(x, n * 2, e8, n / 32) ||
      overlaps(x, n * 2, e8T, n / 32) || overlaps(e8, n / 32, e8T, n / 32) || overlaps(q, n, e8T, n / 32) ||
      overlaps(qT, n, e8, n / 32))
    return fail(FP8BW_ERR_LAYOUT, "%s: outputs overlap the input or each other", name);
  DeviceState* d;
  if (int rc = current_device(&d)) return rc;
  return launched(fp8bw::launch_mx_quant_rowcol(x, G, R, C, q, e8, qT, e8T, mode, as_stream(stream)), name);
}

// ============================================================ blockwise GEMMs

static int gemm_common(const char* name, fp8bw::BlockwiseGemmArgs& g, void* stream) {
  void* out = g.out_acc ? static_cast<void*>(g.out_acc) : static_cast<void*>(g.out);
  const int64_t out_elem = g.out_acc ? 4 : 2;
  if (!g.a || !g.b || !g.sa || !g.sb || !out)
    return fail(FP8BW_ERR_NULL, "%s: every operand, scale and output pointer must be non-NULL", name);
  if (!dim_ok(g.Mo, 128) || !dim_ok(g.No, 256) || !dim_ok(g.Kc, 128))
    return fail(FP8BW_ERR_SHAPE,
                "%s: output rows (%lld) and the contraction (%lld) must be positive multiples of 128, output columns "
                "(%lld) of 256",
                name, (long long)g.Mo, (long long)g.Kc, (long long)g.No);
  if (!aligned16(g.a) || !aligned16(g.b) || !aligned16(g.sa) || !aligned16(g.sb) || !aligned16(out))
    return fail(FP8BW_ERR_ALIGN, "%s: pointers must be 16-byte aligned", name);
  if (overlaps(out, g.Mo * g.No * out_elem, g.a, g.Mo * g.Kc) || overlaps(out, g.Mo * g.No * out_elem, g.b, g.No * g.Kc))
    return fail(FP8BW_ERR_LAYOUT, "%s: the output overlaps an operand", name);
  DeviceState* d;
  if (int rc = current_device(&d)) return rc;
  if (!fp8bw::tensor_map_encoder()) return fail(FP8BW_ERR_CUDA, "%s: cuTensorMapEncodeTiled is unavailable", name);
  g.status = d->error_word;
  g.num_sms = d->num_sms;
  return launched(fp8bw::launch_blockwise_gemm(g, as_stream(stream)), name);
}

FP8BW_API int fp8bw_gemm_fwd(const uint8_t* xq, const float* xs, const uint8_t* wq, const float* ws, fp8bw_bf16* y,
                             int64_t M, int64_t N, int64_t K, void* stream) {
  fp8bw::BlockwiseGemmArgs g{};
  g.a = xq;
  g.b = wq;
  g.sa = xs;
  g.sa_ld = M;
  g.sb = ws;
  g.sb_ld_nb = FP8BW_SCALE_LD_128X128(K);
  g.sb_ld_kb = 1;
  g.b_scale = fp8bw::BScale::kBlock128x128;
  g.out = y;
  g.Mo = M;
  g.No = N;
  g.Kc = K;
  return gemm_common("fp8bw_gemm_fwd", g, stream);
}

FP8BW_API int fp8bw_gemm_fwd_quant(const uint8_t* xq, const float* xs, const uint8_t* wq, const float* ws,
                                   fp8bw_bf16* y, uint8_t* yq, float* ys, uint8_t* yqT, float* ysT, int64_t M,
                                   int64_t N, int64_t K, void* stream) {
  const char* name = "fp8bw_gemm_fwd_quant";
  if (!yq || !ys || (yqT == nullptr) != (ysT == nullptr))
    return fail(FP8BW_ERR_NULL, "%s: yq and ys must be non-NULL, yqT and ysT both set or both NULL", name);
  if (!aligned16(yq) || !aligned16(ys) || (yqT && (!aligned16(yqT) || !aligned16(ysT))))
    return fail(FP8BW_ERR_ALIGN, "%s: pointers must be 16-byte aligned", name);
  if (dim_ok(M, 128) && dim_ok(N, 256)) {
    const int64_t n = M * N;
    if (overlaps(y, n * 2, yq, n) || overlaps(y, n * 2, ys, n / 32) || overlaps(yq, n, ys, n / 32) ||
        (yqT && (overlaps(y, n * 2, yqT, n) || overlaps(yq, n, yqT, n) || overlaps(y, n * 2, ysT, n / 32) ||
                 overlaps(yqT, n, ysT, n / 32) || overlaps(ys, n / 32, ysT, n / 32))) ||
        overlaps(yq, n, xq, M * K) || overlaps(yq, n, wq, N * K) || (yqT && (overlaps(yqT, n, xq, M * K) ||
                                                                          overlaps(yqT, n, wq, N * K))))
      return fail(FP8BW_ERR_LAYOUT, "%s: the outputs overlap each other or an operand", name);
  }
  fp8bw::BlockwiseGemmArgs g{};
  g.a = xq;
  g.b = wq;
  g.sa = xs;
  g.sa_ld = M;
  g.sb = ws;
  g.sb_ld_nb = FP8BW_SCALE_LD_128X128(K);
  g.sb_ld_kb = 1;
  g.b_scale = fp8bw::BScale::kBlock128x128;
  g.out = y;
  g.q_out = yq;
  g.s_out = ys;
  g.qT_out = yqT;
  g.sT_out = ysT;
  g.Mo = M;
  g.No = N;
  g.Kc = K;
  return gemm_common(name, g, stream);
}

FP8BW_API int fp8bw_gemm_dgrad(const uint8_t* dyq, const float* dys, const uint8_t* wq, const uint8_t* wqT,
                               const float* ws, fp8bw_bf16* dx, int64_t M, int64_t N, int64_t K, void* stream) {
  if (!wq) return fail(FP8BW_ERR_NULL, "fp8bw_gemm_dgrad: wq must be non-NULL (wqT is the optional one)");
  if (wqT && !aligned16(wq)) return fail(FP8BW_ERR_ALIGN, "fp8bw_gemm_dgrad: pointers must be 16-byte aligned");
  fp8bw::BlockwiseGemmArgs g{};
  g.a = dyq;
  // With qT the weight is a K-major operand [K, N]; without it, W's own codes
  // [N, K] are read MN-major (contiguous along the output column k).
  g.b = wqT ? wqT : wq;
  g.b_mn_major = wqT == nullptr;
  g.sa = dys;
  g.sa_ld = M;
  g.sb = ws;
  g.sb_ld_nb = 1;                          // B rows are k: block k/128 is the column of ws
  g.sb_ld_kb = FP8BW_SCALE_LD_128X128(K);  // contraction block n/128 is the row of ws
  g.b_scale = fp8bw::BScale::kBlock128x128;
  g.out = dx;
  g.Mo = M;
  g.No = K;
  g.Kc = N;
  return gemm_common("fp8bw_gemm_dgrad", g, stream);
}

FP8BW_API int fp8bw_gemm_wgrad(const uint8_t* dyqT, const float* dysT, const uint8_t* xqT, const float* xsT,
                               fp8bw_bf16* dW, int64_t M, int64_t N, int64_t K, void* stream) {
  fp8bw::BlockwiseGemmArgs g{};
  g.a = dyqT;
  g.b = xqT;
  g.sa = dysT;
  g.sa_ld = N;
  g.sb = xsT;
  g.sb_ld_nb = 0;
  g.sb_ld_kb = K;
  g.b_scale = fp8bw::BScale::kPerRow;
  g.out = dW;
  g.Mo = N;
  g.No = K;
  g.Kc = M;
  return gemm_common("fp8bw_gemm_wgrad", g, stream);
}

FP8BW_API size_t fp8bw_gemm_wgrad_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (!dim_ok(M, 128) || !dim_ok(N, 128) || !dim_ok(K, 256)) return 0;
  int dev = -1, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return fp8bw::wgrad_split_plan(N, K, M, sms).bytes;
}

FP8BW_API int fp8bw_gemm_wgrad_ws(const uint8_t* dyqT, const float* dysT, const uint8_t* xqT, const float* xsT,
                                  fp8bw_bf16* dW, int64_t M, int64_t N, int64_t K, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  const char* name = "fp8bw_gemm_wgrad_ws";
  if (workspace && !aligned16(workspace))
    return fail(FP8BW_ERR_ALIGN, "%s: the workspace must be 16-byte aligned", name);
  fp8bw::BlockwiseGemmArgs g{};
  g.a = dyqT;
  g.b = xqT;
  g.sa = dysT;
  g.sa_ld = N;
  g.sb = xsT;
  g.sb_ld_nb = 0;
  g.sb_ld_kb = K;
  g.b_scale = fp8bw::BScale::kPerRow;
  g.out = dW;
  g.Mo = N;
  g.No = K;
  g.Kc = M;
  if (workspace && dim_ok(M, 128) && dim_ok(N, 128) && dim_ok(K, 256)) {
    DeviceState* d;
    if (int rc = current_device(&d)) return rc;
    const size_t need = fp8bw::wgrad_split_plan(N, K, M, d->num_sms).bytes;
    if (workspace_bytes < need)
      return fail(FP8BW_ERR_ARG, "%s: workspace of %zu bytes is smaller than the %zu bytes these dims need", name,
                  workspace_bytes, need);
    if (overlaps(workspace, static_cast<int64_t>(need), dW, N * K * 2) ||
        overlaps(workspace, static_cast<int64_t>(need), dyqT, N * M) ||
        overlaps(workspace, static_cast<int64_t>(need), xqT, K * M))
      return fail(FP8BW_ERR_LAYOUT, "%s: the workspace overlaps an operand or the output", name);
    g.split_ws = workspace;
    g.split_ws_bytes = workspace_bytes;
  }
  return gemm_common(name, g, stream);
}

FP8BW_API int fp8bw_gemm_wgrad_acc_f32(const uint8_t* dyqT, const float* dysT, const uint8_t* xqT, const float* xsT,
                                       float* dW, int64_t M, int64_t N, int64_t K, void* stream) {
  fp8bw::BlockwiseGemmArgs g{};
  g.a = dyqT;
  g.b = xqT;
  g.sa = dysT;
  g.sa_ld = N;
  g.sb = xsT;
  g.sb_ld_nb = 0;
  g.sb_ld_kb = K;
  g.b_scale = fp8bw::BScale::kPerRow;
  g.out = nullptr;
  g.out_acc = dW;
  g.Mo = N;
  g.No = K;
  g.Kc = M;
  return gemm_common("fp8bw_gemm_wgrad_acc_f32", g, stream);
}

// ============================================================ MXFP8 grouped GEMM

static bool grouped_dims_ok(int kind, int64_t G, int64_t M, int64_t N, int64_t K) {
  if (kind < FP8BW_GROUPED_FWD || kind > FP8BW_GROUPED_WGRAD) return false;
  const int64_t out_cols = kind == FP8BW_GROUPED_FWD ? N : K;
  return dim_ok(G, 1) && G <= 1024 && dim_ok(M, 32) && dim_ok(N, 128) && dim_ok(K, 128) && out_cols % 256 == 0 &&
         G * (kind == FP8BW_GROUPED_FWD ? N : K) <= kMaxDim;
}

FP8BW_API size_t mxfp8_grouped_gemm_workspace_bytes(int kind, int64_t G, int64_t M, int64_t N, int64_t K) {
  if (!grouped_dims_ok(kind, G, M, N, K)) return 0;
  return fp8bw::mx_grouped_gemm_workspace_bytes(kind, G, M, N, K);
}

FP8BW_API int mxfp8_grouped_gemm(int kind, const uint8_t* a, const uint8_t* a_e8, const uint8_t* b,
                                 const uint8_t* b_e8, const int32_t* group_end, int64_t G, int64_t M, int64_t N,
                                 int64_t K, fp8bw_bf16* out, void* workspace, size_t workspace_bytes, void* stream) {
  const char* name = "mxfp8_grouped_gemm";
  if (!a || !a_e8 || !b || !b_e8 || !group_end || !out || !workspace)
    return fail(FP8BW_ERR_NULL, "%s: every operand, scale, group_end, output and workspace pointer must be non-NULL",
                name);
  if (kind < FP8BW_GROUPED_FWD || kind > FP8BW_GROUPED_WGRAD)
    return fail(FP8BW_ERR_ARG, "%s: kind %d is not FWD (0), DGRAD (1) or WGRAD (2)", name, kind);
  if (!grouped_dims_ok(kind, G, M, N, K))
    return fail(FP8BW_ERR_SHAPE,
                "%s: need 0 < G <= 1024, M a multiple of 32, N and K multiples of 128 and the output column count "
                "a multiple of 256",
                name);
  if (!aligned16(a) || !aligned16(a_e8) || !aligned16(b) || !aligned16(b_e8) || !aligned16(group_end) ||
      !aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(FP8BW_ERR_ALIGN, "%s: pointers must be 16-byte aligned and the workspace 256-byte aligned", name);
  const size_t need = fp8bw::mx_grouped_gemm_workspace_bytes(kind, G, M, N, K);
  if (workspace_bytes < need)
    return fail(FP8BW_ERR_ARG, "%s: workspace of %zu bytes is smaller than the %zu bytes these dims need", name,
                workspace_bytes, need);
  DeviceState* d;
  if (int rc = current_device(&d)) return rc;
  if (!fp8bw::tensor_map_encoder()) return fail(FP8BW_ERR_CUDA, "%s: cuTensorMapEncodeTiled is unavailable", name);
  fp8bw::MxGroupedGemmArgs g{kind, a, a_e8, b, b_e8, group_end, G, M, N, K, out, workspace, workspace_bytes,
                             d->error_word, d->num_sms};
  return launched(fp8bw::launch_mx_grouped_gemm(g, as_stream(stream)), name);
}

// Same checks and launch as mxfp8_grouped_gemm, with the library's fixed
// scratch array in place of a caller workspace; nothing is allocated.
FP8BW_API int mxfp8_grouped_gemm_noalloc(int kind, const uint8_t* a, const uint8_t* a_e8, const uint8_t* b,
                                         const uint8_t* b_e8, const int32_t* group_end, int64_t G, int64_t M,
                                         int64_t N, int64_t K, fp8bw_bf16* out, void* stream) {
  const char* name = "mxfp8_grouped_gemm_noalloc";
  if (!a || !a_e8 || !b || !b_e8 || !group_end || !out)
    return fail(FP8BW_ERR_NULL, "%s: every operand, scale, group_end and output pointer must be non-NULL", name);
  if (kind < FP8BW_GROUPED_FWD || kind > FP8BW_GROUPED_WGRAD)
    return fail(FP8BW_ERR_ARG, "%s: kind %d is not FWD (0), DGRAD (1) or WGRAD (2)", name, kind);
  if (!grouped_dims_ok(kind, G, M, N, K))
    return fail(FP8BW_ERR_SHAPE,
                "%s: need 0 < G <= 1024, M a multiple of 32, N and K multiples of 128 and the output column count "
                "a multiple of 256",
                name);
  const size_t need = fp8bw::mx_grouped_gemm_workspace_bytes(kind, G, M, N, K);
  if (need > fp8bw::kStaticScratchBytes)
    return fail(FP8BW_ERR_SHAPE, "%s: these dims need %zu bytes of scratch, more than the fixed %zu-byte array",
                name, need, fp8bw::kStaticScratchBytes);
  if (!aligned16(a) || !aligned16(a_e8) || !aligned16(b) || !aligned16(b_e8) || !aligned16(group_end) ||
      !aligned16(out))
    return fail(FP8BW_ERR_ALIGN, "%s: pointers must be 16-byte aligned", name);
  DeviceState* d;
  if (int rc = current_device(&d)) return rc;
  if (!fp8bw::tensor_map_encoder()) return fail(FP8BW_ERR_CUDA, "%s: cuTensorMapEncodeTiled is unavailable", name);
  void* scratch = nullptr;
  cudaError_t e = fp8bw::static_scratch_address(&scratch);
  if (e != cudaSuccess)
    return fail(FP8BW_ERR_CUDA, "%s: resolving the scratch array's device address: %s", name, cudaGetErrorString(e));
  fp8bw::MxGroupedGemmArgs g{kind, a, a_e8, b, b_e8, group_end, G, M, N, K, out, scratch,
                             fp8bw::kStaticScratchBytes, d->error_word, d->num_sms};
  return launched(fp8bw::launch_mx_grouped_gemm(g, as_stream(stream)), name);
}

// ============================================================ status

FP8BW_API int fp8bw_sync_status(void* stream) {
  DeviceState* d;
  if (int rc = current_device(&d)) return rc;
  cudaError_t e = cudaStreamSynchronize(as_stream(stream));
  if (e != cudaSuccess) return fail(FP8BW_ERR_CUDA, "fp8bw_sync_status: %s", cudaGetErrorString(e));
  int word = 0;
  e = cudaMemcpyFromSymbol(&word, g_error_word, sizeof(int));
  if (e != cudaSuccess) return fail(FP8BW_ERR_CUDA, "fp8bw_sync_status: reading the error word: %s", cudaGetErrorString(e));
  if (word != 0) {
    const int zero = 0;
    cudaMemcpyToSymbol(g_error_word, &zero, sizeof(int));
    if (word == FP8BW_ERR_TIMEOUT) return fail(FP8BW_ERR_TIMEOUT, "a bounded device-side wait expired");
    return fail(word, "a kernel reported error %d (a device-side argument check failed)", word);
  }
  return ok();
}

FP8BW_API const char* fp8bw_last_error(void) { return g_msg; }

FP8BW_API int fp8bw_selftest_bounded_wait(uint32_t timeout_us, void* stream) {
  if (timeout_us < 1 || timeout_us > 2000000)
    return fail(FP8BW_ERR_ARG, "fp8bw_selftest_bounded_wait: timeout_us=%u outside [1, 2000000]", timeout_us);
  DeviceState* d;
  if (int rc = current_device(&d)) return rc;
  return launched(fp8bw::launch_selftest_bounded_wait(timeout_us, d->error_word, as_stream(stream)),
                  "fp8bw_selftest_bounded_wait");
}
