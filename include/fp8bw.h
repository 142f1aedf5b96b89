/*
 * fp8bw.h -- C ABI of libfp8bw.so: blockwise-FP8 and MXFP8 linear-layer
 * training kernels for NVIDIA GB300 (sm_103a).
 *
 * What the calls compute follows three pull-request pages of pytorch/ao:
 *   [PR2386] "[not for land] float8 blockwise scaling training prototype using
 *            deep_gemm" -- description ("What I saw", "path forward");
 *   [PR3037] "[mxfp8 moe training] use new 3d colwise quantization kernel" --
 *            Summary, Microbenchmarks table;
 *   [PR4295] "add FSDP and TP tests for Float8BlockwiseLinear" -- Summary and
 *            the review threads on EPS, BlockWise1x128 scaling,
 *            _pad_blockwise_128x128_scale_k_major and the layout assertions.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every pointer is a DEVICE pointer on the current CUDA device, allocated and
 *   owned by the caller.  The library never allocates device memory, never
 *   frees caller memory and keeps no per-call state (a 4-byte error word per
 *   device, see fp8bw_sync_status, and the fixed scratch array of
 *   mxfp8_grouped_gemm_noalloc are its only globals).  Their device addresses
 *   are resolved on a device's first call and cached; calls on a device after
 *   cudaDeviceReset are not supported.
 * - Every pointer must be 16-byte aligned.  Matrices are dense and row-major
 *   with the leading dimension equal to the row length given.
 * - bf16 tensors are passed as raw 16-bit patterns (fp8bw_bf16); e4m3 codes
 *   and E8M0 bytes as uint8_t.
 * - Work is enqueued asynchronously on `stream` (a cudaStream_t passed as
 *   void*; NULL is the legacy default stream).  A return of FP8BW_OK means
 *   the arguments were valid and the kernel was launched.
 * - Arguments are checked before anything touches the GPU, in this order:
 *   null pointers, shapes, alignment, enum arguments, then the device
 *   (compute capability 10.3 is required).  A layout the kernels do not
 *   take is an error, never a silent copy ([PR4295], layout-assertion thread).
 * - On error the call returns a nonzero FP8BW_ERR_* code and
 *   fp8bw_last_error() holds a message for the calling thread.
 *
 * Scale rule (blockwise calls): for each block, amax = max |x| (exact in
 * fp32), s = fl32(max(amax, 1e-12f) / 448.0f) -- 1e-12 is the EPS of
 * [PR4295], 448 the largest finite e4m3 value -- and each element is stored
 * as q = e4m3_rn_satfinite(fl32(x / s)) with an IEEE float32 division.
 * Results are bit-identical to that definition.
 *
 * Scale rule (MXFP8 calls, blocks of 32): E = smallest integer with
 * 448 * 2^E >= amax (mode FP8BW_MX_RCEIL) or E = floor(log2 amax) - 8 (mode
 * FP8BW_MX_FLOOR), clamped to [-127, 127], E = -127 for an all-zero block;
 * the byte stored is E + 127 and q = e4m3_rn_satfinite(fl32(x * 2^-E)).
 */
#ifndef FP8BW_H
#define FP8BW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t fp8bw_bf16;

enum fp8bw_status {
  FP8BW_OK = 0,
  FP8BW_ERR_NULL = 1,        /* a required pointer is NULL */
  FP8BW_ERR_SHAPE = 2,       /* a dim <= 0, too large, or not a multiple of its block */
  FP8BW_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned */
  FP8BW_ERR_LAYOUT = 4,      /* operands that alias or a layout the kernel does not take */
  FP8BW_ERR_UNSUPPORTED = 5, /* no CUDA device, or its compute capability is not 10.3 */
  FP8BW_ERR_CUDA = 6,        /* a CUDA runtime/driver call or a launch failed */
  FP8BW_ERR_TIMEOUT = 7,     /* a bounded device-side wait expired (fp8bw_sync_status) */
  FP8BW_ERR_ARG = 8          /* an enum argument (mode, kind) is out of range */
};

/* Row stride, in floats, of the 128x128 scale array of a [R, C] weight:
 * ceil(C/128) rounded up to a multiple of 4, so each row of scales starts on
 * a 16-byte boundary (the K-stride padding of [PR4295]'s
 * _pad_blockwise_128x128_scale_k_major thread). */
#define FP8BW_SCALE_LD_128X128(C) ((((C) / 128) + 3) / 4 * 4)

/* ---------------------------------------------------------------------------
 * Blockwise e4m3 quantizers (fp32 scales).
 * ------------------------------------------------------------------------- */

/* 1x128 rowwise ("BlockWise1x128", [PR4295] scaling-type thread): blocks of
 * 128 consecutive elements of each row of x[R, C].  Forward operand x and the
 * dgrad operand dy.
 *   x : bf16 [R, C]          q : e4m3 [R, C]          s : fp32 [C/128][R]
 * R and C must be positive multiples of 128. */
int fp8bw_quant_1x128_row(const fp8bw_bf16* x, int64_t R, int64_t C,
                          uint8_t* q, float* s, void* stream);

/* 1x128 colwise: blocks of 128 consecutive ROWS of each column of x[R, C],
 * written transposed so the contraction over R is contiguous: the operands of
 * the grad_weight GEMM ([PR2386] "128_1_128_1" case).
 *   x : bf16 [R, C]          qT : e4m3 [C, R]         s : fp32 [R/128][C]
 * R and C must be positive multiples of 128. */
int fp8bw_quant_1x128_col(const fp8bw_bf16* x, int64_t R, int64_t C,
                          uint8_t* qT, float* s, void* stream);

/* Both 1x128 quantizations of x[R, C] from one read of x: exactly the outputs
 * of fp8bw_quant_1x128_row (q, s) and of fp8bw_quant_1x128_col (qT, sT).  The
 * training step needs both for x (forward and grad_weight) and for dy (dgrad
 * and grad_weight); one pass moves 2 + 2 + 8/128 bytes per element instead
 * of 2 x (2 + 1 + 4/128).
 *   x : bf16 [R, C]   q : e4m3 [R, C]   s : fp32 [C/128][R]
 *                     qT : e4m3 [C, R]  sT : fp32 [R/128][C]
 * R and C must be positive multiples of 128. */
int fp8bw_quant_1x128_rowcol(const fp8bw_bf16* x, int64_t R, int64_t C,
                             uint8_t* q, float* s, uint8_t* qT, float* sT, void* stream);

/* 128x128 weight quantization in one pass ([PR2386] "What I saw": 128x128
 * scaling of one tensor, and "path forward" item 2, a handwritten kernel).
 *   w : bf16 [R, C]   q : e4m3 [R, C]   qT : e4m3 [C, R] or NULL
 *   s : fp32 [R/128][FP8BW_SCALE_LD_128X128(C)] (padding columns untouched)
 * qT, when given, holds the same codes transposed; fp8bw_gemm_dgrad can take
 * it instead of reading q transposed.
 * R and C must be positive multiples of 128. */
int fp8bw_quant_128x128(const fp8bw_bf16* w, int64_t R, int64_t C,
                        uint8_t* q, uint8_t* qT, float* s, void* stream);

/* ---------------------------------------------------------------------------
 * Blockwise-scaled GEMMs of Float8BlockwiseLinear forward and backward
 * ([PR2386] description: fwd and bwd GEMMs of a dense linear; [PR4295]
 * Summary).  Each accumulates every 128-deep contraction block in fp32 on the
 * tensor cores, multiplies it by the product of the two blocks' scales and
 * sums the blocks in fp32; the result is rounded once to bf16.  Accuracy:
 * |out - exact| <= 2e-3 * ||a_i|| * ||b_j|| per element, a_i and b_j the
 * dequantized contraction vectors.  M, N, K positive multiples of 128 with N
 * (the output's column count) a multiple of 256.
 * ------------------------------------------------------------------------- */

/* y = x W^T  ("128_1_128_128": x in 1x128 blocks, W in 128x128 blocks).
 *   xq : e4m3 [M, K]   xs : fp32 [K/128][M]          (fp8bw_quant_1x128_row of x)
 *   wq : e4m3 [N, K]   ws : fp32 [N/128][LD(K)]      (fp8bw_quant_128x128 of W)
 *   y  : bf16 [M, N]
 * Requires N % 256 == 0. */
int fp8bw_gemm_fwd(const uint8_t* xq, const float* xs, const uint8_t* wq, const float* ws,
                   fp8bw_bf16* y, int64_t M, int64_t N, int64_t K, void* stream);

/* y = x W^T as fp8bw_gemm_fwd, plus, from the same output tiles, the 1x128
 * rowwise quantization of bf16(y) and optionally its colwise one -- the
 * quantized operands the next linear's forward and grad_weight GEMMs take,
 * without reading y back.  Bit-identical to fp8bw_gemm_fwd followed by
 * fp8bw_quant_1x128_row (or fp8bw_quant_1x128_rowcol) of y.  Each 128 x 256
 * output tile holds whole 1x128 row blocks and, its 128 rows being one token
 * block, whole colwise blocks, so the epilogue that writes y quantizes it too.
 * The pages run every scaling as kernels of their own ([PR2386] "What I saw":
 * 128x128 scaling of one tensor takes three kernels) and leave performance
 * work open ("path forward" item 3); this call is such work, not a step the
 * pages define.
 *   xq, xs, wq, ws, y : as fp8bw_gemm_fwd
 *   yq  : e4m3 [M, N]   ys  : fp32 [N/128][M]      (required)
 *   yqT : e4m3 [N, M]   ysT : fp32 [M/128][N]      (both or neither NULL)
 * Requires N % 256 == 0. */
int fp8bw_gemm_fwd_quant(const uint8_t* xq, const float* xs, const uint8_t* wq, const float* ws,
                         fp8bw_bf16* y, uint8_t* yq, float* ys, uint8_t* yqT, float* ysT,
                         int64_t M, int64_t N, int64_t K, void* stream);

/* dx = dy W  (dy in 1x128 blocks along N, W in 128x128 blocks).
 *   dyq : e4m3 [M, N]   dys : fp32 [N/128][M]        (fp8bw_quant_1x128_row of dy)
 *   wq  : e4m3 [N, K]   ws  : fp32 [N/128][LD(K)]    (q and s of fp8bw_quant_128x128 of W)
 *   wqT : e4m3 [K, N] or NULL                         (its qT, optional)
 *   dx  : bf16 [M, K]
 * The contraction runs over W's rows.  Without wqT the kernel reads W's codes
 * as stored, contiguous along the output column (the tensor core's transposed
 * B operand), so the weight quantizer need not write qT; with wqT it reads
 * the transposed copy.  Both give the same result.  wq must be non-NULL.
 * Requires K % 256 == 0. */
int fp8bw_gemm_dgrad(const uint8_t* dyq, const float* dys, const uint8_t* wq, const uint8_t* wqT,
                     const float* ws, fp8bw_bf16* dx, int64_t M, int64_t N, int64_t K, void* stream);

/* dW = dy^T x  ("128_1_128_1": both operands in 1x128 blocks along tokens M).
 *   dyqT : e4m3 [N, M]   dysT : fp32 [M/128][N]      (fp8bw_quant_1x128_col of dy)
 *   xqT  : e4m3 [K, M]   xsT  : fp32 [M/128][K]      (fp8bw_quant_1x128_col of x)
 *   dW   : bf16 [N, K]
 * Requires K % 256 == 0. */
int fp8bw_gemm_wgrad(const uint8_t* dyqT, const float* dysT, const uint8_t* xqT, const float* xsT,
                     fp8bw_bf16* dW, int64_t M, int64_t N, int64_t K, void* stream);

/* fp8bw_gemm_wgrad with a caller workspace that lets the kernel balance its
 * last round of output tiles: when the tile count is not a multiple of the
 * SM count, the remaining tiles are each cut into k contraction parts that
 * run side by side, and the part that finishes last for a region adds the k
 * fp32 partials in part order (so the result does not depend on which part
 * finishes last) and rounds once to bf16.  The result equals
 * fp8bw_gemm_wgrad's within the GEMM accuracy above; the partials are summed
 * in a different order, so bits may differ.  (The pages' wgrad runs over the
 * whole token dimension in one GEMM, [PR2386] "128_1_128_1"; the split is
 * scheduling work, not a step the pages define.)
 * workspace: DEVICE memory of at least fp8bw_gemm_wgrad_workspace_bytes(M, N,
 * K) bytes, 16-byte aligned, owned by the caller; NULL (or a size of 0 from
 * that query) runs fp8bw_gemm_wgrad unchanged.  Calls that use the same
 * workspace concurrently race.  Other arguments as fp8bw_gemm_wgrad. */
int fp8bw_gemm_wgrad_ws(const uint8_t* dyqT, const float* dysT, const uint8_t* xqT, const float* xsT,
                        fp8bw_bf16* dW, int64_t M, int64_t N, int64_t K, void* workspace,
                        size_t workspace_bytes, void* stream);

/* Bytes of workspace fp8bw_gemm_wgrad_ws uses for these dims on the current
 * device: 0 when splitting the last round of tiles would not pay (for one,
 * when the tiles fill whole rounds of SMs), or when the dims are invalid or
 * no device is present.  Enqueues no work. */
size_t fp8bw_gemm_wgrad_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* dW += dy^T x with dW in fp32: the wgrad GEMM above, its tile added to the
 * caller's fp32 gradient instead of overwriting a bf16 one -- gradient
 * accumulation over micro-batches or token shards, whose sum the optimizer
 * step consumes (PR #4295 "Testing": gradients compared after the expected
 * reduction, parameters after the optimizer step; PR #2386: grad_weight of
 * the 128_1_128_1 GEMM).  Arguments as fp8bw_gemm_wgrad; dW : fp32 [N, K],
 * read and written, 16-byte aligned, owned by the caller.  Each element
 * receives one fp32 addition of its fp32-promoted tile value.  Calls that
 * write the same dW must be ordered on one stream. */
int fp8bw_gemm_wgrad_acc_f32(const uint8_t* dyqT, const float* dysT, const uint8_t* xqT, const float* xsT,
                             float* dW, int64_t M, int64_t N, int64_t K, void* stream);

/* ---------------------------------------------------------------------------
 * MXFP8: 1x32 blocks, E8M0 scales, e4m3 data ([PR3037] MoEScalingType.MXFP8).
 * ------------------------------------------------------------------------- */

enum fp8bw_mx_mode { FP8BW_MX_RCEIL = 0, FP8BW_MX_FLOOR = 1 };

/* Rowwise 1x32 along C.  x : bf16 [R, C]  q : e4m3 [R, C]  e8 : u8 [R][C/32].
 * R > 0, C a positive multiple of 32. */
int mxfp8_quant_1x32_row(const fp8bw_bf16* x, int64_t R, int64_t C,
                         uint8_t* q, uint8_t* e8, int mode, void* stream);

/* Colwise 1x32 along R, written transposed.  x : bf16 [R, C]
 * qT : e4m3 [C, R]  e8 : u8 [C][R/32].  R a positive multiple of 32,
 * C a positive multiple of 8. */
int mxfp8_quant_1x32_col(const fp8bw_bf16* x, int64_t R, int64_t C,
                         uint8_t* qT, uint8_t* e8, int mode, void* stream);

/* 3D colwise quantization of expert weights ([PR3037] Summary): for each
 * expert g, 32-blocks along N of w[g] : [N, K], written transposed.
 *   w : bf16 [G, N, K]   qT : e4m3 [G, K, N]   e8 : u8 [G][K][N/32]
 * G > 0, N a positive multiple of 32, K a positive multiple of 8. */
int mxfp8_quant_3d_col(const fp8bw_bf16* w, int64_t G, int64_t N, int64_t K,
                       uint8_t* qT, uint8_t* e8, int mode, void* stream);

/* Both MX quantizations of G stacked matrices x [G, R, C] from one read of
 * x: the rowwise one (1x32 blocks along C) and the colwise one (32-row
 * blocks along R, written transposed per matrix).  Byte-identical to
 * mxfp8_quant_1x32_row on x viewed as [G*R, C] plus mxfp8_quant_1x32_col of
 * each matrix (G = 1: a 2D operand such as x or dy of the MoE step) or
 * mxfp8_quant_3d_col (G experts: W as [G, N, K], R = N, C = K).  On the
 * pages the 3D colwise quantization is a kernel of its own ([PR3037]
 * Summary: the new CUDA kernel in the grouped-mm backward); reading the
 * input once for both outputs is performance work, not a step the pages
 * define.
 *   x   : bf16 [G, R, C]
 *   q   : e4m3 [G*R, C]        e8  : E8M0 [G*R][C/32]
 *   qT  : e4m3 [G, C, R]       e8T : E8M0 [G][C][R/32]
 * G >= 1; R and C positive multiples of 32. */
int mxfp8_quant_1x32_rowcol(const fp8bw_bf16* x, int64_t G, int64_t R, int64_t C, uint8_t* q, uint8_t* e8,
                            uint8_t* qT, uint8_t* e8T, int mode, void* stream);

enum fp8bw_grouped_kind { FP8BW_GROUPED_FWD = 0, FP8BW_GROUPED_DGRAD = 1, FP8BW_GROUPED_WGRAD = 2 };

/* MoE grouped GEMM on MXFP8 operands ([PR3037] Microbenchmarks: grouped mm
 * forward and backward).  The dims are those of the MoE linear: M tokens split
 * into G groups, K input and N output features per expert.  group_end is a
 * DEVICE int32 array [G] of cumulative token counts: group g owns tokens
 * [group_end[g-1], group_end[g]) with group_end[-1] = 0; sizes must be
 * multiples of 32 (empty groups allowed) and group_end[G-1] == M.  The kernel
 * clamps every range into [0, M] (ends rounded down to multiples of 32) and
 * raises FP8BW_ERR_SHAPE through fp8bw_sync_status when group_end breaks these
 * rules.
 *   FWD   : a = xq [M, K], a_e8 [M][K/32]; b = wq [G, N, K], b_e8 [G*N][K/32]
 *           (mxfp8_quant_1x32_row of x and of w viewed as [G*N, K]);
 *           out = y bf16 [M, N]
 *   DGRAD : a = dyq [M, N], a_e8 [M][N/32]; b = wqT [G, K, N], b_e8 [G][K][N/32]
 *           (mxfp8_quant_3d_col of w); out = dx bf16 [M, K]
 *   WGRAD : a = dyqT [N, M], a_e8 [N][M/32]; b = xqT [K, M], b_e8 [K][M/32]
 *           (mxfp8_quant_1x32_col of dy and x); out = dW bf16 [G, N, K];
 *           an empty group's dW is written as zeros.
 * workspace: caller-owned DEVICE scratch of at least
 * mxfp8_grouped_gemm_workspace_bytes(kind, G, M, N, K) bytes, 256-byte
 * aligned.  The call first rewrites the scale bytes into it, in the layout the
 * tensor core's scale-factor copy consumes, then runs the GEMM; calls that use
 * the same workspace concurrently (on different streams) race.
 * Requirements: M multiple of 32, N and K multiples of 128, and the output
 * column count (N for FWD, K for DGRAD and WGRAD) a multiple of 256. */
int mxfp8_grouped_gemm(int kind, const uint8_t* a, const uint8_t* a_e8,
                       const uint8_t* b, const uint8_t* b_e8, const int32_t* group_end,
                       int64_t G, int64_t M, int64_t N, int64_t K,
                       fp8bw_bf16* out, void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace mxfp8_grouped_gemm needs for these dims (0 if the dims
 * or kind are invalid).  Host-only; touches no GPU. */
size_t mxfp8_grouped_gemm_workspace_bytes(int kind, int64_t G, int64_t M, int64_t N, int64_t K);

/* Largest scratch, in bytes, mxfp8_grouped_gemm_noalloc can use. */
#define FP8BW_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/* mxfp8_grouped_gemm for callers that cannot allocate device memory: code that
 * only receives device pointers from a framework owning every allocation
 * (its caching allocator), or a training/serving loop whose device footprint
 * is fixed before the first step.  It computes exactly what
 * mxfp8_grouped_gemm computes, with the same arguments minus the workspace;
 * the scratch lives in a fixed array of FP8BW_NOALLOC_SCRATCH_BYTES (16 MiB)
 * inside the library, which every GPU that loads the library holds until the
 * process exits.  The pages describe nothing like it; it is an addition for
 * such callers.
 * - Dims whose mxfp8_grouped_gemm_workspace_bytes exceeds that size are
 *   rejected with FP8BW_ERR_SHAPE and a message naming both sizes.
 * - The first call on a device resolves the array's device address for that
 *   device (with that device current); make that first call before any stream
 *   capture.  No call allocates or frees device memory.
 * - That address is cached per device for the life of the process.  After
 *   cudaDeviceReset it no longer names the array (the library's device image
 *   is loaded again), so do not call the library on a device after resetting
 *   it; the same holds for every entry point, whose error word address is
 *   cached the same way.
 * - Every call on a device shares the one array and leaves its contents
 *   behind; each call rewrites all of the scratch it reads, so nothing needs
 *   to start at zero.  Calls whose executions overlap on the GPU (different
 *   streams, same device) race on the array and give wrong results. */
int mxfp8_grouped_gemm_noalloc(int kind, const uint8_t* a, const uint8_t* a_e8,
                               const uint8_t* b, const uint8_t* b_e8, const int32_t* group_end,
                               int64_t G, int64_t M, int64_t N, int64_t K,
                               fp8bw_bf16* out, void* stream);

/* ---------------------------------------------------------------------------
 * Status.
 * ------------------------------------------------------------------------- */

/* Synchronizes `stream`, then reads and clears the current device's error
 * word, which kernels set when a bounded wait expires (FP8BW_ERR_TIMEOUT) or
 * a device-side argument check fails (FP8BW_ERR_SHAPE).  Returns FP8BW_OK,
 * that code, or FP8BW_ERR_CUDA if the synchronization itself failed. */
int fp8bw_sync_status(void* stream);

/* Message of the calling thread's last error ("" if none).  The pointer stays
 * valid until the thread's next call into the library. */
const char* fp8bw_last_error(void);

/* Launches one block whose single thread waits, through the same bounded
 * wait the GEMM pipelines use, on a barrier nothing will ever signal, for
 * `timeout_us` microseconds (1 .. 2,000,000), then records FP8BW_ERR_TIMEOUT
 * in the error word and returns.  It lets a test observe the timeout path
 * without faulting or hanging the GPU. */
int fp8bw_selftest_bounded_wait(uint32_t timeout_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8BW_H */
