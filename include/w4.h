/*
 * w4.h — C ABI of libw4, a GB300 (sm_103a) 4-bit-weight mixed-precision GEMM.
 *
 *   out[M,N] = a[M,K] x dequant(W)[K,N]
 *
 * W holds 4-bit weights.  Three modes:
 *   W4A16 symmetric : uint4b8 nibbles (value q-8), fp16/bf16 group scales.
 *   W4A16 asymmetric: uint4 nibbles (value q) with pre-scaled zero-points.
 *   W4A8 (QQQ style): int4 weights, int8 activations with per-token fp32
 *                     scales, per-channel fp32 weight scales, optional int8
 *                     per-group (g128) weight scales.
 *
 * Sources (web pages, cited by title and section):
 *   [MR]  Machete Readme, "Machete (Mixed Precision Cutlass-Based GEMM)":
 *         "Overview" (the dequant formula, w_z pre-scaled so the step is one
 *         FMA), "API" (prepack the weights to a tensor-core-friendly layout,
 *         then call the GEMM with b_type, b_scales, b_group_size),
 *         "Code Generation" (schedules chosen by a default heuristic, with an
 *         optional `schedule` override).
 *   [PR9855] vLLM PR #9855 "[Kernel] Initial Machete W4A8 support +
 *         Refactors": QQQ-style W4A8; uint4b8 and uint4 share one prepack
 *         because prepacking only moves data.
 *   [RDNA] vLLM API page "rdna_hybrid_w4a16": ExLlama shuffle packing
 *         (pack_int4_exllama_shuffle), ZP_BIAS 8, the argument checks of
 *         triton_w4a16_skinny_fmt_gemm (contiguity, shapes, group_size -1
 *         meaning K).
 *   [QQQ] pytorch/ao PR #1113 "support W4A8 Marlin kernel": W4A8 per-channel
 *         and per-group (g128), symmetric weights only, fp16 output only.
 *   [PT]  vLLM PR #6547 "Enable Dynamic Per Token fp8": per-token activation
 *         scales applied in the GEMM epilogue.
 *
 * Conventions for every entry point:
 *   - All matrices are dense, contiguous, row-major, in DEVICE memory owned
 *     by the caller.  The library allocates no memory and keeps no pointer
 *     after a call returns.
 *   - Every array must be aligned to its element size (2 bytes for fp16 /
 *     bf16, 4 for fp32 / int32), and the prepacked weights and packed int32
 *     words to 4 bytes; a misaligned pointer is W4_ERR_INVALID_ARGUMENT.
 *     The tensor-core and streamed GEMM schedules also want a, b_packed,
 *     b_scales and b_zeros 16-byte aligned: without that the default
 *     heuristic runs the CUDA-core schedule, and an explicit schedule
 *     returns W4_ERR_UNSUPPORTED.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued on it; calls return after enqueue.
 *   - Argument errors are reported synchronously, before anything is
 *     enqueued; w4_last_error() then holds a one-line message.  The library
 *     never aborts the process and its kernels never trap.
 */
#ifndef W4_H_
#define W4_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum w4_status {
  W4_OK = 0,
  W4_ERR_INVALID_ARGUMENT = 1, /* null pointer, bad enum, bad shape or group size */
  W4_ERR_UNSUPPORTED = 2,      /* well-formed, but outside what the kernels tile */
  W4_ERR_WORKSPACE = 3,        /* workspace missing or smaller than required */
  W4_ERR_CUDA = 4,             /* a CUDA runtime call or launch failed */
  W4_ERR_TIMEOUT = 5           /* a device-side wait gave up (w4_check_status) */
} w4_status;

/* Weight types ([PR9855] summary; [RDNA] ZP_BIAS; [QQQ] symmetric int4). */
typedef enum w4_wtype {
  W4_UINT4B8 = 0, /* stored q in 0..15, value q - 8 */
  W4_UINT4 = 1,   /* stored q in 0..15, value q (use with zero-points) */
  W4_INT4 = 2     /* two's complement nibble, value in -8..7 */
} w4_wtype;

/* Input layouts of the packed int32 weights (8 nibbles per word, K packed). */
typedef enum w4_layout {
  W4_LAYOUT_KN_SEQ = 0,    /* [K/8][N] words, K-value j of a word at bits 4j */
  W4_LAYOUT_NK_SEQ = 1,    /* [N][K/8] words, K-value j at bits 4j */
  W4_LAYOUT_NK_EXLLAMA = 2 /* [N][K/8] words, ExLlama order [0,2,4,6,1,3,5,7]:
                              K-value j at bits (j/2)*4 + (j%2)*16 ([RDNA]) */
} w4_layout;

/* Element types.  W4_E4M3: OCP fp8 E4M3 activations (bias 7, largest value
 * 448, S.1111.111 NaN), one byte each ([PR9855]: W4A8 "including fp8
 * activations"). */
typedef enum w4_dtype { W4_F16 = 0, W4_BF16 = 1, W4_S8 = 2, W4_S32 = 3, W4_E4M3 = 4 } w4_dtype;

/* Version of the prepacked weight layout produced by w4_prepack_B.  A
 * buffer prepacked under one version must not be used with another. */
int w4_layout_version(void);

/* Bytes of the prepacked buffer for a K x N weight: ceil(N/128)*128 * K/2.
 * Returns 0 for K <= 0, N <= 0 or K % 64 != 0. */
size_t w4_prepacked_size(int64_t K, int64_t N);

/* Rearrange packed 4-bit weights into the tensor-core tile order ([MR] API:
 * "prepacking the weight matrix to more closely match the tensor core
 * layouts").  w_q: int32 words in `in_layout` (device).  b_packed: device
 * buffer of w4_prepacked_size(K, N) bytes, written in full (padding rows
 * zeroed).  uint4 and uint4b8 prepack identically ([PR9855]); int4 nibbles
 * are stored with their top bit flipped (offset binary, value q' - 8).
 * Errors: INVALID_ARGUMENT for null pointers, bad enums, K % 8 != 0,
 * K <= 0 or N <= 0; UNSUPPORTED for K % 64 != 0. */
w4_status w4_prepack_B(const int32_t* w_q, int wtype, int in_layout, int64_t K, int64_t N,
                       void* b_packed, void* stream);

/* Inverse of w4_prepack_B (for tests and tooling): writes w_q in
 * `out_layout` from a prepacked buffer with the same wtype, K and N. */
w4_status w4_unprepack_B(const void* b_packed, int wtype, int out_layout, int64_t K, int64_t N,
                         int32_t* w_q, void* stream);

/* Workspace bytes w4_gemm needs for this problem under any schedule
 * (always >= 256).  The workspace holds a status word, split-K tile
 * counters and partial sums, and (W4A8) a bf16 copy of the activations.
 * It must be zero-filled before its first use; every call leaves its
 * counters at zero again.  Calls that share a workspace must not overlap
 * on the GPU. */
size_t w4_gemm_workspace_size(int64_t M, int64_t N, int64_t K, int a_type, int64_t group_size);

/* out = a x dequant(W)  ([MR] Overview and API; [QQQ]; [PT]).
 *
 *   a         [M,K] activations: W4_F16 / W4_BF16 (W4A16) or W4_S8 (W4A8).
 *   b_packed  output of w4_prepack_B for this K, N and wtype.
 *   group_size  a multiple of 64 that divides K, or -1 / K for one group
 *             per column ([RDNA]: -1 resolves to K).  G = K / group_size.
 *   W4A16: b_scales [G,N] with scale_type == a_type; b_zeros [G,N] of the
 *          same type holding PRE-SCALED zero-points w_z, or NULL.
 *          w_hat[k][n] = v(q) * s[g][n] - w_z[g][n], rounded once to the
 *          activation type (one fused multiply-add, [MR] Overview NOTE);
 *          out = sum_k a*w_hat accumulated in fp32, rounded to out_type,
 *          which must equal a_type.  a_token_scales and ch_scales NULL.
 *   W4A8:  wtype W4_INT4 or W4_UINT4B8 (symmetric only, [QQQ]); b_zeros
 *          NULL; b_scales = int8 group scales sg [G,N] (scale_type W4_S8)
 *          for per-group, or NULL for per-channel (group_size -1 or K).
 *          The integer weight v*sg must lie in [-128,127] (sg in 1..16).
 *          acc = sum_k a*v*sg exactly in int32 (|acc| < 2^31 required).
 *          out_type W4_F16: out = fp16_rn((float)acc * s_tok[m] * s_ch[n]),
 *          multiplied left to right in fp32, with a_token_scales = s_tok [M]
 *          and ch_scales = s_ch [N] (fp32, device).
 *          out_type W4_S32: out = acc, both scale pointers NULL.
 *   W4A8 with fp8 activations (a_type W4_E4M3): per-channel only (b_scales
 *          NULL, group_size -1 / K), K a multiple of 128, fp16 output:
 *          out = fp16_rn(acc * s_tok[m] * s_ch[n]) with acc the fp32 sum of
 *          the exact products decode(a) * v(q) (every int4 value is an E4M3
 *          value); NaN codes (0x7F, 0xFF) are outside the contract.
 *   workspace  device buffer of at least w4_gemm_workspace_size(...) bytes,
 *             16-byte aligned (W4_ERR_WORKSPACE otherwise).
 *
 * M == 0 is a no-op; K == 0 writes zeros.  Errors: INVALID_ARGUMENT
 * (null required pointer, dtype mismatch, K % 8 != 0, group_size not
 * dividing K, negative sizes), UNSUPPORTED (K % 64 != 0, group_size not a
 * multiple of 64, W4A8 with zero-points, uint4 or a non-fp16/int32 output),
 * WORKSPACE, CUDA. */
w4_status w4_gemm(const void* a, int a_type, int64_t M, int64_t K, const void* b_packed,
                  int wtype, int64_t N, const void* b_scales, int scale_type,
                  const void* b_zeros, int64_t group_size, const float* a_token_scales,
                  const float* ch_scales, void* out, int out_type, void* workspace,
                  size_t workspace_bytes, void* stream);

/* w4_gemm with an explicit schedule ([MR] Code Generation: the optional
 * `schedule` argument).  schedule < 0 means the default heuristic;
 * otherwise an index in [0, w4_num_schedules()).  A schedule that cannot
 * run this problem returns UNSUPPORTED. */
w4_status w4_gemm_ex(const void* a, int a_type, int64_t M, int64_t K, const void* b_packed,
                     int wtype, int64_t N, const void* b_scales, int scale_type,
                     const void* b_zeros, int64_t group_size, const float* a_token_scales,
                     const float* ch_scales, void* out, int out_type, void* workspace,
                     size_t workspace_bytes, void* stream, int schedule);

/* w4_gemm_ex with a bias added to every output row ([RDNA]
 * _rdna_hybrid_w4a16_apply_impl: the layer bias is added to the product).
 *   bias  [N] device array of the output type (fp16 / bf16 for W4A16, fp16
 *         for W4A8), or NULL (then this is exactly w4_gemm_ex).  It is added
 *         in fp32 to the product before the single rounding to the output
 *         type: W4A16 out = round(sum_k a*w_hat + bias[n]); W4A8
 *         out = fp16_rn((float)acc * s_tok[m] * s_ch[n] + bias[n]).
 * Errors as w4_gemm_ex, plus INVALID_ARGUMENT for a bias with the raw int32
 * output (out_type W4_S32) or a bias not aligned to 2 bytes.  With K == 0
 * every output is its column's bias. */
w4_status w4_gemm_bias(const void* a, int a_type, int64_t M, int64_t K, const void* b_packed,
                       int wtype, int64_t N, const void* b_scales, int scale_type,
                       const void* b_zeros, int64_t group_size, const float* a_token_scales,
                       const float* ch_scales, const void* bias, void* out, int out_type,
                       void* workspace, size_t workspace_bytes, void* stream, int schedule);

/* Schedules: their count, names, and the one the default heuristic picks
 * for a problem (-1 when none can run it). */
int w4_num_schedules(void);
const char* w4_schedule_name(int schedule);
int w4_default_schedule(int64_t M, int64_t N, int64_t K, int a_type, int64_t group_size);

/* Install a per-shape override of the default heuristic ([MR] Code
 * Generation: per-shape schedule choices; [RDNA] a per-shape override
 * table): problems of this activation type with M in [m_lo, m_hi] and
 * exactly this N, K and group_size (-1 = K) run `schedule` by default,
 * when it can run them (else the heuristic decides).  A later entry for the
 * same key replaces the earlier one; schedule -1 removes it.  Entries
 * installed here are consulted before the library's built-in table, which
 * holds measured exceptions to the heuristic.  Host-side only; thread-safe;
 * at most 256 entries (UNSUPPORTED beyond).  Errors: INVALID_ARGUMENT for
 * a bad a_type, range, shape, group size or schedule index. */
w4_status w4_override_schedule(int a_type, int64_t m_lo, int64_t m_hi, int64_t N, int64_t K,
                               int64_t group_size, int schedule);

/* Synchronize `stream`, then report (and clear) a device-side timeout that
 * a kernel recorded in `workspace`: W4_ERR_TIMEOUT, else W4_OK.  On a
 * timeout the split-K counters are zeroed again. */
w4_status w4_check_status(void* workspace, size_t workspace_bytes, void* stream);

/* w4_gemm without a workspace argument.  The source pages have no
 * counterpart to this entry point; it exists for callers that cannot
 * allocate device memory where they run the GEMM (a plug-in inside a
 * framework that owns all device memory and offers its extensions no
 * allocator, or a latency-critical loop that must not call cudaMalloc,
 * which can synchronize the whole device).
 *
 * Arguments and results are those of w4_gemm; the caller still passes every
 * input and the output.  Instead of a workspace, the call uses a scratch
 * array of W4_NOALLOC_SCRATCH_BYTES compiled into the library: it exists once
 * on every GPU that loads libw4 and stays allocated until the process exits.
 * The call allocates and frees nothing (no cudaMalloc, no allocating library
 * routine).
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Every call clears the status word and split-K counters of the scratch
 *     on `stream`, then runs exactly what w4_gemm would.
 *   - All calls on a device share the one array and it keeps the last call's
 *     contents: calls that overlap on the GPU (other streams, other host
 *     threads) race and may corrupt each other's results.  Order them.
 *   - A problem whose scratch need is above W4_NOALLOC_SCRATCH_BYTES is
 *     rejected before anything runs, with W4_ERR_WORKSPACE (w4_last_error()
 *     names the bytes it would need); use w4_gemm with a workspace then.
 *   - A device-side wait that gives up (see w4_check_status) is NOT reported
 *     on this path: its record lives in the shared scratch, which the next
 *     call clears.  Callers that must detect such timeouts use w4_gemm with
 *     their own workspace and w4_check_status.
 *   - The scratch address is looked up once per device and kept for the life
 *     of the process: do not use this entry point after cudaDeviceReset (or
 *     anything else that destroys the device's primary context). */
#define W4_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
w4_status w4_gemm_noalloc(const void* a, int a_type, int64_t M, int64_t K, const void* b_packed,
                          int wtype, int64_t N, const void* b_scales, int scale_type,
                          const void* b_zeros, int64_t group_size, const float* a_token_scales,
                          const float* ch_scales, void* out, int out_type, void* stream);

/* Dynamic per-token int8 quantization of activations for W4A8: the step
 * that makes the `a` (W4_S8) and `a_token_scales` arguments of w4_gemm
 * from fp16/bf16 activations ([PT]: one activation scale per token,
 * computed at run time from that token's values; [QQQ]: symmetric int8
 * activations).  For every row m of a [M,K] (a_type W4_F16 or W4_BF16):
 *   s_tok[m]  = max_k |a[m][k]| / 127, in fp32 (one rounding);
 *   a_q[m][k] = a[m][k] / s_tok[m] rounded once to fp32, then to the
 *               nearest integer, ties to even (always within [-127,127]).
 * A row of zeros gets s_tok 0 and codes 0, so the W4A8 product of that row
 * is 0.  Values must be finite (a row holding Inf or NaN gets unspecified
 * codes and scale).
 *   a      [M,K] device, contiguous rows; 16-byte aligned with K % 8 == 0
 *          for the vectorised path (any other K or alignment runs a
 *          slower element-wise path with the same results).
 *   a_q    [M,K] int8 device output; s_tok [M] fp32 device output.
 * M == 0 is a no-op; K == 0 sets every s_tok to 0.  Errors:
 * INVALID_ARGUMENT (negative size, bad a_type, a null pointer that the
 * sizes need), UNSUPPORTED (M > 2^31 - 1), CUDA. */
w4_status w4_quantize_per_token(const void* a, int a_type, int64_t M, int64_t K, int8_t* a_q,
                                float* s_tok, void* stream);

/* Dynamic per-token fp8 quantization of activations for W4A8 with E4M3
 * activations (a_type W4_E4M3 of the GEMM calls): the same step as
 * w4_quantize_per_token with E4M3 codes ([PT]: one scale per token from its
 * own values; [PR9855]: fp8 activations).  For every row m:
 *   s_tok[m]  = max_k |a[m][k]| / 448, in fp32 (one rounding);
 *   a_q[m][k] = the E4M3 value nearest to a[m][k] / s_tok[m] rounded once
 *               to fp32, ties to the even mantissa, magnitudes beyond 448
 *               saturated to 448 (never NaN).
 * A row of zeros gets s_tok 0 and codes 0.  Arguments, alignment and errors
 * as w4_quantize_per_token (a_q: [M,K] bytes). */
w4_status w4_quantize_per_token_fp8(const void* a, int a_type, int64_t M, int64_t K,
                                    uint8_t* a_q, float* s_tok, void* stream);

/* W4A8 with dynamic per-token quantization inside the call ([PT]: the
 * activation scale of each token computed at run time from that token and
 * applied in the epilogue; [QQQ] / [PR9855]: int8 or fp8 activations).
 * Computes, from fp16 / bf16 activations a [M,K] (a_type W4_F16 / W4_BF16):
 *   (a_q, s_tok) = w4_quantize_per_token (act_type W4_S8) or
 *                  w4_quantize_per_token_fp8 (act_type W4_E4M3) of a;
 *   out [M,N] fp16 = the W4A8 product of a_q with the weights, exactly as
 *                  w4_gemm_bias would compute it with a_token_scales = s_tok
 *                  (and the same schedule).
 * The codes and scales live in the workspace (token_scales_out, when not
 * NULL, receives s_tok [M] instead); on the tensor-core schedule the int8
 * codes are written straight in the form that schedule reads, which saves
 * a pass over the activations.  b_scales / scale_type / group_size / wtype /
 * ch_scales / bias as in w4_gemm_bias; out_type is fp16.
 * workspace: at least w4_gemm_dynamic_workspace_size(M, N, K, act_type,
 * group_size) bytes, 16-byte aligned, zero-filled before its first use.
 * Errors as w4_gemm_bias and w4_quantize_per_token; K must be a positive
 * multiple of 64 (128 for fp8), else UNSUPPORTED. */
size_t w4_gemm_dynamic_workspace_size(int64_t M, int64_t N, int64_t K, int act_type,
                                      int64_t group_size);
w4_status w4_gemm_dynamic(const void* a, int a_type, int64_t M, int64_t K, const void* b_packed,
                          int wtype, int64_t N, const void* b_scales, int scale_type,
                          int64_t group_size, const float* ch_scales, int act_type,
                          const void* bias, void* out, float* token_scales_out,
                          void* workspace, size_t workspace_bytes, void* stream);

/* Static text for a status code; message of the last failed call on this
 * host thread ("" when none). */
const char* w4_status_string(int status);
const char* w4_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* W4_H_ */
