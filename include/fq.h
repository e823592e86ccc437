/*
 * fq.h - C ABI of the GB300 (sm_103a) decode quant + quantized-linear library.
 *
 * One process, one GPU.  Every entry point is asynchronous on the caller's
 * CUDA stream, takes plain pointers and sizes, allocates nothing, and
 * returns an fq_status.  No exception crosses this boundary and nothing
 * aborts.
 *
 * Sources (page title, then section), cited per entry point below:
 *   [W8A8] "DeepSeek-V4 W8A8 performance analysis: small M, NZ layout and
 *          measurement method".
 *   [PR]   "SGLang PR #34277 digest: the DSV4 FP8 quant kernel writes
 *          DeepGEMM's TMA-aligned packed UE8M0 scales".
 *   [DF]   "Reshaping LLM inference dataflow: DeepSeek V4 950 low-precision
 *          optimisation retrospective".
 *
 * Conventions shared by all entry points
 *   - Pointers named x, xq, w, y, s, ... are DEVICE pointers owned by the
 *     caller, valid for the sizes stated, and 16-byte aligned (the
 *     analogue of the 16-byte output_s check in [PR] implementation
 *     breakdown item 1).  A misaligned pointer returns FQ_ERR_ALIGN.
 *   - bf16 values travel as uint16_t bit patterns, E4M3 values as uint8_t
 *     codes, UE8M0 scales as bytes packed four to an int32.
 *   - Row-major ("C") layouts.  Weights are stored K-major: the logical
 *     W[k, n] of a linear is w_nk[n * K + k].  This is the one-time,
 *     load-time layout choice that plays the role of the FRACTAL_NZ weight
 *     cast in [W8A8] section 4.
 *   - A zero-sized problem (M == 0, T == 0, rows == 0) returns FQ_OK
 *     without launching anything ([PR] item 2: the wrapper skips the
 *     launch when numel() == 0).
 *   - Shape rules (else FQ_ERR_SHAPE): sizes >= 0; K % 16 == 0 and
 *     N % 16 == 0 for int8 operands (the INT8 precheck K % 16, N % 32 of
 *     [W8A8] section 4, relaxed to what TMA needs); D % 128 == 0 and
 *     N % 128 == 0 for the FP8 path (whole 128-element groups / blocks).
 *   - Workspace: calls that split K take a caller-owned device workspace of
 *     at least fq_workspace_bytes(...) bytes.  It MUST be zero-filled once
 *     before its first use (e.g. cudaMemsetAsync).  Its head holds per-tile
 *     arrival counters that every completed call returns to zero; the rest
 *     is scratch for split-K partial sums.  So a workspace is reused across
 *     calls without clearing, but calls that may run concurrently
 *     (different streams) must not share one, and after a call that
 *     reported FQ_ERR_DEVICE_TIMEOUT it must be zero-filled again.
 *   - Device-side problems that the host cannot see before launch (an
 *     expert id out of range, a pipeline wait that ran out of time) are
 *     recorded in a device error word and read with fq_device_error().
 *   - The library needs an sm_103 device; anything else returns
 *     FQ_ERR_UNSUPPORTED_DEVICE.
 *   - Kernels are launched with programmatic dependent launch (unless the
 *     environment sets FQ_PDL=0): a linear may start while the previous
 *     kernel on the stream is still running and stream its WEIGHTS (and
 *     weight scales) before it waits for that kernel; everything else it
 *     reads after the wait.  The calls whose output can be a weight operand
 *     (dynamic_quant_int8, quant_mxfp8, fq_quantize_weight_fp8_block) let
 *     the next kernel start only once they have finished, so weights they
 *     write are complete.  Weights written by other code that also launches
 *     its kernels early must be separated from the linear by an ordinary
 *     stream operation.
 */
#ifndef FQ_H_
#define FQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st* fq_stream_t;

typedef enum fq_status {
  FQ_OK = 0,
  FQ_ERR_NULL = 1,               /* a required pointer is NULL */
  FQ_ERR_SHAPE = 2,              /* a size is negative, too large, or breaks a divisibility rule */
  FQ_ERR_ALIGN = 3,              /* a pointer is not 16-byte aligned */
  FQ_ERR_WORKSPACE = 4,          /* workspace missing or smaller than fq_workspace_bytes() */
  FQ_ERR_UNSUPPORTED_DEVICE = 5, /* current device is not sm_103 */
  FQ_ERR_CUDA = 6,               /* a CUDA runtime/driver call failed; see fq_last_cuda_error() */
  FQ_ERR_DEVICE_TIMEOUT = 7,     /* a bounded device wait gave up (reported by fq_device_error) */
  FQ_ERR_DEVICE_INPUT = 8,       /* device data broke the contract, e.g. expert id out of range */
  FQ_ERR_ARG = 9                 /* an argument value is invalid: unknown enum, non-finite eps, overlapping buffers */
} fq_status;

/* Text for a status code; never NULL. */
const char* fq_status_string(int status);

/* The last CUDA error code seen by this thread inside the library (0 = none). */
int fq_last_cuda_error(void);

/* Synchronises `stream`, then reads and clears the device error word of the
 * current device.  Returns FQ_OK, FQ_ERR_DEVICE_TIMEOUT or
 * FQ_ERR_DEVICE_INPUT; *detail (nullable) receives the raw word. */
fq_status fq_device_error(fq_stream_t stream, uint32_t* detail);

/* The same check without the raw word: synchronises `stream`, reads and
 * clears the device error word, and returns FQ_OK, FQ_ERR_DEVICE_TIMEOUT or
 * FQ_ERR_DEVICE_INPUT (or FQ_ERR_CUDA if the synchronisation failed). */
fq_status fq_check_device_error(fq_stream_t stream);

/* Failure-detection self-test of the bounded device waits (no counterpart
 * in the pages; it exercises the same wait loop every pipelined kernel uses).
 * Launches one 32-thread block that initialises an mbarrier expecting one
 * arrival and waits on it for at most `budget_ns` nanoseconds of
 * %globaltimer time (clamped to [1000, 1e9]).  With arrive == 0 nothing ever
 * arrives, the wait gives up, the kernel sets the timeout flag in the device
 * error word and returns, so a following fq_device_error() reports
 * FQ_ERR_DEVICE_TIMEOUT and the context stays usable.  With arrive != 0 the
 * block arrives first and the wait completes (the control case).
 * Returns FQ_OK once launched; asynchronous on `stream`. */
fq_status fq_selftest_wait_timeout(uint64_t budget_ns, int arrive, fq_stream_t stream);

/* Workspace sizing.  `op` is one of fq_op; the four sizes are read as:
 *   FQ_OP_W8A8_LINEAR, FQ_OP_W8A8_QUANT_LINEAR:   (M, K, N, unused)
 *   FQ_OP_FP8_GROUP_EINSUM:                       (T, D, N, G)
 *   FQ_OP_MOE_SORT:                               (T*topk, unused, unused, E)
 *   FQ_OP_W8A8_GROUPED_LINEAR:                    (R rows, K, N, E)
 *   FQ_OP_MXFP8_LINEAR:                           (M, K, N, unused)
 * Returns 0 for an unknown op or invalid sizes. */
typedef enum fq_op {
  FQ_OP_W8A8_LINEAR = 1,
  FQ_OP_W8A8_QUANT_LINEAR = 2,
  FQ_OP_FP8_GROUP_EINSUM = 3,
  FQ_OP_MOE_SORT = 4,
  FQ_OP_W8A8_GROUPED_LINEAR = 5,
  FQ_OP_MXFP8_LINEAR = 6
} fq_op;
size_t fq_workspace_bytes(int op, int64_t a, int64_t b, int64_t c, int64_t d);

/* --------------------------------------------------- load-time weight layout */

/* One-time repack of weights to the K-major layout every linear here reads.
 * [W8A8] section 4: weights are cast once at load time to the layout the
 * matmul streams best (npu_format_cast to FRACTAL_NZ there); here a logical
 * W[k, n] is stored as w_nk[n * K + k], so each TMA box is a run of output
 * channels with contiguous K bytes.  Untimed, off the decode path.
 *   w_kn : int8 [B, K, N] (B stacked matrices, e.g. experts; B = 1 for one
 *          linear), row-major logical weights         in
 *   w_nk : int8 [B, N, K]                               out
 * K % 16 == 0 and N % 16 == 0 (the INT8 rules); the two buffers must not
 * overlap (FQ_ERR_ARG).  Asynchronous on `stream`; the next kernel on the
 * stream starts only after it has finished. */
fq_status fq_repack_weight_kmajor_i8(const int8_t* w_kn, int64_t B, int64_t K, int64_t N, int8_t* w_nk,
                                     fq_stream_t stream);

/* The same repack for the einsum's E4M3 weights ([PR] item 3: the grouped
 * einsum's weight operand), logical [G, D, N] -> stored [G, N, D].
 *   w_gdn : E4M3 [G, D, N] in;  w_gnd : E4M3 [G, N, D] out.
 * D % 128 == 0 and N % 128 == 0 (whole 128 x 128 scale blocks).  Block
 * scales [G, D/128, N/128] keep their layout and need no repack. */
fq_status fq_repack_weight_kmajor_fp8(const uint8_t* w_gdn, int64_t G, int64_t D, int64_t N, uint8_t* w_gnd,
                                      fq_stream_t stream);

/* ------------------------------------------------------------------ INT8 */

/* Per-token INT8 dynamic quantization.
 * [W8A8] section 1 (BF16 X -> npu_dynamic_quant -> INT8 X + per-token
 * scale) and section 2 (a row is the last dimension; one token per row).
 *   x  : bf16 [M, K]            in
 *   xq : int8 [M, K]            out, q = clamp(rint(x / s), -127, 127), ties to even
 *   sx : fp32 [M]               out, s = absmax(row) / 127 (IEEE fp32 division)
 * An all-zero row gives s = 0 and q = 0. */
fq_status dynamic_quant_int8(const uint16_t* x, int64_t M, int64_t K,
                             int8_t* xq, float* sx, fq_stream_t stream);

/* W8A8 linear on pre-quantized activations.
 * [W8A8] section 1 (npu_quant_matmul -> BF16 Y; a linear may consume an
 * upstream (int8, scale) tuple directly, skipping the quant).
 *   xq   : int8 [M, K]   sx : fp32 [M]
 *   w_nk : int8 [N, K] (K-major; logical W[k, n] = w_nk[n*K + k])
 *   sw   : fp32 [N]      per-output-channel weight scale
 *   y    : bf16 [M, N]   y = bf16_RN((fp32(acc) * sx[m]) * sw[n]),
 *                        acc = exact int32 sum_k xq[m,k] * W[k,n]
 *   ws   : workspace of fq_workspace_bytes(FQ_OP_W8A8_LINEAR, M, K, N, 0) bytes
 * K <= 2^31 / (127*127) keeps acc inside int32. */
fq_status w8a8_linear(const int8_t* xq, const float* sx, int64_t M, int64_t K,
                      const int8_t* w_nk, const float* sw, int64_t N, uint16_t* y,
                      void* ws, size_t ws_bytes, fq_stream_t stream);

/* BF16 X -> per-token INT8 quant -> W8A8 linear, in one call.
 * [W8A8] section 1: T_W8A8_linear = T_dynamic_quant + T_quant_matmul + ...
 * Results are bit-identical to dynamic_quant_int8 followed by w8a8_linear.
 *   xq_out, sx_out : nullable; when given they receive the quantized
 *                    activations and scales (int8 [M, K], fp32 [M]).
 *   ws : fq_workspace_bytes(FQ_OP_W8A8_QUANT_LINEAR, M, K, N, 0) bytes. */
fq_status w8a8_quant_linear(const uint16_t* x, int64_t M, int64_t K,
                            const int8_t* w_nk, const float* sw, int64_t N, uint16_t* y,
                            int8_t* xq_out, float* sx_out,
                            void* ws, size_t ws_bytes, fq_stream_t stream);

/* W8A8 linear that allocates nothing - no counterpart in the pages.
 * For callers that cannot allocate device memory: code that runs where
 * cudaMalloc is unavailable or not allowed (an allocator-free runtime, a
 * plugin that must not touch its host's memory pool), so that it cannot
 * provide the workspace w8a8_linear needs.  Same arguments and bit-identical
 * results as w8a8_linear, without the workspace.
 *   Scratch: a fixed ~10.5 MB array in device memory (16 KiB of arrival
 *   counters + 10 MiB of partial sums).  The CUDA driver reserves it when it
 *   loads this library's W8A8 module on a device - with lazy module loading
 *   possibly inside the first call of any W8A8 entry point on that device -
 *   and holds it until the process exits; every process that uses a W8A8
 *   entry point pays for it, whether or not it calls this one.  If the device
 *   has no room for it, that first call returns FQ_ERR_CUDA with an
 *   out-of-memory code in fq_last_cuda_error().
 *   Limits: M <= 64, N <= 524288 (ceil(N/128) <= 4096 tiles), at most 160
 *   SMs; larger sizes return FQ_ERR_SHAPE (FQ_ERR_UNSUPPORTED_DEVICE for more
 *   SMs).  No cudaMalloc/cudaFree or allocating library call is made.
 *   The first call on a device looks up the array's device address (once per
 *   device, with that device current) and keeps it for the life of the
 *   process; make that first call before any stream capture.  Resetting the
 *   device (cudaDeviceReset, or a reset of its primary context) while the
 *   library is loaded is not supported.  Each call zeroes the counters it
 *   uses with cudaMemsetAsync on `stream`, then launches the GEMM.
 *   All calls share the one array: calls that may overlap on the GPU
 *   (different streams, or different host threads) race and give wrong
 *   results; serialise them. */
fq_status w8a8_linear_noalloc(const int8_t* xq, const float* sx, int64_t M, int64_t K,
                              const int8_t* w_nk, const float* sw, int64_t N, uint16_t* y,
                              fq_stream_t stream);

/* ------------------------------------------------------------------- FP8 */

/* FP8 E4M3 per-128-element group quant writing packed UE8M0 scales.
 * [PR] implementation breakdown items 1-2 and the key source snippets.
 *   x        : bf16 [T, G, D], D % 128 == 0       in
 *   xq       : E4M3 [T, G, D]                     out
 *   s_packed : int32 [G, P, Ta], P = ceil((D/128)/4), Ta = align_up(T, 4)  out
 * For each (t, g, j) with j the 128-wide hidden group:
 *   e = clamp(ceil(log2(absmax / 448)), -127, 127)   (absmax == 0 -> -127)
 *   xq = E4M3_RN_satfinite(x * 2^-e)
 *   byte (e + 127) at byte offset ((g*P + j/4)*Ta + t)*4 + j%4
 * Every other byte of s_packed is written as zero: the bytes of the last
 * pack past the last group (as in [PR]) and the token-padding words
 * t in [T, Ta) (stronger than [PR], which leaves them uninitialised).
 * The logical scale view is [T, G, P] with element strides (1, P*Ta, Ta). */
fq_status quant_fp8_group_ue8m0_packed(const uint16_t* x, int64_t T, int64_t G, int64_t D,
                                       uint8_t* xq, int32_t* s_packed, fq_stream_t stream);

/* Same quant, writing unpacked fp32 scales 2^e as fp32 [T, G, D/128].
 * This is the producer's form before the PR ([PR] motivation); kept as the
 * A/B control together with fq_pack_scales_ue8m0. */
fq_status quant_fp8_group_fp32(const uint16_t* x, int64_t T, int64_t G, int64_t D,
                               uint8_t* xq, float* s_f32, fq_stream_t stream);

/* fp32 power-of-two scales [T, G, NG] -> packed UE8M0 int32 [G, ceil(NG/4), align_up(T,4)],
 * zero in the unused bytes and token padding.  The separate conversion
 * ([PR] motivation: transpose_and_pack_fp32_into_ue8m0) that writing the
 * packed layout directly removes.  Values that are not powers of two in
 * [2^-127, 2^127] are outside the contract. */
fq_status fq_pack_scales_ue8m0(const float* s_f32, int64_t T, int64_t G, int64_t NG,
                               int32_t* s_packed, fq_stream_t stream);

/* Load-time FP8 weight prep with fp32 per-128x128 block scales.
 *   w_gnd : fp32 [G, N, D] (logical W[g, d, n] = w_gnd[(g*N + n)*D + d])
 *   wq    : E4M3 [G, N, D]          wq = E4M3_RN_satfinite(fp32(w / sw_blk))
 *   sw_blk: fp32 [G, D/128, N/128]  sw_blk = fp32(absmax(block) / 448)
 * An all-zero block gives sw_blk = 0 and codes 0.  Untimed, offline step;
 * the plain absmax reading of "fp32 per-128x128 block scales". */
fq_status fq_quantize_weight_fp8_block(const float* w_gnd, int64_t G, int64_t N, int64_t D,
                                       uint8_t* wq, float* sw_blk, fq_stream_t stream);

typedef enum fq_scale_fmt {
  FQ_SCALE_UE8M0_PACKED = 0, /* sx is int32 [G, ceil((D/128)/4), align_up(T,4)] (the producer's layout) */
  FQ_SCALE_FP32 = 1          /* sx is fp32 [T, G, D/128] holding 2^e */
} fq_scale_fmt;

/* Block-scaled FP8 grouped einsum (the consumer of the packed scales).
 * [PR] motivation / item 3: deep_gemm.fp8_einsum reading the TMA-aligned
 * packed activation scales; the packed and fp32 scale paths must give
 * bit-identical Y.
 *   xq     : E4M3 [T, G, D]
 *   sx     : scales in format `fmt`
 *   w_gnd  : E4M3 [G, N, D] (logical W[g, d, n])
 *   sw_blk : fp32 [G, D/128, N/128]
 *   y      : bf16 [T, G, N]
 *   Y[t,g,n] = bf16( sum_kb sx[t,g,kb] * sw[g,kb,n/128] * sum_{d in kb} xq[t,g,d] * W[g,d,n] )
 * accumulated in fp32 with a fixed, data-independent order (deterministic).
 *   ws : fq_workspace_bytes(FQ_OP_FP8_GROUP_EINSUM, T, D, N, G) bytes. */
fq_status fp8_group_einsum(const uint8_t* xq, const void* sx, int fmt,
                           int64_t T, int64_t G, int64_t D,
                           const uint8_t* w_gnd, const float* sw_blk, int64_t N, uint16_t* y,
                           void* ws, size_t ws_bytes, fq_stream_t stream);

/* ------------------------------------------------- RMSNorm + quant producer */

/* RMSNorm fused with the activation quant, the producer of a linear's
 * quantized input ([DF] section 2.3, first fusion: the normalised row stays
 * in registers and only the quantized activation is written; [W8A8]
 * section 1: the linear consumes the ready (int8, scale) tuple).
 *   x     : bf16 [M, K] (or [T, K])   in, row-major
 *   gamma : bf16 [K]                  in
 *   eps   : finite, >= 0              (else FQ_ERR_ARG)
 * Per row: ss = sum x^2 exactly, rounded once to fp64;
 *          r  = fp32(1 / sqrt(ss / K + eps)) (fp64 steps; 0 if the argument is 0);
 *          y  = fp32(fp32(x * r) * gamma), kept in fp32 (never rounded to bf16).
 * rmsnorm_quant_int8: the per-token INT8 rule of dynamic_quant_int8 on y:
 *   xq int8 [M, K], sx fp32 [M].  K % 16 == 0.
 * rmsnorm_quant_fp8_ue8m0_packed: the per-128-group rule of
 *   quant_fp8_group_ue8m0_packed on y with one outer group (G = 1, D = K):
 *   xq E4M3 [T, K], s_packed int32 [1, ceil(K/512), align_up(T, 4)] (unused
 *   pack bytes and token-padding words written as zero).  K % 128 == 0.
 * Both: K <= 16384; all pointers 16-byte aligned; asynchronous on `stream`.
 * Rows whose r overflows fp32 (eps == 0 and ss / K below about 2^-254) are
 * outside the contract. */
fq_status rmsnorm_quant_int8(const uint16_t* x, const uint16_t* gamma, float eps, int64_t M, int64_t K,
                             int8_t* xq, float* sx, fq_stream_t stream);
fq_status rmsnorm_quant_fp8_ue8m0_packed(const uint16_t* x, const uint16_t* gamma, float eps, int64_t T, int64_t K,
                                         uint8_t* xq, int32_t* s_packed, fq_stream_t stream);

/* ------------------------------------------ 32-element block-scaled FP8 */

/* MXFP8-like block scaling ([DF] section 2.1: every 32 elements share one
 * 8-bit scale, E4M3 payloads); the per-128-group rule of
 * quant_fp8_group_ue8m0_packed applied to 32-element blocks along K.
 * Scale storage is blocked for the linear's tensor-core scale copy: for every
 * 128 rows x 128 K one 512-byte chunk, chunk (r / 128, k / 128) at byte offset
 * ((r / 128) * (K / 128) + k / 128) * 512; row r's byte for K block b = k / 32
 * at (r % 32) * 16 + ((r % 128) / 32) * 4 + b % 4 within it; rows past R in
 * the last chunk row are zero bytes.
 *
 * quant_mxfp8: x bf16 [R, K] -> q E4M3 [R, K] and sf_blocked uint8
 *   [ceil(R / 128), K / 128, 512].  Used for activations (rows = tokens) and
 *   for load-time weight prep (rows = output channels).  K % 128 == 0. */
fq_status quant_mxfp8(const uint16_t* x, int64_t R, int64_t K, uint8_t* q, uint8_t* sf_blocked, fq_stream_t stream);

/* Y[m, n] = bf16( sum_k (qx[m,k] * 2^(sx[m,k/32]-127)) * (qw[n,k] * 2^(sw[n,k/32]-127)) ),
 * accumulated in fp32 by the tensor cores (tcgen05 block-scaled MMA).
 *   xq, xsf : activations [M, K] and their blocked scales (quant_mxfp8)
 *   wq, wsf : weights [N, K] (K-major) and their blocked scales
 *   y       : bf16 [M, N]
 *   ws      : fq_workspace_bytes(FQ_OP_MXFP8_LINEAR, M, K, N, 0) bytes
 * K % 128 == 0, N % 16 == 0.  Partial tiles are summed in a fixed order, so
 * repeated calls give identical bits. */
fq_status mxfp8_linear(const uint8_t* xq, const uint8_t* xsf, int64_t M, int64_t K, const uint8_t* wq,
                       const uint8_t* wsf, int64_t N, uint16_t* y, void* ws, size_t ws_bytes, fq_stream_t stream);

/* ------------------------------------------------------------------- MoE */

/* Stable sort of the (token, slot) pairs of topk_ids [T, topk] by expert id.
 * [DF] section 3.2 (sort tokens by expert id before dispatch so each
 * expert's rows are contiguous) and [W8A8] section 5 (group_list =
 * expert_tokens).
 *   offsets  : int32 [E + 1]    out, exclusive scan of per-expert counts
 *   perm     : int32 [T*topk]   out, perm[i] = flat pair index t*topk + j of sorted row i
 *   pair_row : int32 [T*topk]   out (nullable), the inverse: sorted row of pair t*topk + j
 * Ties keep pair order.  Ids outside [0, E) are dropped and flagged in the
 * device error word (FQ_ERR_DEVICE_INPUT).  E <= 1024.
 *   ws : fq_workspace_bytes(FQ_OP_MOE_SORT, T*topk, 0, 0, E) bytes. */
fq_status moe_sort(const int32_t* topk_ids, int64_t T, int64_t topk, int64_t E,
                   int32_t* offsets, int32_t* perm, int32_t* pair_row,
                   void* ws, size_t ws_bytes, fq_stream_t stream);

/* Gather of quantized token rows into expert order (the "gather" of
 * [DF] section 3.2): row i of (xq_g, sx_g) is token perm[i] / topk of (xq, sx).
 *   xq : int8 [T, K]  sx : fp32 [T]  ->  xq_g : int8 [R, K]  sx_g : fp32 [R], R = T*topk. */
fq_status moe_gather_rows_i8(const int8_t* xq, const float* sx, const int32_t* perm,
                             int64_t T, int64_t topk, int64_t K,
                             int8_t* xq_g, float* sx_g, fq_stream_t stream);

/* Grouped W8A8 linear: expert e multiplies rows [offsets[e], offsets[e+1])
 * by its own weight.  [W8A8] section 5 (npu_grouped_matmul with
 * group_list = expert_tokens; expert-local M_e).  Empty experts cost
 * nothing.  Per row, exactly w8a8_linear with that expert's weight.
 *   xq : int8 [R, K]  sx : fp32 [R]  offsets : int32 [E + 1] (device), offsets[E] == R
 *   w_enk : int8 [E, N, K]   sw_en : fp32 [E, N]   y : bf16 [R, N]
 *   ws : fq_workspace_bytes(FQ_OP_W8A8_GROUPED_LINEAR, R, K, N, E) bytes. */
fq_status w8a8_grouped_linear(const int8_t* xq, const float* sx, const int32_t* offsets,
                              int64_t R, int64_t E, int64_t K,
                              const int8_t* w_enk, const float* sw_en, int64_t N, uint16_t* y,
                              void* ws, size_t ws_bytes, fq_stream_t stream);

/* SwiGLU fused with per-token INT8 re-quant.
 * [DF] section 2.3 (activation fused with quantization, saving one write
 * and read of the activation).
 *   gu : bf16 [rows, 2*I]: gate g = columns [0, I), up u = columns [I, 2I)
 *   h  = bf16_RN(fp32(silu(g)) * u), silu(g) = g / (1 + exp(-g)) in fp32
 *   hq : int8 [rows, I], sh : fp32 [rows]  - dynamic_quant_int8 of h
 *   h_out : bf16 [rows, I], nullable; receives h (for inspection). */
fq_status swiglu_quant_int8(const uint16_t* gu, int64_t rows, int64_t I,
                            int8_t* hq, float* sh, uint16_t* h_out, fq_stream_t stream);

/* Weighted combine back to token order ([W8A8] section 1: T_combine).
 *   y_rows   : bf16 [T*topk, H] in sorted (expert) order
 *   pair_row : int32 [T*topk], sorted row of pair t*topk + j (from moe_sort)
 *   topk_w   : fp32 [T, topk]
 *   out[t]   = bf16_RN(running fp32 sum over j = 0..topk-1 of fp32(w[t,j] * y[pair_row[t*topk+j]]))
 */
fq_status moe_combine(const uint16_t* y_rows, const int32_t* pair_row, const float* topk_w,
                      int64_t T, int64_t topk, int64_t H, uint16_t* out, fq_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* FQ_H_ */
