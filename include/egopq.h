/*
 * egopq.h -- C ABI of the GB300 (sm_103a) W4A8 packed-linear GEMM library.
 *
 * The operation (y = a_s * sum_g s * (sum_k a_q*w_q - z * sum_k a_q), bf16 out)
 * is the linear that the quantized serving stacks on these pages turn on:
 *  - "The 4-bit CPU path" (vllm-omni docs/edge/cpu-4bit.md), section
 *    "W4A8 - _C::int4_scaled_mm_cpu": GPTQ-packed int4 weights, activations
 *    quantized to int8 at run time, zero points from the checkpoint or the
 *    constant 8 for a symmetric export.
 *  - "EgoPQ Real-Serving Handoff", section 2 "External Artifacts": native
 *    W4A8 serving needs exact per-group _gptq_scale / _gptq_zero metadata.
 *  - "The 4-bit CPU path", sections "W4A16 - PyTorch tinygemm" and "Building a
 *    checkpoint": weight-only int4, group size 128.
 *  - "Serve a pre-quantized int8 weight-only DiT via compressed-tensors ..."
 *    (vllm-omni issue 5), sections "Context" and "Plan": int8 weight-only
 *    (W8A16) linears; sections "Directive after the int8-wo result" and
 *    "Round two": W8A8 int8-dynamic.
 *
 * Conventions for every call:
 *  - Pointers are caller-owned DEVICE memory unless stated otherwise, 16-byte
 *    aligned. The library allocates nothing per call (its only device state:
 *    a 4-byte error word per kernel unit and the 16 MiB staging array of
 *    egopq_w4a8_linear_noalloc).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream). They validate arguments on the host first and return a negative
 *    egopq_status without launching anything when a check fails; a failed
 *    launch returns EGOPQ_ERR_CUDA. egopq_last_error_string() describes the
 *    last failure of the calling thread.
 *  - Matrices are row-major. bf16 and fp16 values travel as their 16-bit
 *    patterns (uint16_t).
 *  - Shape gate: group == 128, K % 128 == 0, N % 128 == 0, M >= 0 (M == 0 is a
 *    no-op), every size below 2^31 (larger: EGOPQ_ERR_UNSUPPORTED_SHAPE).
 *    Shapes that do not tile the 128-row weight block are refused rather
 *    than computed wrong ("The 4-bit CPU path", section "The weight
 *    layout, measured": a reshape gate keeps an untiled N from being
 *    mis-read).
 */
#ifndef EGOPQ_H
#define EGOPQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  EGOPQ_OK = 0,
  EGOPQ_ERR_INVALID_ARG = -1,       /* null pointer, bad enum, negative size */
  EGOPQ_ERR_UNSUPPORTED_SHAPE = -2, /* group != 128, K % 128, N % 128, size >= 2^31 */
  EGOPQ_ERR_MISALIGNED = -3,        /* an operand pointer is not 16-byte aligned */
  EGOPQ_ERR_ARCH = -4,              /* current device is not sm_103 */
  EGOPQ_ERR_CUDA = -5,              /* a CUDA runtime call or launch failed */
  EGOPQ_ERR_TIMEOUT = -6,           /* a kernel's bounded wait expired */
  EGOPQ_ERR_DEVICE_INDEX = -7       /* a debug build's device-side index check failed */
} egopq_status;

/* Kernel path. AUTO picks by M (W4A8, W4A16 and W8A16: CUDA-core GEMV for
 * M <= 4, the tcgen05 tensor-core GEMM otherwise; W8A8: GEMV for M <= 64);
 * egopq_auto_path reports the choice. The others force one
 * path for tests and benchmarks. The choice is always this explicit argument,
 * never global or environment state ("The 4-bit CPU path", section "Why the
 * path choice is a config field"). */
typedef enum { EGOPQ_PATH_AUTO = 0, EGOPQ_PATH_GEMV = 1, EGOPQ_PATH_TC = 2 } egopq_path;

typedef enum {
  EGOPQ_VARIANT_W4A8 = 0,
  EGOPQ_VARIANT_W4A16 = 1,
  EGOPQ_VARIANT_W8A16 = 2,
  EGOPQ_VARIANT_W8A8 = 3
} egopq_variant;

/* The path EGOPQ_PATH_AUTO takes for M tokens of `variant` (EGOPQ_PATH_GEMV
 * or EGOPQ_PATH_TC), or EGOPQ_ERR_INVALID_ARG for an unknown variant or
 * M < 0. Host-only; no device is touched. */
int egopq_auto_path(int64_t M, int variant);

/* The token tile (the MMA's N: tokens per output tile) the tensor-core path
 * runs an M x N x K call of `variant` with, for inspection and tests: 16, 32
 * or 64 for M <= 64; above that 192 or 128 -- 192-token tiles run the tensor
 * pipe at its full rate, and the library takes them unless the grid they
 * make over the current device's SMs takes longer. EGOPQ_ERR_INVALID_ARG for an unknown variant or
 * M <= 0; EGOPQ_ERR_UNSUPPORTED_SHAPE for a refused shape or W8A8 with
 * M <= 64 (no tensor-core form). Reads the current device's SM count. */
int egopq_tc_token_tile(int64_t M, int64_t N, int64_t K, int variant);

/* Kernel launches the tensor-core path makes for an M x N x K call of
 * `variant` (and for a grouped call whose outputs total N rows), for
 * inspection, tests and launch accounting: 1, or 2 where a persistent grid of
 * wide tiles would end in a short last round -- its full rounds run first,
 * then the remaining tiles as a second launch with K split over clusters. The
 * errors of egopq_tc_token_tile. Reads the current device's SM count. */
int egopq_tc_launches(int64_t M, int64_t N, int64_t K, int variant);

typedef void* egopq_stream_t; /* cudaStream_t */

/* Library version, major*10000 + minor*100 + patch. */
int egopq_version(void);

/* ---- weight packing --------------------------------------------------------
 * Size in bytes of the packed form of an N x K int4 weight with group 128, or
 * 0 if the shape is refused (N*K/2 + 5*N*G/2 bytes otherwise). The packed
 * buffer is a sequence of 8512-byte records, one per (128-row block t,
 * group g), record (t, g) at byte (t*G + g) * 8512, so that a kernel fetches
 * everything one group of a row block needs with a single copy:
 *   [0, 8192)     codes: the 16-byte unit of chunk c (32 codes, k = 128g+32c..)
 *                 of row r = n - 128t at (c*128 + r) * 16; little-endian word
 *                 j of a unit holds k0 = 128g+32c+8j .. k0+7, nibble p carrying
 *                 k0 + 2p (p < 4) or k0 + 2(p-4) + 1 (p >= 4);
 *   [8192, 8448)  fp16 scale s[n,g] of row r at 8192 + 2r;
 *   [8448, 8512)  zero points: z[n,g] of row r in byte 8448 + r/2, low nibble
 *                 for even r, high nibble for odd r.
 * The layout is this library's own (the pages fix only the logical codes,
 * scales and zero points below). */
size_t egopq_packed_w4_bytes(int64_t N, int64_t K, int group);

/* Pack logical GPTQ-style int4 weights into `packed` (device,
 * egopq_packed_w4_bytes(N,K,group) bytes). Inputs (device):
 *   w_q        uint8 [N][K], codes 0..15 (bits above the low nibble ignored)
 *   scale_f16  fp16  [N][G], per-group scale s[n,g]      (_gptq_scale)
 *   zero       uint8 [N][G], per-group zero point 0..15  (_gptq_zero)
 * Dequantized weight: s[n,g] * (w_q[n,k] - z[n,g]); zero = 8 everywhere is the
 * symmetric grid ("The 4-bit CPU path", section "W4A8"). */
int egopq_pack_w4(const uint8_t* w_q, const uint16_t* scale_f16, const uint8_t* zero,
                  int64_t N, int64_t K, int group, void* packed, egopq_stream_t stream);

/* Dequantize a packed weight once to dense bf16 (device w_bf16 [N][K],
 * row-major, caller-allocated 2*N*K bytes):
 *   w[n][k] = bf16( s[n,g] * (w_q[n,k] - z[n,g]) ),  g = k / 128,
 * the product exact in fp32, one round-to-nearest-even conversion. This is the
 * operand of the dense comparison path that large batches can take (dequantize
 * once, then an ordinary bf16 GEMM: "The 4-bit CPU path", section "W4A16 -
 * PyTorch tinygemm"). Asynchronous on `stream`; shape errors as for
 * egopq_pack_w4. */
int egopq_dequant_w4(const void* packed, int64_t N, int64_t K, int group, uint16_t* w_bf16,
                     egopq_stream_t stream);

/* Pack a GPTQ checkpoint's tensors (device) directly into `packed`:
 *   qweight     int32 [K/8][N]: word (r, n) holds the codes of rows k = 8r+i
 *               (i = 0..7) of output n in bits 4i..4i+3, low nibble first;
 *   qzeros      int32 [G][N/8]: word (g, c) holds the zero points of outputs
 *               n = 8c+j in bits 4j..4j+3;
 *   scales_f16  fp16  [G][N]   (_gptq_scale);
 *   zero_offset 0 or 1: z = stored nibble + zero_offset (1 for exporters that
 *               store z - 1)                          (_gptq_zero).
 * The pages name this metadata ("EgoPQ Real-Serving Handoff", section 2;
 * "The 4-bit CPU path", section "W4A8") but not its byte layout; the layout
 * above is the common GPTQ export convention. Group-ordered checkpoints only
 * (row k in group k / 128; no activation-order permutation). The result equals
 * egopq_pack_w4 of the unpacked codes, scales and zero points. A zero point
 * outside [0, 15] after the offset cannot be stored: it is kept modulo 16 and
 * the next egopq_device_status returns EGOPQ_ERR_INVALID_ARG. Shape errors as
 * for egopq_pack_w4. */
int egopq_pack_w4_gptq(const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales_f16,
                       int64_t N, int64_t K, int group, int zero_offset, void* packed,
                       egopq_stream_t stream);

/* Inverse of egopq_pack_w4 (test and inspection aid). */
int egopq_unpack_w4(const void* packed, int64_t N, int64_t K, int group, uint8_t* w_q,
                    uint16_t* scale_f16, uint8_t* zero, egopq_stream_t stream);

/* ---- activation quantization -------------------------------------------------
 * Per-token symmetric int8 quantization of x (bf16 [M][K]), fused with the
 * per-group sums that fold the zero points into the epilogue:
 *   a_s[m]      = max_k |x[m,k]| / 127                 (fp32 quotient)
 *   a_q[m,k]    = clamp(round_half_even(x / a_s), -127, 127)  (fp32 quotient)
 *   a_gsum[m,g] = sum_{k in g} a_q[m,k]
 * A row of zeros gives a_s = 0 and a_q = 0. Outputs (device): a_q int8
 * [M][K], a_s fp32 [M], a_gsum int32 [M][G]. a_q may be NULL when a_tc is
 * given: the codes are then written only in the operand form, which is all
 * the tensor-core path reads (the GEMV path reads a_q). a_tc (optional, may be NULL;
 * egopq_tc_operand_bytes(M, K, group) bytes) receives the same codes in the
 * operand form the tensor-core path loads with TMA. The library chooses that
 * form from M (egopq_tc_operand_form); a buffer written for one M is valid
 * only for GEMM calls with the same M. Its layout, for inspection only:
 *   EGOPQ_TC_FORM_E4M3_PLANES (M <= 64): two e4m3 planes [2][M][K] bytes,
 *            plane 0 holding a_q >> 4 (arithmetic shift, in [-8, 7]) and
 *            plane 1 holding a_q & 15, so a_q = 16 * plane0 + plane1, both
 *            exact in e4m3; inside every aligned run of 8 K values the bytes
 *            are ordered k0, k0+2, k0+4, k0+6, k0+1, k0+3, k0+5, k0+7 (the
 *            nibble order of the packed weights);
 *   EGOPQ_TC_FORM_F16 (M > 64): fp16 [M][K], the codes as exact fp16 integers.
 * Callers that do not want to hold this buffer use egopq_w4a8_linear, which
 * keeps it inside its workspace.
 * ("The 4-bit CPU path", section "W4A8": the kernel quantizes activations to
 * int8.) */
typedef enum { EGOPQ_TC_FORM_E4M3_PLANES = 1, EGOPQ_TC_FORM_F16 = 2 } egopq_tc_form;

/* Bytes of the tensor-core operand buffer a_tc for M x K codes (2*M*K), or 0
 * for a refused shape (M <= 0, K not a multiple of 128, group != 128). */
size_t egopq_tc_operand_bytes(int64_t M, int64_t K, int group);
/* The form egopq_quant_act_i8 writes a_tc in for M tokens (an
 * egopq_tc_form), or EGOPQ_ERR_INVALID_ARG for M <= 0. */
int egopq_tc_operand_form(int64_t M);

int egopq_quant_act_i8(const uint16_t* x_bf16, int64_t M, int64_t K, int group, int8_t* a_q,
                       float* a_s, int32_t* a_gsum, void* a_tc, egopq_stream_t stream);

/* ---- W4A8 GEMM -----------------------------------------------------------------
 * y[m,n] = bf16( a_s[m] * sum_g s[n,g] * (sum_{k in g} a_q[m,k] w_q[n,k]
 *                                         - z[n,g] * a_gsum[m,g]) )
 * Inputs from egopq_quant_act_i8 and egopq_pack_w4; y is bf16 [M][N]. The
 * GEMV path reads a_q and a_gsum (a_q required when it runs: NULL gives
 * EGOPQ_ERR_INVALID_ARG); the tensor-core path reads a_tc (required when it
 * runs; a_q may then be NULL) and, for M > 64, folds z into its weight operand, for
 * M <= 64 subtracts z * a_gsum in its epilogue. Every path forms each group's
 * integer partial exactly before scaling. */
int egopq_w4a8_gemm(const int8_t* a_q, const void* a_tc, const float* a_s,
                    const int32_t* a_gsum, const void* packed, int64_t M, int64_t N, int64_t K,
                    int group, uint16_t* y_bf16, egopq_stream_t stream);
int egopq_w4a8_gemm_ex(const int8_t* a_q, const void* a_tc, const float* a_s,
                       const int32_t* a_gsum, const void* packed, int64_t M, int64_t N,
                       int64_t K, int group, uint16_t* y_bf16, int path, egopq_stream_t stream);

/* Sibling W4A8 linears that read the same activations -- a layer's query, key
 * and value projections, or the gate and up projections of its MLP -- in ONE
 * kernel launch over all their output tiles (fewer dependent launches per
 * decode step; the fused query/key/value loading of "Serve a pre-quantized
 * int8 weight-only DiT via compressed-tensors ...", section "Round two").
 * For j < count (1..8): y_bf16[j] = the egopq_w4a8_gemm_ex result of
 * (a, packed[j]) with N[j] output rows (N[j] % 128 == 0), on `path`. packed,
 * N and y_bf16 are HOST arrays of `count` entries; the pointers they hold are
 * device memory (16-byte aligned). Each output is formed from the same exact
 * integer group partials as a separate call; the kernel grid (and so the
 * fp32 order in which split-K partial sums are added) depends on all the
 * linears together, so outputs can differ from separate calls in rounding,
 * always within the output bar. Deterministic. */
int egopq_w4a8_gemm_grouped(const int8_t* a_q, const void* a_tc, const float* a_s,
                            const int32_t* a_gsum, int count, const void* const* packed,
                            const int64_t* N, int64_t M, int64_t K, int group,
                            uint16_t* const* y_bf16, int path, egopq_stream_t stream);

/* One-call W4A8 linear from bf16 activations: per-token int8 quantization as
 * in egopq_quant_act_i8 into `workspace`, then the W4A8 GEMM on `path`, y bf16
 * [M][N]. `workspace` is caller-owned device memory of at least
 * egopq_w4a8_linear_workspace_bytes(M, K, group, path) bytes, 16-byte
 * aligned, holding the quantized activations between the two kernels; calls
 * sharing one workspace must be ordered on one stream. Results are
 * bit-identical to egopq_quant_act_i8 followed by egopq_w4a8_gemm_ex on the
 * same path (the byte count is 0 for shapes the call refuses). */
size_t egopq_w4a8_linear_workspace_bytes(int64_t M, int64_t K, int group, int path);
int egopq_w4a8_linear(const uint16_t* x_bf16, const void* packed, int64_t M, int64_t N, int64_t K,
                      int group, uint16_t* y_bf16, void* workspace, size_t workspace_bytes,
                      int path, egopq_stream_t stream);

/* egopq_w4a8_linear for sibling linears: one quantization of x, then
 * egopq_w4a8_gemm_grouped over the `count` weights (arrays as there). The
 * workspace is egopq_w4a8_linear_workspace_bytes(M, K, group, path) bytes,
 * the same as for a single linear. */
int egopq_w4a8_linear_grouped(const uint16_t* x_bf16, int count, const void* const* packed,
                              const int64_t* N, int64_t M, int64_t K, int group,
                              uint16_t* const* y_bf16, void* workspace, size_t workspace_bytes,
                              int path, egopq_stream_t stream);

/* egopq_w4a8_linear for callers that cannot allocate device memory -- a
 * plugin inside a framework that owns every device buffer, or a serving loop
 * that must never enter cudaMalloc. The pages have no counterpart; this is a
 * deployment convenience. Same arguments and results as egopq_w4a8_linear
 * minus the workspace: the quantized activations are staged in a 16 MiB
 * file-scope device array that every GPU loading the library holds until the
 * process exits. Calls whose staging exceeds 16 MiB (about 2*M*K bytes on the
 * tensor-core path, M*K on the GEMV path) return EGOPQ_ERR_UNSUPPORTED_SHAPE.
 * All calls share the array: calls that overlap on the GPU race on it. The
 * first call in each CUDA context looks the array's address up with that
 * context's device current (and a call after a device reset, in the new
 * context, looks it up again); make that first call before any stream
 * capture. Shape and size checks are those of egopq_w4a8_linear. Allocates
 * nothing. */
int egopq_w4a8_linear_noalloc(const uint16_t* x_bf16, const void* packed, int64_t M, int64_t N,
                              int64_t K, int group, uint16_t* y_bf16, int path,
                              egopq_stream_t stream);

/* Test readout: the integer group partials Q[m][n][g] (int32 [M][N][G]) the
 * chosen path forms before scaling, from the same main loop:
 *   Q[m,n,g] = sum_{k in g} a_q[m,k] w_q[n,k] - z[n,g] * sum_{k in g} a_q[m,k].
 * a_q and a_tc as for egopq_w4a8_gemm_ex (each required by its own path). */
int egopq_w4a8_group_partials(const int8_t* a_q, const void* a_tc, const int32_t* a_gsum,
                              const void* packed, int64_t M, int64_t N, int64_t K, int group,
                              int32_t* Q, int path, egopq_stream_t stream);

/* ---- W4A16 GEMM ------------------------------------------------------------------
 * y[m,n] = bf16( sum_g s[n,g] * sum_{k in g} x[m,k] * (w_q[n,k] - z[n,g]) )
 * x bf16 [M][K]; packed as for W4A8; y bf16 [M][N]. ("The 4-bit CPU path",
 * section "W4A16 - PyTorch tinygemm".) */
int egopq_w4a16_gemm(const uint16_t* x_bf16, const void* packed, int64_t M, int64_t N,
                     int64_t K, int group, uint16_t* y_bf16, egopq_stream_t stream);
int egopq_w4a16_gemm_ex(const uint16_t* x_bf16, const void* packed, int64_t M, int64_t N,
                        int64_t K, int group, uint16_t* y_bf16, int path,
                        egopq_stream_t stream);

/* ---- W8A16 GEMM ------------------------------------------------------------------
 * y[m,n] = bf16( s[n] * sum_k x[m,k] * w_q[n,k] )
 * x bf16 [M][K]; w_q int8 [N][K] row-major in [-127, 127] (symmetric,
 * per-output-channel; no pack step); scale_f16 fp16 [N]; y bf16 [M][N].
 * ("Serve a pre-quantized int8 weight-only DiT ...", sections "Context" and
 * "Plan".) */
int egopq_w8a16_gemm(const uint16_t* x_bf16, const int8_t* w_q, const uint16_t* scale_f16,
                     int64_t M, int64_t N, int64_t K, uint16_t* y_bf16, egopq_stream_t stream);
int egopq_w8a16_gemm_ex(const uint16_t* x_bf16, const int8_t* w_q, const uint16_t* scale_f16,
                        int64_t M, int64_t N, int64_t K, uint16_t* y_bf16, int path,
                        egopq_stream_t stream);

/* ---- W8A8 int8-dynamic GEMM ------------------------------------------------------
 * y[m,n] = bf16( a_s[m] * s[n] * sum_k a_q[m,k] * w_q[n,k] )
 * Activations as egopq_quant_act_i8 produces them (per-token int8 a_q [M][K],
 * a_s fp32 [M]; a_tc, the tensor-core operand form, is read only on the
 * tensor-core path and only exists there for M > 64; a_q is read only on
 * the GEMV path and may be NULL when the tensor cores run); weights int8 [N][K]
 * row-major in [-127, 127] with fp16 per-output-channel scales [N], as for
 * W8A16. The integer dot products are exact (int32). AUTO runs the GEMV for
 * M <= 64 and the tensor cores above; EGOPQ_PATH_TC with M <= 64 returns
 * EGOPQ_ERR_UNSUPPORTED_SHAPE. ("Serve a pre-quantized int8 weight-only DiT
 * via compressed-tensors ...", sections "Directive after the int8-wo result"
 * and "Round two": W8A8 int8-dynamic.) */
int egopq_w8a8_gemm(const int8_t* a_q, const void* a_tc, const float* a_s, const int8_t* w_q,
                    const uint16_t* scale_f16, int64_t M, int64_t N, int64_t K, uint16_t* y_bf16,
                    egopq_stream_t stream);
int egopq_w8a8_gemm_ex(const int8_t* a_q, const void* a_tc, const float* a_s, const int8_t* w_q,
                       const uint16_t* scale_f16, int64_t M, int64_t N, int64_t K,
                       uint16_t* y_bf16, int path, egopq_stream_t stream);

/* ---- dense bf16 twin (comparison kernel) -------------------------------------------
 * y[m,n] = bf16( sum_k x[m,k] * w[n,k] ), x bf16 [M][K], w dense bf16 [N][K]
 * row-major, y bf16 [M][N]; K % 128 == 0, N % 128 == 0.
 * The W4A16 tensor-core pipeline with the int4 unpack taken out: the same
 * warp roles, shared-memory stages, TMEM buffers, per-128-K-group drains and
 * epilogue, with the weight tile staged by TMA and copied into the MMA operand
 * as it is. Timed beside the packed kernels it measures what the int4 unpack
 * costs ("OSCAR PR #20", commit message: a bf16 twin kernel of identical
 * structure as the fair speed baseline); egopq_dequant_w4 plus any dense
 * library GEMM is the other comparison. Not a quantized path. */
int egopq_bf16_gemm_twin(const uint16_t* x_bf16, const uint16_t* w_bf16, int64_t M, int64_t N,
                         int64_t K, uint16_t* y_bf16, egopq_stream_t stream);

/* ---- support, status --------------------------------------------------------------
 * 1 if (M, N, K, group, variant) is accepted by the parity-tested kernels on
 * the current device, 0 if not. It claims nothing the kernels do not run (a
 * capability query that accepted a format its kernel then broke on is the
 * failure recorded in "Serve a pre-quantized int8 weight-only DiT ...",
 * amendment comment). */
int egopq_supported(int64_t M, int64_t N, int64_t K, int group, int variant);

/* Synchronize `stream`, then read and clear the device error word: EGOPQ_OK,
 * EGOPQ_ERR_TIMEOUT if a kernel's bounded wait expired since the last call,
 * EGOPQ_ERR_DEVICE_INDEX if a debug build's index check failed,
 * EGOPQ_ERR_INVALID_ARG if egopq_pack_w4_gptq met a zero point it cannot store, or
 * EGOPQ_ERR_CUDA if the synchronization itself failed. Every wait inside the
 * kernels is bounded (2 s); once one expires its kernel's results are invalid,
 * and kernels launched before this call reads the word may give up early. */
int egopq_device_status(egopq_stream_t stream);

/* Human-readable text for the calling thread's most recent failure. */
const char* egopq_last_error_string(void);

/* ---- debug build -------------------------------------------------------------------
 * The library also builds as libegopq_debug.so (EGOPQ_DEBUG): the same kernels
 * with device-side read-index checks on the packed-weight record copies, the
 * per-group scale reads and the activation, group-sum and token reads of the
 * GEMV and tensor-core paths. A failed check records itself in the device
 * error word (egopq_device_status then returns EGOPQ_ERR_DEVICE_INDEX) and the
 * read goes to a known-valid address instead, so a bad index never becomes a
 * memory fault; results of such a call are invalid.
 * egopq_debug_build: 1 in the debug build, 0 otherwise.
 * egopq_debug_set_record_limit: lower the byte size the packed-record checks
 * allow (0 restores each buffer's own size), for tests that make the checks
 * fire while every read stays inside the real buffer; EGOPQ_ERR_INVALID_ARG
 * in a release build. Not thread-safe against kernels in flight. */
int egopq_debug_build(void);
int egopq_debug_set_record_limit(uint64_t bytes);

/* Self-test of the bounded-wait machinery: launches one CTA that waits on an
 * mbarrier nothing will complete, with a deadline of `timeout_us`
 * microseconds (1..1000000). The kernel gives up, records the timeout in the
 * device error word and returns; egopq_device_status then reports
 * EGOPQ_ERR_TIMEOUT. No fault, trap or hang is involved. */
int egopq_selftest_timeout(int timeout_us, egopq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* EGOPQ_H */
