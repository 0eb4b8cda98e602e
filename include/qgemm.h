/*
 * qgemm.h -- C ABI of the GB300 (sm_103a) quantized-weight GEMM library.
 *
 * The library computes Y = X . dequant(Wq)^T where the weights are 4-bit codes that are
 * dequantized inside the kernel:
 *   - INT4, symmetric: two's-complement q in [-8, 7], w = q * s[n, k/g], BF16 scales;
 *   - INT4 with zero points: q, z in [0, 15], w = (q - z) * s[n, k/g], BF16 scales;
 *   - MXFP4: e2m1 codes with one E8M0 exponent e per 32 K-elements, w = e2m1(q) * 2^(e-127).
 * Activations are BF16 (W4A16) or FP8 e4m3 with one float32 scale per token (W4A8).
 * There is a dense form and an MoE grouped form over expert-sorted rows.
 *
 * The problem statement follows "Humming wird angekündigt" (vLLM blog, German edition):
 * section "Eine einheitliche Quantisierungsdarstellung" (weight format, scale granularity,
 * scale dtype, zero points and secondary scales as separate parameters; activations with
 * their own format), section "Tuning und JIT-Kompilierung für jeden Workload" (a
 * preprocessing step validates, pads and repacks weights into a kernel layout; a layer is
 * described by shapes, dtypes and quantization parameters), and sections "WnA16" and
 * "W8A8 / W4A8 / W4A4" (dense and MoE grouped paths).
 *
 * Conventions for every call:
 *   - Pointers named as device pointers must be CUDA device memory of the current device;
 *     the caller owns all memory.  The library allocates nothing.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).  Calls are
 *     asynchronous on it.  Argument errors are returned synchronously before any launch;
 *     a failed launch returns QGEMM_ERR_CUDA.
 *   - Conditions that only the GPU can see (a packed buffer whose header does not match
 *     the descriptor, an invalid scale or zero point found by qgemm_repack, a bounded wait
 *     that gave up) are recorded in a per-device status word; read it with
 *     qgemm_device_status() after synchronizing.
 *   - Matrices are row-major with an explicit leading dimension counted in elements.
 *   - Y is overwritten (no accumulation into Y).  M = 0 is a no-op that returns QGEMM_OK.
 *   - Concurrent calls on different streams are safe when they use separate workspaces.
 */
#ifndef QGEMM_H
#define QGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QGEMM_OK = 0,
  QGEMM_ERR_INVALID_ARG = 1,   /* bad pointer, size, stride or descriptor field        */
  QGEMM_ERR_UNSUPPORTED = 2,   /* valid but not implemented combination                */
  QGEMM_ERR_ALIGNMENT = 3,     /* pointer or leading dimension misaligned for TMA      */
  QGEMM_ERR_WORKSPACE = 4,     /* workspace missing or smaller than required           */
  QGEMM_ERR_BAD_PACKED = 5,    /* (device status) packed header does not match desc    */
  QGEMM_ERR_CUDA = 6,          /* a CUDA runtime call or launch failed                 */
  QGEMM_ERR_TIMEOUT = 7,       /* (device status) a bounded device wait gave up (limit:
                                  4 s, or QGEMM_TIMEOUT_MS milliseconds from the env)  */
  QGEMM_ERR_NO_DEVICE = 8,     /* no sm_103 device is current                          */
  QGEMM_ERR_BAD_VALUE = 9      /* (device status) repack met an E8M0 of 255, a non-finite
                                  BF16 scale or a zero point above 15; a MoE call met
                                  invalid offsets or a row index past the end of X     */
} qgemm_status;

typedef enum {
  QGEMM_W_INT4_SYM = 0, QGEMM_W_UINT4_ZP = 1, QGEMM_W_MXFP4 = 2, QGEMM_W_MXINT4 = 3,
  QGEMM_W_NVFP4 = 4
} qgemm_wfmt;
typedef enum { QGEMM_SCALE_BF16 = 0, QGEMM_SCALE_E8M0 = 1, QGEMM_SCALE_E4M3 = 2 } qgemm_sdtype;
typedef enum {
  QGEMM_A_BF16 = 0, QGEMM_A_FP8E4M3_TOKEN = 1, QGEMM_A_MXFP4 = 2,
  QGEMM_A_FP8E4M3_TOKEN_FP4MMA = 3
} qgemm_afmt;

/*
 * Weight descriptor ("layer config"): one quantized weight matrix W of logical shape
 * [N, K] (Y = X . W^T).  Supported combinations:
 *   wfmt INT4_SYM : sdtype BF16, has_zp 0, group_size 32 or a multiple of 64, K % group == 0
 *   wfmt UINT4_ZP : sdtype BF16, has_zp 1, group_size as above
 *   wfmt MXFP4    : sdtype E8M0, has_zp 0, group_size 32 (afmt BF16, FP8E4M3_TOKEN,
 *                   FP8E4M3_TOKEN_FP4MMA, or MXFP4 for W4A4; only MXFP4 weights pair with
 *                   FP8 or MXFP4 activations)
 *   wfmt MXINT4   : sdtype E8M0, has_zp 0, group_size 32, afmt BF16
 *                   (w = q * 2^(e - 127), q the two's-complement nibble)
 *   wfmt NVFP4    : sdtype E4M3, has_zp 0, group_size 16, afmt BF16
 *                   (w = e2m1(q) * s * g, g the per-tensor scale of qgemm_repack_scaled)
 * K must be a multiple of 32; N >= 1 is arbitrary (the packed form pads it).
 * MXINT4 and NVFP4 are the formats of the B300 MoE results in "Humming wird
 * angekündigt", section "WnA16".
 * afmt names the activation format the packed weights will be multiplied with.  The two FP8
 * forms are two W4A8 kernels for the same arithmetic: FP8E4M3_TOKEN widens each e2m1 weight
 * to an e4m3 byte in registers and feeds the tensor core FP8 x FP8; FP8E4M3_TOKEN_FP4MMA
 * keeps the weights as they are and feeds them to the tensor core as FP4 operands of the
 * block-scaled FP8/FP6/FP4 MMA (no decode, the weight codes go from HBM to shared memory by
 * TMA).  qgemm_w4a8 and the MoE calls with QGEMM_A_FP8E4M3_TOKEN activations accept either
 * packing.
 * flags: QGEMM_FLAG_BATCH_INVARIANT (below) or 0; other bits are invalid.  The packed form
 * does not depend on flags.
 */
/*
 * Batch invariance ("Humming wird angekündigt", section "Tuning und JIT-Kompilierung für
 * jeden Workload": a Compute Config option).  Calls on a descriptor with this flag run one
 * schedule for every M: 128-token tiles with one MMA issuer, no K cut and no stream-K.  Each
 * output row is then computed with the same operations in the same order whatever the
 * batch: the same bits for X row m at any M, and in an MoE grouped call whatever the other
 * experts' rows.  Small M runs slower than with the default schedules (a full 128-token
 * MMA per stage); qgemm_moe_indexed refuses the flag (QGEMM_ERR_UNSUPPORTED).
 */
#define QGEMM_FLAG_BATCH_INVARIANT 1
typedef struct {
  int32_t wfmt;        /* qgemm_wfmt   */
  int32_t sdtype;      /* qgemm_sdtype */
  int32_t group_size;  /* K elements per scale */
  int32_t has_zp;      /* 1 iff wfmt == QGEMM_W_UINT4_ZP */
  int32_t afmt;        /* qgemm_afmt   */
  int32_t flags;       /* 0 or QGEMM_FLAG_BATCH_INVARIANT */
  int64_t N;
  int64_t K;
} qgemm_wdesc;

/* Library version (major * 10000 + minor * 100 + patch). */
int32_t qgemm_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* qgemm_status_str(qgemm_status s);

/*
 * Validate a descriptor without touching any device (QGEMM_OK if supported).
 * ("Humming wird angekündigt", section "Tuning und JIT-Kompilierung für jeden Workload":
 * the preprocessing validates the parameters.)
 */
qgemm_status qgemm_check_desc(const qgemm_wdesc* desc);

/*
 * Size in bytes of the packed (repacked) form of one weight matrix, or 0 if `desc` is
 * invalid.  For an MoE layer, expert e's packed weights start at e * qgemm_packed_bytes().
 * The size is a multiple of 256.  (Same section: the preprocessing pads the dimensions
 * and repacks into the kernel layout.)
 */
size_t qgemm_packed_bytes(const qgemm_wdesc* desc);

/*
 * Offline preprocessing ("Humming wird angekündigt", section "Tuning und
 * JIT-Kompilierung für jeden Workload": validate parameters, pad dimensions, repack into
 * the kernel layout).  Reads the canonical weight tensors and writes the packed form.
 *   codes  : device uint8 [N, K/2]; element k of row n is in byte k/2, even k in the low
 *            nibble.  INT4_SYM and MXINT4 nibbles are two's complement; UINT4_ZP nibbles
 *            are 0..15; MXFP4 and NVFP4 nibbles are e2m1 codes (bit 3 sign).
 *   scales : device [N, K/group] row-major: uint16 BF16 bit patterns, or uint8 E8M0, or
 *            uint8 E4M3 (OCP "fn": bit 7 sign, exponent bias 7, S.1111.111 NaN).
 *   zeros  : device uint8 [N, K/group] with values 0..15 (UINT4_ZP), else NULL.
 *   packed : device buffer of qgemm_packed_bytes(desc) bytes, 256-byte aligned.
 * Values the format forbids (E8M0 = 255, a NaN/Inf BF16 scale, a NaN E4M3 scale, a zero
 * point > 15) set QGEMM_ERR_BAD_VALUE in the device status word.  An NVFP4 matrix packed
 * here has per-tensor scale 1.
 */
qgemm_status qgemm_repack(const qgemm_wdesc* desc, const uint8_t* codes, const void* scales,
                          const uint8_t* zeros, void* packed, void* stream);

/*
 * qgemm_repack, recording NVFP4's per-tensor (second-level) scale g in the packed header:
 * every GEMM on these weights multiplies its output by g (in FP32, with the per-channel
 * scale, before the BF16 rounding of Y), so an MoE layer has one g per expert.  g must be
 * finite (QGEMM_ERR_INVALID_ARG) and 1 for the other formats (QGEMM_ERR_UNSUPPORTED).
 * "Humming wird angekündigt", section "Eine einheitliche Quantisierungsdarstellung"
 * (secondary scales are a parameter of the weight description).
 */
qgemm_status qgemm_repack_scaled(const qgemm_wdesc* desc, const uint8_t* codes,
                                 const void* scales, const uint8_t* zeros, float global_scale,
                                 void* packed, void* stream);

/*
 * Workspace bytes that qgemm_w4a16 / qgemm_w4a8 need for any M <= M_max.  In this order:
 *   - INT4 weights with BF16 scales only: an FP16 copy of X, [M][K] FP16 plus one FP32 row
 *     scale per row (qgemm_act_copy_bytes).  These layouts run the tensor cores on FP16
 *     operands: a dequantized weight (q - z) * s needs up to 12 significant bits, BF16
 *     holds 8 and FP16 11, so the kernel rounds it to FP16; X is converted exactly (each
 *     row times a power of two, 2^-e_m, into FP16's range) by a pre-pass launched before
 *     the GEMM, and the epilogue takes the powers of two back;
 *   - the FP32 partial sums of the output tiles whose K range the schedule cuts over
 *     several CTAs (split-K or stream-K; one 128 x token-tile slot per contributing CTA)
 *     and one arrival counter per cut tile.  Cuts are made up to M = 1024; above it only
 *     stream-K over the leftover tiles, for K >= 16384, and only when the workspace
 *     passed holds its partial sums (a smaller one gets whole tiles, never an error).
 * 0 when neither applies to any M <= M_max.  The workspace must be 256-byte aligned and
 * zero-filled before its first use; every successful call leaves the counters zero again
 * (the partial sums and the activation copy are overwritten by every call), so one
 * zero-filled buffer can be reused by consecutive calls on one stream.
 * The K cuts are the pages' Stream-K planning ("Humming wird angekündigt", section
 * "Leistungsoptimierung basierend auf Geräteparametern"); FP16 and BF16 are both 16-bit
 * activation types of the W4A16 path (same page, section "WnA16").
 */
size_t qgemm_workspace_bytes(const qgemm_wdesc* desc, int64_t M_max);

/*
 * Bytes of the FP16 activation copy that the GEMMs on INT4 weights with BF16 scales keep
 * at the head of their workspace for x_rows rows of X (see qgemm_workspace_bytes): the
 * smallest workspace the MoE calls accept for such weights (x_rows = R for
 * qgemm_moe_grouped, T for qgemm_moe_indexed).  0 for every other layout, an invalid
 * descriptor or x_rows <= 0.
 */
size_t qgemm_act_copy_bytes(const qgemm_wdesc* desc, int64_t x_rows);

/*
 * Dense W4A16:  Y[m, n] = c[n] * sum_k X[m, k] * W[n, k] + b[n]   (c = 1 when
 *               chan_scale == NULL, b = 0 when bias == NULL; for NVFP4, W includes the
 *               per-tensor scale g, applied to the FP32 sum; the sum, scaled, plus the bias
 *               is rounded to BF16 once)
 *   packed     : device, from qgemm_repack with desc->afmt == QGEMM_A_BF16
 *   X          : device BF16 [M, ldx], 16-byte aligned, ldx % 8 == 0, ldx >= K
 *   chan_scale : device float32 [N] secondary per-channel scale, or NULL
 *   bias       : device float32 [N], 4-byte aligned, added after every scale, or NULL
 *   Y          : device BF16 [M, ldy], 4-byte aligned, ldy >= N, ldy even
 *   ws         : device workspace (see qgemm_workspace_bytes), may be NULL when
 *                qgemm_workspace_bytes(desc, M) == 0
 * "Humming wird angekündigt", section "WnA16"; scaling and bias addition fused into the
 * output stage: section "Gemeinsam genutzte CUDA-Komponenten".
 */
qgemm_status qgemm_w4a16(const qgemm_wdesc* desc, const void* packed, const void* X, int64_t M,
                         int64_t ldx, const float* chan_scale, const float* bias, void* Y,
                         int64_t ldy, void* ws, size_t ws_bytes, void* stream);

/*
 * Device staging bytes that qgemm_w4a16_host needs for any M <= M_max: two buffers of a
 * chunk's X rows and two of its Y rows (a chunk is all M rows up to 512, else M / 16
 * rounded up to a multiple of 256 and at least 512).  0 for an invalid descriptor or
 * M_max <= 0.
 */
size_t qgemm_host_staging_bytes(const qgemm_wdesc* desc, int64_t M_max);

/*
 * Dense W4A16 with X and Y in host memory: Y_host = qgemm_w4a16(X_host) with the copies
 * overlapped.  The rows are cut into chunks (see qgemm_host_staging_bytes); chunk i is
 * copied in on a library-owned stream, multiplied on `stream` into `staging`, and copied out
 * on a second library-owned stream while chunk i + 1 is multiplied (a single chunk runs all
 * three steps on `stream`).  Returns once the work is enqueued; work ordered after the call
 * on `stream` sees Y_host complete.
 *   X_host  : host BF16 [M, ldx] (ldx >= K); page-locked memory (cudaHostAlloc /
 *             cudaHostRegister) lets the copies run asynchronously and at full speed
 *   Y_host  : host BF16 [M, ldy] (ldy >= N), same advice
 *   staging : device buffer of qgemm_host_staging_bytes(desc, M) bytes, 256-byte aligned,
 *             owned by the caller and busy until `stream` reaches the end of the call
 *   ws, chan_scale, bias, stream : as for qgemm_w4a16 (the chunks run one after another
 *             on `stream`, so they share one workspace)
 * Errors: QGEMM_ERR_INVALID_ARG (descriptor, null pointers, ld too small, FP8 descriptor),
 * QGEMM_ERR_WORKSPACE (staging missing or too small), QGEMM_ERR_ALIGNMENT, any status of
 * qgemm_w4a16, QGEMM_ERR_CUDA when a copy or an event could not be enqueued (chunks already
 * enqueued then still run, and `stream` is not ordered after them: synchronize the device
 * before reusing staging or reading Y_host).  Calls from several host threads are
 * serialized while they enqueue (the library streams and events are shared per device).
 * The pages time the GEMM kernels alone; this entry point is a library convenience that
 * the end-to-end measurement uses.
 */
qgemm_status qgemm_w4a16_host(const qgemm_wdesc* desc, const void* packed, const void* X_host,
                              int64_t M, int64_t ldx, const float* chan_scale, const float* bias,
                              void* Y_host, int64_t ldy, void* staging, size_t staging_bytes,
                              void* ws, size_t ws_bytes, void* stream);

/*
 * Tokenwise FP8 activation quantization (the input of W4A8): per row m,
 * s[m] = max_k |X[m, k]| / 448 (1 when the row is zero) and Xq[m, k] = e4m3 code of
 * X[m, k] / s[m], rounded to nearest even with saturation, all in float32.
 *   X : device BF16 [M, ldx];  Xq : device uint8 [M, ldq];  tok_scale : device float32 [M]
 * "Humming wird angekündigt", section "End-to-End-Inferenzleistung" (tokenwise FP8).
 */
qgemm_status qgemm_quant_act_fp8(const void* X, int64_t M, int64_t K, int64_t ldx, uint8_t* Xq,
                                 int64_t ldq, float* tok_scale, void* stream);

/*
 * Dense W4A8 (MXFP4 weights x tokenwise FP8 activations):
 *   Y[m, n] = tok_scale[m] * c[n] * sum_k e4m3(Xq[m, k]) * W[n, k] + b[n]
 *   packed : device, from qgemm_repack with desc->wfmt == MXFP4 and desc->afmt ==
 *            FP8E4M3_TOKEN or FP8E4M3_TOKEN_FP4MMA (the kernel follows the packing)
 *   Xq     : device uint8 e4m3 [M, ldx], 16-byte aligned, ldx % 16 == 0
 *   tok_scale : device float32 [M];  other arguments as for qgemm_w4a16.
 * "Humming wird angekündigt", section "W8A8 / W4A8 / W4A4".
 */
qgemm_status qgemm_w4a8(const qgemm_wdesc* desc, const void* packed, const uint8_t* Xq, int64_t M,
                        int64_t ldx, const float* tok_scale, const float* chan_scale,
                        const float* bias, void* Y, int64_t ldy, void* ws, size_t ws_bytes,
                        void* stream);

/*
 * MXFP4 activation quantization (the input of W4A4), the OCP Microscaling conversion: per
 * row m and block of 32 K-elements b, E = floor(log2 max |X[m, 32b .. 32b+31]|) - 2 + 127
 * clamped to [0, 254] (127 for an all-zero block), and each element X / 2^(E - 127) rounded
 * to the nearest e2m1 value (ties to even, saturating at +-6).
 *   X      : device BF16 [M, ldx], K % 32 == 0, ldx >= K
 *   Xq     : device uint8 [M, ldq] codes, ldq >= K / 2, 4-byte aligned rows; element 2j
 *            of a row in the low nibble of byte j
 *   x_exps : device uint8 [M, ld_exps] E8M0 exponents, one per 32 K, 16-byte aligned;
 *            ld_exps a multiple of 16 and >= ceil(K / 128) * 4 (blocks past K up to a whole
 *            128-K block are written as 127; the rest of the row is not touched)
 * "Humming wird angekündigt", section "W8A8 / W4A8 / W4A4" (MX formats on Blackwell's tensor
 * cores); the conversion itself is the OCP Microscaling format's.
 */
qgemm_status qgemm_quant_act_mxfp4(const void* X, int64_t M, int64_t K, int64_t ldx, uint8_t* Xq,
                                   int64_t ldq, uint8_t* x_exps, int64_t ld_exps, void* stream);

/*
 * Dense W4A4 (MXFP4 weights x MXFP4 activations, both block-scaled by E8M0 per 32 K):
 *   Y[m, n] = c[n] * sum_k e2m1(Xq[m, k]) 2^(x_exps[m, k/32] - 127) W[n, k] + b[n]
 * computed by the tensor cores' block-scaled FP4 MMA (kind::mxf4): both operands' products
 * are exact, the sum is FP32, Y is rounded to BF16 once.
 *   packed : device, from qgemm_repack with desc->wfmt == MXFP4, desc->afmt == QGEMM_A_MXFP4
 *   Xq, ldq, x_exps, ld_exps : from qgemm_quant_act_mxfp4; Xq 16-byte aligned, ldq % 16 == 0,
 *            x_exps 16-byte aligned, ld_exps % 16 == 0 (both are read by TMA)
 *   chan_scale, bias, Y, ldy, ws, ws_bytes, stream : as for qgemm_w4a16
 * "Humming wird angekündigt", section "W8A8 / W4A8 / W4A4" (W4A4 on B300 and SM121).
 */
qgemm_status qgemm_w4a4(const qgemm_wdesc* desc, const void* packed, const uint8_t* Xq, int64_t M,
                        int64_t ldq, const uint8_t* x_exps, int64_t ld_exps,
                        const float* chan_scale, const float* bias, void* Y, int64_t ldy,
                        void* ws, size_t ws_bytes, void* stream);

/*
 * MoE grouped GEMM over expert-sorted rows: for each expert e, rows
 * expert_offsets[e] .. expert_offsets[e+1]-1 of X are multiplied by expert e's weights.
 *   desc           : per-expert weight descriptor (all experts share it)
 *   packed         : device, E packed matrices, expert e at e * qgemm_packed_bytes(desc)
 *   afmt           : QGEMM_A_BF16 (X is BF16) or QGEMM_A_FP8E4M3_TOKEN (X is e4m3 and
 *                    tok_scale holds one float32 per row; desc->afmt either FP8 form)
 *   X              : device [R, ldx] sorted rows; padding rows should be zero
 *   bias           : device float32 [E][N] (expert e's bias at e * N), added to that
 *                    expert's rows after every scale, or NULL
 *   expert_offsets : device int32 [E+1], non-decreasing, offsets[0] = 0, offsets[E] = R
 *   Y              : device BF16 [R, ldy]; rows of every expert are written
 *   ws, ws_bytes   : device workspace, 256-byte aligned and zero-filled before its first
 *                    use (calls leave it reusable, as for qgemm_w4a16).  Required for INT4
 *                    weights with BF16 scales: at least qgemm_act_copy_bytes(desc, R), the
 *                    FP16 activation copy (QGEMM_ERR_WORKSPACE otherwise); optional (NULL)
 *                    for the other formats.  With ws_bytes >=
 *                    qgemm_moe_workspace_bytes(desc, E, R) the kernel may cut the K range
 *                    of the tiles left over after whole rounds of tiles over several CTAs
 *                    (stream-K), which evens out the work when few tiles exist; with less
 *                    every CTA runs whole tiles.
 * "Humming wird angekündigt", section "WnA16" (Indexed and Grouped MoE paths; tokens are
 * distributed over experts and the work per expert varies with the load).
 */
qgemm_status qgemm_moe_grouped(const qgemm_wdesc* desc, const void* packed, int32_t E,
                               int32_t afmt, const void* X, int64_t R, int64_t ldx,
                               const float* tok_scale, const float* bias,
                               const int32_t* expert_offsets, void* Y, int64_t ldy, void* ws,
                               size_t ws_bytes, void* stream);

/*
 * MoE GEMM over rows gathered by index (the "Indexed" MoE path): sorted position r of
 * expert e's block [expert_offsets[e], expert_offsets[e+1]) takes X row row_index[r], so
 * the caller needs no copy of X sorted by expert.
 *   Y[r, :] = X[row_index[r], :] * W_e^T   (times tok_scale[row_index[r]] for FP8 X)
 *             + bias[e, :]
 * and a padding position (row_index[r] < 0) reads a zero row of X (its output is the bias).
 *   X              : device [T, ldx] rows in token order (BF16, or e4m3 with tok_scale [T])
 *   bias           : as for qgemm_moe_grouped ([E][N] or NULL)
 *   expert_offsets : device int32 [E+1], non-decreasing, offsets[0] = 0, offsets[E] = R
 *   row_index      : device int32 [R], values in [0, T) or negative; 4-byte aligned
 *   Y              : device BF16 [R, ldy] in sorted order
 *   ws, ws_bytes   : as for qgemm_moe_grouped, with the activation copy for the T rows
 *                    of X: qgemm_act_copy_bytes(desc, T) at least for INT4 weights with
 *                    BF16 scales; qgemm_moe_indexed_workspace_bytes(desc, E, afmt, T, R)
 *                    for the fastest schedule (below)
 * Up to 255 rows, or with less workspace, the kernel copies the indexed rows into its
 * activation tiles itself (token tiles of 16, 32 or 64 rows, from R / E), which suits the
 * few rows of decode-sized routing.  From 256 rows on, given
 * qgemm_moe_indexed_workspace_bytes, a gather kernel first writes the rows (and their token
 * or row scales) in sorted order into the workspace, and the grouped kernel with its wider
 * tiles runs on that copy: the same result, one more launch, and the rows are read from X
 * once per call instead of once per weight tile.  An index >= T is an error
 * (QGEMM_ERR_BAD_VALUE in the device status word, see qgemm_device_status) and that row
 * reads as zeros.  QGEMM_ERR_UNSUPPORTED when qgemm_force_config forces a token tile
 * above 64 (a forced token tile also keeps the in-kernel gather).
 * "Humming wird angekündigt", section "WnA16" (Indexed and Grouped MoE paths).
 */
qgemm_status qgemm_moe_indexed(const qgemm_wdesc* desc, const void* packed, int32_t E,
                               int32_t afmt, const void* X, int64_t T, int64_t ldx,
                               const float* tok_scale, const float* bias,
                               const int32_t* expert_offsets, const int32_t* row_index,
                               int64_t R, void* Y, int64_t ldy, void* ws, size_t ws_bytes,
                               void* stream);

/*
 * Workspace bytes that let qgemm_moe_grouped or qgemm_moe_indexed use stream-K for E
 * experts and R sorted rows (token tile from R / E): the FP16 activation copy of R rows
 * for INT4 weights with BF16 scales (qgemm_act_copy_bytes), then FP32 partial-sum slots
 * for twice the SM count plus one arrival counter per SM.  0 for an invalid descriptor,
 * E < 1 or R <= 0.
 */
size_t qgemm_moe_workspace_bytes(const qgemm_wdesc* desc, int32_t E, int64_t R);

/*
 * Workspace bytes for the fastest schedule of qgemm_moe_indexed with afmt activations
 * (QGEMM_A_BF16 or QGEMM_A_FP8E4M3_TOKEN), T rows of X and R sorted positions: the FP16
 * activation copy of the T rows for INT4 weights with BF16 scales, then from R = 2048 on the
 * sorted copy of the R rows (R * K * 2 bytes, or R * K for FP8, each part rounded up to 256)
 * and their FP32 scales (FP8 or FP16 activations), then the stream-K slots as in
 * qgemm_moe_workspace_bytes.  0 for an invalid descriptor or afmt, E < 1, T < 0 or R <= 0.
 */
size_t qgemm_moe_indexed_workspace_bytes(const qgemm_wdesc* desc, int32_t E, int32_t afmt,
                                         int64_t T, int64_t R);

/*
 * Test hook: unpack a packed matrix back to BF16 W[n, k] = RNE_bf16(dequant) through the
 * same register decode the GEMM kernels use.  W_out: device BF16 [N, K] (row stride K).
 * NVFP4: the decoded e2m1 * s (exact) times the per-tensor scale g, rounded to BF16 once.
 */
qgemm_status qgemm_dequant_debug(const qgemm_wdesc* desc, const void* packed, void* W_out,
                                 void* stream);

/*
 * Read (and, if clear != 0, reset) the current device's status word: QGEMM_OK or the
 * first device-side error recorded since the last reset.  Synchronizes the device.
 */
qgemm_status qgemm_device_status(int32_t clear);

/*
 * Size of the device scratch built into the library for qgemm_w4a16_noalloc (8 MiB).
 */
#define QGEMM_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)

/*
 * Dense W4A16 for callers that cannot allocate a workspace -- for example code whose
 * device memory is entirely owned by another allocator (a serving framework's reserved
 * pool), or a latency-critical path that must not call cudaMalloc and its implicit
 * device synchronization.  The pages have no counterpart; this is a library convenience.
 * Same arguments and result as qgemm_w4a16 without `ws`/`ws_bytes`: the split-K scratch
 * is a fixed QGEMM_NOALLOC_SCRATCH_BYTES device array inside the library, held by every
 * GPU that loads it until the process exits.  A call needs only what its own schedule for
 * this M uses (qgemm_plan): the partial sums of the tiles it cuts (above M = 1024 only a
 * stream-K schedule, which gives way to whole tiles when the array cannot hold it), after
 * the FP16 activation copy for INT4 weights with BF16 scales (qgemm_act_copy_bytes).  A
 * call that needs more than the array returns QGEMM_ERR_WORKSPACE; use qgemm_w4a16 with a
 * workspace for it.  Arguments are checked as qgemm_w4a16 checks them, before anything is
 * enqueued.
 * Allocates nothing: no cudaMalloc/cudaFree or allocating library routine.  The first
 * call on a device that needs scratch looks up the array's device address (once per
 * device, with that device current); make that first call before any stream capture.
 * Such a call zeroes the arrival counters of its schedule inside the array, on `stream`
 * (the partial sums are written before they are read).  All calls share the one array, so
 * calls that may overlap on the GPU (different streams, or different host threads) race and
 * give wrong results; serialize them on one stream.
 */
qgemm_status qgemm_w4a16_noalloc(const qgemm_wdesc* desc, const void* packed, const void* X,
                                 int64_t M, int64_t ldx, const float* chan_scale, void* Y,
                                 int64_t ldy, void* stream);

/*
 * The schedule qgemm_w4a16 / qgemm_w4a8 would run for M rows on the current device (152
 * SMs assumed when no device is visible), given a workspace of qgemm_workspace_bytes(desc,
 * M): out[0] token tile, out[1] uniform K cut (1 = none), out[2] stream-K tiles (0 = none),
 * out[3] partial-sum slots per cut tile, out[4] CTAs.
 * Host-only (launches nothing); honours qgemm_force_config.
 * The choice is the pages' Tuning Config (tile shape, Stream-K planning; "Humming wird
 * angekündigt", sections "Tuning und JIT-Kompilierung für jeden Workload" and
 * "Leistungsoptimierung basierend auf Geräteparametern"), made by a cost model here.
 */
qgemm_status qgemm_plan(const qgemm_wdesc* desc, int64_t M, int32_t out[5]);

/*
 * Tuning override for tests and sweeps: force the token tile (16, 32, 64, 128 or 256) and
 * the schedule of the dense kernels: splits >= 1 cuts every tile's K range into that many
 * equal parts (1 = no cut), splits = -1 selects the stream-K schedule (an even share of the
 * leftover tiles' K blocks per CTA, then whole tiles; falls back to no cut where it does not
 * apply); 0 restores the built-in heuristic for that part.  Process-wide, not thread-safe.
 */
qgemm_status qgemm_force_config(int32_t token_tile, int32_t splits);

/*
 * Test aid for the kernels' bounded waits (off by default).  With skip_first_x = 1 the
 * dense calls' activation producer never issues the first activation load of each CTA,
 * so the MMA issuers' wait for it, and after it every other role's, runs into the time
 * limit: the kernel then winds down (it waits for every copy it did issue), sets
 * QGEMM_ERR_TIMEOUT in the status word (qgemm_device_status) and returns, and the context
 * stays usable.  Nothing is left in flight and no wait is removed.  timeout_ms > 0
 * replaces the wait limit (QGEMM_TIMEOUT_MS, default 4000 ms) for the following calls;
 * 0 restores it.  Process-wide, not thread-safe.  The pages' counterpart is the
 * isolation of failures so that inference survives them (the Chinese release notes,
 * v0.1.1: kernel compilation in a separate process).
 * Returns QGEMM_ERR_INVALID_ARG for skip_first_x outside {0, 1} or timeout_ms outside
 * 0..60000.
 */
qgemm_status qgemm_debug_stall(int32_t skip_first_x, int32_t timeout_ms);

#ifdef __cplusplus
}
#endif

#endif /* QGEMM_H */
