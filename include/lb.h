/*
 * lb.h -- C ABI of the GB300 (sm_103a) low-bit product library.
 *
 * The library computes the products of packed low-bit weights and quantized activations that
 * dominate per-token time in low-bit LLM inference:
 *   - ggml Q1_0     : 128 sign bits + an fp16 scale per 18-byte block;
 *   - ggml Q2_0_g64 : 64 two-bit codes (code c means weight c-1) + an fp16 scale per 18 bytes;
 *   - planar ternary: one 16-byte {u64 pos, u64 neg} beat per 64 columns of a row;
 *   - a bf16 dense head.
 *
 * Sources the operations follow:
 *   [TR] "bankml: verified low-bit inference on commodity CPUs -- a technical report",
 *        sections III.2 (Q1_0 and its arithmetic), III.3 (float order, per-token activation
 *        scales, prefill tile), III.5 (Q2_0_g64), III.8 (offset code).
 *   [BH] bankml BUILD_HISTORY.md, ledger item "P2 -- own the kernels" (q8_0 quantizer: 127/amax,
 *        round half to even; Q2_0 codes (v >> 2r) & 3).
 *   [TA] tritium.technology "Architecture": section 1 (select-accumulate), 2 (bit planes),
 *        3 (bf16 dense head), 4.1 (int32 accumulators, x = -128), 5 (w_scale and x_scale applied
 *        as two multiplies).
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is a DEVICE pointer unless stated otherwise, allocated and owned
 *     by the caller; the library allocates nothing and keeps no per-call state.
 *   - Every pointer must be 16-byte aligned (LB_ERR_ALIGN otherwise).
 *   - Matrices are row-major. Weights W are [N][K]: N output rows, K input columns.
 *     Activations are token-major [B][K] (or [M][K]); outputs are [B][N] (or [M][N]) fp32.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream). Every call
 *     only enqueues work on it and returns; results are ready when the stream is.
 *   - Every call returns LB_OK (0) or a negative LB_ERR_* code. Arguments are checked on the
 *     host before anything is enqueued; a refused call enqueues nothing. There is no fallback
 *     path: a device that is not sm_103 is refused with LB_ERR_ARCH.
 *   - Inputs must be finite; NaN or Inf activations give unspecified (but in-bounds) results.
 *   - Calls that write the same output buffer must not overlap on the GPU.
 *   - Kernels are launched with programmatic dependent launch: a GEMV may start streaming its
 *     WEIGHTS while the previous kernel of this library in the stream is still finishing, and
 *     waits for that kernel before touching activations or outputs.  lb_repack_* (the only call
 *     that writes weights) always completes before the next kernel starts; weights written by
 *     other code are read only after that code's kernels have completed.
 */
#ifndef LB_H_
#define LB_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LB_OK 0
#define LB_ERR_NULL (-1)    /* a required pointer is NULL */
#define LB_ERR_ALIGN (-2)   /* a pointer is not 16-byte aligned */
#define LB_ERR_SHAPE (-3)   /* a size is out of range or not a multiple of the block */
#define LB_ERR_BATCH (-4)   /* GEMV batch outside [1, 8] */
#define LB_ERR_ARCH (-5)    /* the current device is not compute capability 10.3 */
#define LB_ERR_LAUNCH (-6)  /* a CUDA launch or kernel setup call failed (lb_last_cuda_error) */
#define LB_ERR_DEVICE (-7)  /* a kernel gave up on a bounded wait (see lb_device_status) */

/* Name of a status code ("LB_OK", "LB_ERR_SHAPE", ...); never NULL. */
const char *lb_status_string(int status);

/* The cudaError_t value of the last CUDA call of this library that failed on the calling thread
 * (the cause behind LB_ERR_LAUNCH), then reset to 0; 0 if none failed since the last read. */
int lb_last_cuda_error(void);

/* CUDA's name for a cudaError_t value ("cudaErrorInvalidValue", ...); never NULL. */
const char *lb_cuda_error_name(int code);

/* Library version as 10000*major + 100*minor + patch. */
int lb_version(void);

/* Synchronizes `stream`, then reads and clears the current device's error word (a device
 * variable of the library whose address is looked up once per device and kept: do not use the
 * library across cudaDeviceReset).  Returns LB_OK,
 * or LB_ERR_DEVICE if a kernel of this library gave up on a bounded wait since the last call
 * (its outputs are then incomplete).  Kernels never hang: every wait gives up after about 2 s. */
int lb_device_status(void *stream);

/* Test hook for failure detection: the next Q1_0 / Q2_0_g64 / planar GEMV call (plain or
 * grouped) that runs on the streaming or lane-per-row kernel (1-2 tokens, or 3-8 tokens outside
 * the tensor-core kernel's shapes) makes its first CTA copy no weights, so that CTA's bounded
 * wait gives up after `wait_us` microseconds instead of about 2 s: the call then leaves part of
 * y unwritten and lb_device_status() reports LB_ERR_DEVICE.  Nothing faults, traps or hangs.
 * One-shot, process-wide.  1 <= wait_us <= 10^6, else LB_ERR_SHAPE.  Not for production use. */
int lb_test_inject_wait_timeout(int wait_us);

/* ---------------------------------------------------------------------------------------
 * Activation quantizers
 * ------------------------------------------------------------------------------------- */

/* q8_0 ([TR] III.2, [BH]): for every token b and every block of 32 values,
 *   amax = max|x|, d = fp16_rne(amax / 127), id = amax != 0 ? 127 / amax : 0,
 *   q[i] = round_half_even(x[i] * id)  (binary32 arithmetic, IEEE division).
 *   x : [B][K] fp32.   q : [B][K] int8 (codes in [-127, 127]).
 *   d : [B][K/32] fp16 bit patterns.
 * K % 32 == 0, K >= 32, B >= 1 (LB_ERR_SHAPE otherwise). */
int lb_quantize_q8_0(const float *x, int8_t *q, uint16_t *d, int64_t B, int64_t K,
                     void *stream);

/* Per-token absmax int8 for the planar path (the pages say only "int8 activations"; the
 * reading is the plainest one): amax = max_k |x[b][k]|, s = amax != 0 ? 127/amax : 0,
 *   q[b][k] = clamp(round_half_even(x[b][k] * s), -128, 127), x_scale[b] = amax / 127.
 *   x : [B][K] fp32.  q : [B][K] int8.  x_scale : [B] fp32.
 * K % 16 == 0, K >= 16, B >= 1. */
int lb_quantize_i8_absmax(const float *x, int8_t *q, float *x_scale, int64_t B, int64_t K,
                          void *stream);

/* ---------------------------------------------------------------------------------------
 * Load-time repack: split the 18-byte source blocks into two aligned planes.
 *   blocks18 : [N][K/QK][18] source bytes (fp16 d little-endian, then 16 data bytes);
 *              QK = 128 for Q1_0, 64 for Q2_0_g64. This pointer needs no alignment.
 *   bits     : [N][K/QK * 16] data bytes, bit order unchanged.
 *   scales   : [N][S] fp16 bit patterns, S = LB_SCALE_STRIDE(K, QK) = K/QK rounded up to a
 *              multiple of 8, so every row of scales is 16-byte aligned; the S - K/QK padding
 *              entries of each row are written as 0.
 * Q1_0: K % 128 == 0. Q2_0_g64: K % 64 == 0. N >= 1.
 * ------------------------------------------------------------------------------------- */
#define LB_SCALE_STRIDE(K, QK) ((((K) / (QK)) + 7) / 8 * 8)
int lb_repack_q1_0(const void *blocks18, int64_t N, int64_t K, uint8_t *bits, uint16_t *scales,
                   void *stream);
int lb_repack_q2_0_g64(const void *blocks18, int64_t N, int64_t K, uint8_t *codes,
                       uint16_t *scales, void *stream);

/* ---------------------------------------------------------------------------------------
 * Decode GEMVs (batch B in [1, 8] tokens sharing the weights)
 *
 * Every GEMV exists in a single-matrix form and a grouped form.  The grouped form computes the
 * products of up to LB_MAX_GROUP weight matrices with the SAME activation in one launch (for
 * example the q, k and v projections, or gate and up), which amortizes the launch over all of
 * them; each matrix has its own rows N, weights and output.  The descriptor array is read on the
 * host during the call (it may be freed on return).  Output buffers must not overlap.
 * Shared memory bounds the activation: B * K * 1.25 bytes must stay below about 120 KB
 * (LB_ERR_SHAPE otherwise).
 * ------------------------------------------------------------------------------------- */
#define LB_MAX_GROUP 64

typedef struct lb_q_matrix {
    const uint8_t *bits;     /* [N][K/QK*16] repacked sign bytes (Q1_0) or code bytes (Q2_0_g64) */
    const uint16_t *scales;  /* [N][LB_SCALE_STRIDE(K, QK)] fp16 scales */
    float *y;                /* [B][N] fp32 output */
    int32_t *isum_opt;       /* NULL, or [B][N][K/32] int32 block sums (test hook) */
    int64_t N;               /* rows, 1 <= N <= 2^30 */
} lb_q_matrix;

typedef struct lb_trit_matrix {
    const uint64_t *planes;  /* [N][K/64][2] {pos, neg} beats */
    float w_scale;           /* per-tensor weight scale */
    float *y;                /* [B][N] fp32 output */
    int32_t *acc_opt;        /* NULL, or [B][N] int32 accumulators */
    int64_t N;               /* rows, 1 <= N <= 2^30 */
} lb_trit_matrix;

/* Q1_0 x q8_0 ([TR] III.2-III.3). For token b, row n, weight block k (128 weights) and its
 * four q8_0 blocks j:
 *   isum_j = sum_{i in j} s_i * q_i  (s_i = +1 for a set bit, -1 otherwise; integer, exact)
 *   y[b][n] = sum_k d_w[n][k] * sum_j d_x[b][j] * isum_j      (fp32 accumulation)
 *   bits   : [N][K/8] repacked sign bytes (lb_repack_q1_0).
 *   scales : [N][LB_SCALE_STRIDE(K, 128)] fp16 (lb_repack_q1_0).
 *   q, d   : q8_0 activations [B][K] int8, [B][K/32] fp16 (lb_quantize_q8_0 layout).
 *   y      : [B][N] fp32.
 *   isum_opt : NULL, or [B][N][K/32] int32 that receives every isum_j (a test hook; the same
 *              kernel writes it).
 * Accuracy: |y - exact| <= 1e-5 * sum |d_w d_x isum| + 1e-6, where exact is the real-number
 * value of the formula above. K % 128 == 0; N >= 1; B in [1, 8]. */
int lb_gemv_q1_0(const uint8_t *bits, const uint16_t *scales, const int8_t *q,
                 const uint16_t *d, float *y, int32_t *isum_opt, int64_t N, int64_t K, int B,
                 void *stream);

/* Grouped Q1_0 GEMV: mats[0..G-1] (host array, 1 <= G <= LB_MAX_GROUP) against one q8_0
 * activation q, d of B tokens and K columns; same arithmetic and limits as lb_gemv_q1_0. */
int lb_gemv_q1_0_grouped(const lb_q_matrix *mats, int G, const int8_t *q, const uint16_t *d,
                         int64_t K, int B, void *stream);

/* Q2_0_g64 x q8_0 ([TR] III.5, III.8): as lb_gemv_q1_0 with 64-weight blocks, weight i of a
 * block = ((codes byte i/4) >> 2*(i%4)) & 3, minus 1, in {-1, 0, +1, +2}, and two q8_0
 * blocks per weight block.
 *   codes : [N][K/4] repacked code bytes (lb_repack_q2_0_g64).
 *   scales : [N][LB_SCALE_STRIDE(K, 64)] fp16.
 * K % 64 == 0; N >= 1; B in [1, 8]. */
int lb_gemv_q2_0_g64(const uint8_t *codes, const uint16_t *scales, const int8_t *q,
                     const uint16_t *d, float *y, int32_t *isum_opt, int64_t N, int64_t K,
                     int B, void *stream);

/* Grouped Q2_0_g64 GEMV (see lb_gemv_q1_0_grouped). */
int lb_gemv_q2_0_g64_grouped(const lb_q_matrix *mats, int G, const int8_t *q, const uint16_t *d,
                             int64_t K, int B, void *stream);

/* Planar ternary select-accumulate ([TA] 1, 2, 4.1, 5):
 *   acc[b][r] = sum_{c: pos bit set} q[b][c] - sum_{c: neg bit set} q[b][c]   (int32, exact,
 *               correct for q = -128)
 *   y[b][r]   = (float(acc) * x_scale[b]) * w_scale   (two binary32 roundings, in this order)
 *   planes  : [N][K/64][2] u64, beat g of row r = {pos, neg}, bit c <-> column 64g + c,
 *             little-endian. A column set in both planes gives an unspecified result.
 *   q       : [B][K] int8.   x_scale : [B] fp32.   y : [B][N] fp32.
 *   acc_opt : NULL, or [B][N] int32 that receives acc.
 * K % 64 == 0; K <= 2^24 / 128 (so acc is exact in int32 and in binary32); N >= 1; B in [1,8].*/
int lb_gemv_trit_planes(const uint64_t *planes, float w_scale, const int8_t *q,
                        const float *x_scale, float *y, int32_t *acc_opt, int64_t N, int64_t K,
                        int B, void *stream);

/* Grouped planar GEMV: mats[0..G-1] (host array) against one activation q, x_scale. */
int lb_gemv_trit_planes_grouped(const lb_trit_matrix *mats, int G, const int8_t *q,
                                const float *x_scale, int64_t K, int B, void *stream);

/* Dense bf16 head ([TA] 3): y[b][n] = sum_k float(W[n][k]) * x[b][k], fp32 accumulation,
 * bf16 widened exactly (16-bit left shift).
 *   w : [N][K] bf16 bit patterns.   x : [B][K] fp32.   y : [B][N] fp32.
 * Accuracy: |y - exact| <= 1e-5 * sum_k |w x| + 1e-6. K % 8 == 0; N >= 1; B in [1, 8]. */
int lb_gemv_bf16(const uint16_t *w, const float *x, float *y, int64_t N, int64_t K, int B,
                 void *stream);

/* ---- Prefill GEMM ([TR] III.3: one weight block reused across several activation columns,
 * the prefill tile).  Same arithmetic and accuracy as the GEMVs above, for M tokens:
 *   y[m][n] = sum_k d_w[n][k] * sum_j d_x[m][j] * isum_j
 * computed on the tensor cores as exact per-32-column partial products d_w * isum_j (integers
 * times an fp16 scale, exact in binary32), each scaled by d_x[m][j] with one fused multiply-add
 * into a binary32 accumulator of at most 32 + K/1024 additions.
 *   bits / codes, scales : as lb_gemv_q1_0 / lb_gemv_q2_0_g64 (repacked).
 *   q, d      : q8_0 activations [M][K] int8 and [M][K/32] fp16.
 *   y         : [M][N] fp32, overwritten.
 *   workspace : device scratch of at least lb_gemm_workspace_bytes(M, K) bytes, owned by the
 *               caller; it receives the activations converted to the tensor-core operand
 *               layout, and must not be used by another call that may run at the same time.
 * Limits: 1 <= M, N <= 2^30; K % QK == 0 (QK = 128 for Q1_0, 64 for Q2_0_g64), K <= 2^24.
 * Q2_0_g64 weight scales must satisfy |d_w| <= 32752 (so that 2 * d_w is finite in fp16);
 * fp16 scales of real weights are many orders of magnitude smaller.
 * Errors: LB_ERR_NULL, LB_ERR_ALIGN, LB_ERR_SHAPE (shape limits, or a workspace too small),
 * LB_ERR_ARCH, LB_ERR_LAUNCH; a bounded wait that gives up sets the device status
 * (lb_device_status). */
size_t lb_gemm_workspace_bytes(int64_t M, int64_t K);  /* 0 for M < 1 or K < 1 */

int lb_gemm_q1_0(const uint8_t *bits, const uint16_t *scales, const int8_t *q, const uint16_t *d,
                 float *y, int64_t M, int64_t N, int64_t K, void *workspace,
                 size_t workspace_bytes, void *stream);

int lb_gemm_q2_0_g64(const uint8_t *codes, const uint16_t *scales, const int8_t *q,
                     const uint16_t *d, float *y, int64_t M, int64_t N, int64_t K,
                     void *workspace, size_t workspace_bytes, void *stream);

/* Grouped prefill GEMM: mats[0..G-1] (host array, 1 <= G <= LB_GEMM_MAX_GROUP, read during
 * the call) against ONE q8_0 activation q, d of M tokens and K columns, in one launch -- for
 * example the q, k and v projections, or gate and up.  Same arithmetic, accuracy, workspace and
 * errors as the single-matrix calls, whose results it reproduces bit for bit; each matrix has
 * its own rows N, weights and output y [M][N].  Outputs must not overlap.  A convenience of this
 * library (the pages run projections one at a time); it lets small matrices (k, v: N = 1024)
 * share the GPU with the others instead of running alone. */
#define LB_GEMM_MAX_GROUP 8
typedef struct lb_gemm_matrix {
    const uint8_t *bits;     /* repacked sign bytes (Q1_0) or code bytes (Q2_0_g64) */
    const uint16_t *scales;  /* [N][LB_SCALE_STRIDE(K, QK)] fp16 */
    float *y;                /* [M][N] fp32 output */
    int64_t N;               /* rows, 1 <= N <= 2^30 */
} lb_gemm_matrix;

int lb_gemm_q1_0_grouped(const lb_gemm_matrix *mats, int G, const int8_t *q, const uint16_t *d,
                         int64_t M, int64_t K, void *workspace, size_t workspace_bytes,
                         void *stream);
int lb_gemm_q2_0_g64_grouped(const lb_gemm_matrix *mats, int G, const int8_t *q,
                             const uint16_t *d, int64_t M, int64_t K, void *workspace,
                             size_t workspace_bytes, void *stream);

/* ---- Planar ternary prefill GEMM ([TA] 1, 2, 4.1, 5 for the arithmetic; [TR] III.3 for the
 * prefill tile that reuses one weight tile across many tokens).  lb_gemv_trit_planes for each
 * of M tokens:
 *   acc[m][n] = sum_{c: pos bit set} q[m][c] - sum_{c: neg bit set} q[m][c]   (int32, exact)
 *   y[m][n]   = (float(acc) * x_scale[m]) * w_scale    (two binary32 roundings, in this order)
 * computed on the tensor cores with exact integer sums, so acc and y are bit-identical to the
 * GEMV's for the same token.
 *   planes    : [N][K/64][2] u64 {pos, neg} beats (layout of lb_gemv_trit_planes).
 *   q         : [M][K] int8 (for example lb_quantize_i8_absmax).   x_scale : [M] fp32.
 *   y         : [M][N] fp32, overwritten.   acc_opt : NULL, or [M][N] int32 that receives acc.
 *   workspace : device scratch of at least lb_gemm_trit_workspace_bytes(M, K) bytes (the same
 *               size as lb_gemm_workspace_bytes), owned by the caller and rewritten by every
 *               call with the activations in the tensor-core operand layout; it must not be
 *               used by another call that may run at the same time.  Its contents need no
 *               initialization.
 * Calls with few tiles split K across the CTAs of a thread-block cluster; the integer partial
 * sums are added exactly, so the split never changes a result.
 * Limits: 1 <= M, N <= 2^30; K % 64 == 0, 64 <= K <= 2^24 / 128 (so |acc| <= 2^24 and every
 * partial sum is exact in binary32).  A column set in both planes gives an unspecified result.
 * Errors: LB_ERR_NULL, LB_ERR_ALIGN, LB_ERR_SHAPE (limits, or a workspace too small),
 * LB_ERR_ARCH, LB_ERR_LAUNCH; a bounded wait that gives up sets the device status. */
size_t lb_gemm_trit_workspace_bytes(int64_t M, int64_t K);  /* 0 for M < 1 or K < 1 */

int lb_gemm_trit_planes(const uint64_t *planes, float w_scale, const int8_t *q,
                        const float *x_scale, float *y, int32_t *acc_opt, int64_t M, int64_t N,
                        int64_t K, void *workspace, size_t workspace_bytes, void *stream);

/* Grouped planar prefill GEMM: mats[0..G-1] (host array of lb_trit_matrix, 1 <= G <=
 * LB_GEMM_MAX_GROUP, read during the call) against ONE activation q, x_scale of M tokens, in one
 * launch (for example q, k and v, or gate and up).  Same arithmetic, limits, workspace and
 * errors as lb_gemm_trit_planes; each matrix has its own rows N, w_scale, output y [M][N] and
 * optional acc [M][N]; outputs must not overlap. */
int lb_gemm_trit_planes_grouped(const lb_trit_matrix *mats, int G, const int8_t *q,
                                const float *x_scale, int64_t M, int64_t K, void *workspace,
                                size_t workspace_bytes, void *stream);

/* Quantize-then-GEMM in two launches instead of three: lb_quantize_i8_absmax_tiles quantizes x
 * [M][K] fp32 exactly as lb_quantize_i8_absmax (q and x_scale bit-identical) and also writes into
 * `workspace` the activation operand tiles that lb_gemm_trit_planes* would build from q in a
 * prologue launch; lb_gemm_trit_planes_grouped_tiles then runs the grouped planar GEMM from those
 * tiles (no q argument, no prologue).  Outputs, limits and errors as lb_gemm_trit_planes_grouped.
 *   workspace : at least lb_gemm_trit_workspace_bytes(M, K) bytes; between the two calls it must
 *               not be used by any other call (the GEMM reads the tiles the quantizer wrote;
 *               several GEMMs may read them in turn, for example q|k|v and a second group).
 * Limits of the quantizer: 1 <= M <= 2^30; K % 64 == 0, 64 <= K <= 2^24 / 128.  Errors:
 * LB_ERR_NULL, LB_ERR_ALIGN (x, q, x_scale or workspace not 16-byte aligned), LB_ERR_SHAPE
 * (limits, or a workspace too small), LB_ERR_ARCH, LB_ERR_LAUNCH. */
int lb_quantize_i8_absmax_tiles(const float *x, int8_t *q, float *x_scale, int64_t M, int64_t K,
                                void *workspace, size_t workspace_bytes, void *stream);
int lb_gemm_trit_planes_grouped_tiles(const lb_trit_matrix *mats, int G, const float *x_scale,
                                      int64_t M, int64_t K, void *workspace,
                                      size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------------------------
 * Dequantization ([TR] III.4 and IV.2: every weight of a tensor dequantized and compared with
 * the reference's floats; III.2 and III.5 define w).  Every weight as the binary32 product
 *   out[n][k] = (float)w[n][k] * d      (exact: w in {-1, +1} or {-1, 0, +1, +2})
 * with d the fp16 block scale widened to binary32 (Q1_0, Q2_0_g64, from the repacked planes)
 * or w_scale (planar, w in {-1, 0, +1}).  A zero weight gives +0 or -0 with the sign of d.
 *   out_format LB_OUT_F32  : out [N][K] fp32.
 *   out_format LB_OUT_BF16 : out [N][K] bf16 bit patterns, the binary32 value rounded to
 *                            nearest, ties to even (the pages print no bf16 weights; this is
 *                            the plainest reading).
 * Q1_0: K % 128 == 0; Q2_0_g64 and planar: K % 64 == 0; 1 <= N <= 2^30, K <= 2^26.
 * Errors: LB_ERR_NULL, LB_ERR_ALIGN, LB_ERR_SHAPE (also an unknown out_format), LB_ERR_ARCH,
 * LB_ERR_LAUNCH. */
#define LB_OUT_F32 0
#define LB_OUT_BF16 1
int lb_dequantize_q1_0(const uint8_t *bits, const uint16_t *scales, int64_t N, int64_t K,
                       int out_format, void *out, void *stream);
int lb_dequantize_q2_0_g64(const uint8_t *codes, const uint16_t *scales, int64_t N, int64_t K,
                           int out_format, void *out, void *stream);
int lb_dequantize_trit_planes(const uint64_t *planes, float w_scale, int64_t N, int64_t K,
                              int out_format, void *out, void *stream);

/* ---------------------------------------------------------------------------------------
 * Base-3 packed ternary weights ([TR] III.8: 3^5 = 243 <= 256, five trits per byte, 1.6 bits
 * per trit; [TA] open questions: base-3 packing against its unpack cost).  The pages fix no
 * layout; this library's reading: byte j of 16-byte group g of a row holds columns
 * 80g + 5j + i (i = 0..4) as sum_i (t + 1) * 3^i, the lowest column in the lowest digit; a row
 * is LB_BASE3_ROW_BYTES(K) = ceil(K/80) * 16 bytes and columns past K hold trit 0.
 * ------------------------------------------------------------------------------------- */
#define LB_BASE3_ROW_BYTES(K) ((((K) + 79) / 80) * 16)

/* Load-time packing from the planar layout:
 *   planes : [N][K/64][2] u64 {pos, neg} (layout of lb_gemv_trit_planes; a column set in both
 *            planes gives an unspecified byte).
 *   packed : [N][LB_BASE3_ROW_BYTES(K)] bytes, every byte written (values 0..242).
 * Like lb_repack_*, it completes before the next kernel of this library starts.
 * K % 64 == 0, 64 <= K <= 2^24 / 128; 1 <= N <= 2^30. */
int lb_pack_base3(const uint64_t *planes, int64_t N, int64_t K, uint8_t *packed, void *stream);

/* Decode GEMV on base-3 packed weights, the planar arithmetic ([TA] 1, 4.1, 5):
 *   acc[b][r] = sum_{c: t = +1} q[b][c] - sum_{c: t = -1} q[b][c]     (int32, exact)
 *   y[b][r]   = (float(acc) * x_scale[b]) * w_scale                    (two roundings)
 * bit-identical to lb_gemv_trit_planes on the same trits.  A byte above 242 (never written by
 * lb_pack_base3) gives an unspecified, in-bounds result.
 *   packed : [N][LB_BASE3_ROW_BYTES(K)] (lb_pack_base3).   q : [B][K] int8.
 *   x_scale : [B] fp32.   y : [B][N] fp32.   acc_opt : NULL or [B][N] int32.
 * K % 64 == 0, 64 <= K <= 2^24 / 128; 1 <= N <= 2^30; B in [1, 8]; shared memory bounds the
 * activation: 32 KB + B * ceil(K/80) * 80 bytes must stay within 200 KB (LB_ERR_SHAPE). */
int lb_gemv_base3(const uint8_t *packed, float w_scale, const int8_t *q, const float *x_scale,
                  float *y, int32_t *acc_opt, int64_t N, int64_t K, int B, void *stream);

/* ---- Q2_0_g64 prefill GEMM without caller scratch.
 * No counterpart in the source pages: a convenience of this library for callers that cannot
 * allocate device memory.  Same arithmetic, accuracy, layouts and errors as lb_gemm_q2_0_g64,
 * but the converted activations go to a fixed scratch array of LB_NOALLOC_SCRATCH_BYTES inside
 * the library (a file-scope device array; the call itself allocates nothing).
 *   Limit: round_up(M, 128) * K * 2 <= LB_NOALLOC_SCRATCH_BYTES (8 MiB), e.g. M = 512 with
 *   K <= 8192, or M <= 256 with K = 12288; larger sizes are refused with LB_ERR_SHAPE before any
 *   device work.  Nothing in the scratch needs to start at zero.
 *   There is one scratch per device: calls that may run at the same time on one device (another
 *   stream, another host thread) race on it and give wrong results; serialize them.
 *   The first call on each device looks the scratch up (cudaGetSymbolAddress).  Under lazy
 *   module loading that lookup may load the library's device code, and the driver then
 *   reserves the 8 MiB array: a one-time allocation by the driver, not by this call.  Make one
 *   warm-up call per device before an allocation-free region or a stream capture.
 *   The looked-up address is kept for the life of the process: do not use the library across
 *   cudaDeviceReset (the same holds for every entry point's device error word). */
#define LB_NOALLOC_SCRATCH_BYTES (8u << 20)

int lb_gemm_q2_0_g64_noalloc(const uint8_t *codes, const uint16_t *scales, const int8_t *q,
                             const uint16_t *d, float *y, int64_t M, int64_t N, int64_t K,
                             void *stream);

#ifdef __cplusplus
}
#endif

#endif /* LB_H_ */
