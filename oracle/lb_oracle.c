/*
 * lb_oracle.c -- plain, slow, scalar CPU oracle for the packed low-bit products.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is compiled into liboracle.so, which only
 * tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg load.  The GPU
 * library (bit_matvec_lb_gb300/csrc) never includes, links or calls anything here,
 * and nothing here includes anything from it.
 *
 * Every function follows a definition printed on the source pages, step by step,
 * with no blocking, fusion or reordering beyond what that definition states:
 *
 *   [TR]  "bankml: verified low-bit inference on commodity CPUs -- a technical report"
 *         (bankml docs/TECHNICAL.md), sections III.2, III.3, III.5, III.8.
 *   [BH]  bankml BUILD_HISTORY.md, phase ledger item "P2 -- own the kernels".
 *   [TA]  tritium.technology "Architecture", sections 1, 2, 3, 4.1, 5, 8.
 *
 * Readings taken where the pages are silent:
 *   R1  q8_0 reciprocal is 127/amax (as [TR] III.2 and [BH] state), not 1/d.
 *   R2  q8_0 rounding is round-half-to-even ([TR] III.2, [BH]).
 *   R3  Q1_0 sign polarity: bit 1 means +1, bit 0 means -1 (the all-bits-set block
 *       equals +d * sum(x)).
 *   R4  Q2_0_g64 "lowest bits first": weight 4k+r of a block sits in bits 2r..2r+1
 *       of code byte k ([TR] III.5, [BH] "(v >> 2r) & 3").
 *   R5  Planar beat: little-endian u64 pos then u64 neg; bit c of each word is
 *       column 64g+c of beat g ([TA] section 2).  pos and neg both set is invalid.
 *   R6  Planar output y = (float(acc) * x_scale) * w_scale, two roundings, in that
 *       order ([TA] section 5: the reference "multiplies twice").
 *   R7  Planar activations: per-token absmax, s = 127/absmax, q = clamp(rne(x*s)),
 *       x_scale = absmax/127 (the pages say only "int8").
 *   R8  bf16 head: weight widened by a 16-bit left shift, activations fp32,
 *       y = sum_k w*x ([TA] section 3: the dense head is stored bf16 and run in f32).
 *   R9  y is token-major [B][N]; W is row-major [N][K] (rows are outputs).
 *   R10 Dequantization gives every weight as the binary32 product (float)w * d
 *       ([TR] III.4 and IV.2 compare every dequantized weight with the reference's
 *       floats); a bf16 copy is that binary32 value rounded to nearest, ties to even
 *       (the pages print no bf16 weights).  Planar weights dequantize to
 *       (float)w * w_scale with w = +1 / -1 / 0 ([TA] sections 2 and 5).
 *   R15 Base-3 packing ([TR] III.8: 3^5 = 243 <= 256, five trits per byte): byte j
 *       of 16-byte group g of a row holds columns 80g + 5j + i, i = 0..4, as the
 *       base-3 number sum_i (t + 1) * 3^i (digit i = column 80g + 5j + i, lowest
 *       column in the lowest digit); a row is ceil(K/80) groups, columns >= K hold
 *       trit 0.  The product has the planar arithmetic (R6, R7).
 *
 * Outputs of the Q1_0 / Q2_0_g64 products are produced three ways: the integer
 * block sums isum (exact), the exact value E in double, and the magnitude
 * sum_blocks |d_w * d_x * isum| that scales the acceptance bound, plus the fp32
 * chain of [TR] III.3 ("one fused multiply-add per q8_0 block, then per Q1_0
 * block") for reference.
 *
 * Compile with floating-point contraction OFF so that a*b+c is never silently
 * fused: fmaf() is written out wherever a fused operation is meant.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>

#define ORACLE_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------- */
/* IEEE 754 binary16 <-> binary32, written from the format definition.         */
/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.          */
/* ------------------------------------------------------------------------- */

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

ORACLE_API float oracle_f16_to_f32(uint16_t h)
{
    uint32_t sign = (uint32_t)(h >> 15) & 1u;
    uint32_t exp = (uint32_t)(h >> 10) & 0x1Fu;
    uint32_t frac = (uint32_t)h & 0x3FFu;
    double mag;
    if (exp == 0x1F) {
        if (frac == 0)
            return sign ? -INFINITY : INFINITY;
        /* NaN: keep the payload in the top fraction bits, quiet. */
        return bits_f32((sign << 31) | 0x7F800000u | 0x00400000u | (frac << 13));
    }
    if (exp == 0)
        mag = ldexp((double)frac, -24);            /* subnormal: frac * 2^-24 */
    else
        mag = ldexp((double)(1024u + frac), (int)exp - 25); /* (1.frac) * 2^(exp-15) */
    return (float)(sign ? -mag : mag);             /* exact: every binary16 fits binary32 */
}

/* Round-to-nearest, ties-to-even encoding of a binary32 value as binary16. */
ORACLE_API uint16_t oracle_f32_to_f16(float f)
{
    uint32_t u = f32_bits(f);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    if (isnan(f))
        return (uint16_t)(sign | 0x7E00u | ((u >> 13) & 0x3FFu));
    double a = fabs((double)f);
    if (a == 0.0)
        return sign;
    /* The representable binary16 magnitudes are k * 2^(e-10) for k in [1024, 2047]
     * in the normal range e in [-14, 15], and k * 2^-24 for k in [0, 1023] below it.
     * Find the quantum q of the binade that holds a, round a/q to an integer with
     * ties to even, and rebuild. */
    int e;
    frexp(a, &e);              /* a = m * 2^e, m in [0.5, 1)  =>  a in [2^(e-1), 2^e) */
    int unbiased = e - 1;      /* a in [2^unbiased, 2^(unbiased+1)) */
    if (unbiased < -14)
        unbiased = -14;        /* subnormal range shares the quantum 2^-24 */
    double quantum = ldexp(1.0, unbiased - 10);
    double scaled = a / quantum;                    /* exact: power-of-two divide */
    double fl = floor(scaled);
    double rem = scaled - fl;
    double k = fl;
    if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0))
        k = fl + 1.0;
    double r = k * quantum;                         /* rounded magnitude */
    if (r > 65504.0)                                /* overflow rounds to infinity */
        return (uint16_t)(sign | 0x7C00u);
    if (r < ldexp(1.0, -14)) {                      /* subnormal (or rounded to 0) */
        uint32_t sub = (uint32_t)(r / ldexp(1.0, -24));
        return (uint16_t)(sign | sub);
    }
    int re;
    double rm = frexp(r, &re);                      /* r = rm * 2^re, rm in [0.5,1) */
    uint32_t exp_field = (uint32_t)(re - 1 + 15);
    uint32_t frac_field = (uint32_t)(rm * 2048.0) - 1024u;
    return (uint16_t)(sign | (exp_field << 10) | frac_field);
}

/* bf16 is the top half of a binary32: widening is a 16-bit left shift ([TA] 3). */
ORACLE_API float oracle_bf16_to_f32(uint16_t b)
{
    return bits_f32((uint32_t)b << 16);
}

/* Round half to even, to an integer, of a finite binary32 value. */
static float round_half_even(float v)
{
    double d = (double)v;
    double fl = floor(d);
    double rem = d - fl;
    if (rem > 0.5)
        return (float)(fl + 1.0);
    if (rem < 0.5)
        return (float)fl;
    return (float)((fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0);
}

/* ------------------------------------------------------------------------- */
/* q8_0 activation quantizer ([TR] III.2; [BH] "AVX2 quantizer: 127/amax,       */
/* round-half-even").  Per block of 32:                                        */
/*   amax = max |x_i|; d = fp16(amax / 127); id = amax != 0 ? 127/amax : 0;    */
/*   q_i = round_half_even(x_i * id), all in binary32.                         */
/* x [B][K] fp32 -> q [B][K] int8, d [B][K/32] fp16 bits.  K % 32 == 0.         */
/* Returns 0, or -1 if a code falls outside [-127, 127] (never for finite x).  */
/* ------------------------------------------------------------------------- */
ORACLE_API int oracle_quantize_q8_0(const float *x, int64_t B, int64_t K,
                                    int8_t *q, uint16_t *d)
{
    int64_t nb = K / 32;
    for (int64_t b = 0; b < B; b++) {
        for (int64_t j = 0; j < nb; j++) {
            const float *xb = x + b * K + j * 32;
            float amax = 0.0f;
            for (int i = 0; i < 32; i++) {
                float a = fabsf(xb[i]);
                if (a > amax)
                    amax = a;
            }
            float dd = amax / 127.0f;
            float id = (amax != 0.0f) ? 127.0f / amax : 0.0f;
            d[b * nb + j] = oracle_f32_to_f16(dd);
            for (int i = 0; i < 32; i++) {
                float v = round_half_even(xb[i] * id);
                if (v > 127.0f || v < -127.0f)
                    return -1;
                q[b * K + j * 32 + i] = (int8_t)v;
            }
        }
    }
    return 0;
}

/* Per-token absmax int8 quantizer for the planar path (reading R7). */
ORACLE_API int oracle_quantize_i8_absmax(const float *x, int64_t B, int64_t K,
                                         int8_t *q, float *x_scale)
{
    for (int64_t b = 0; b < B; b++) {
        const float *xb = x + b * K;
        float amax = 0.0f;
        for (int64_t k = 0; k < K; k++) {
            float a = fabsf(xb[k]);
            if (a > amax)
                amax = a;
        }
        float s = (amax != 0.0f) ? 127.0f / amax : 0.0f;
        x_scale[b] = amax / 127.0f;
        for (int64_t k = 0; k < K; k++) {
            float v = round_half_even(xb[k] * s);
            if (v > 127.0f) v = 127.0f;
            if (v < -128.0f) v = -128.0f;
            q[b * K + k] = (int8_t)v;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Weight decoding, one weight at a time, from the 18-byte source blocks.      */
/* ------------------------------------------------------------------------- */

/* Q1_0 ([TR] III.2): fp16 d in bytes 0..1 (little-endian), then 16 bytes of   */
/* signs, least-significant bit first.  Weight i of the block: bit             */
/* (qs[i/8] >> (i%8)) & 1, sign +1 for a set bit (reading R3).                 */
static int q1_0_sign(const uint8_t *block18, int i)
{
    const uint8_t *qs = block18 + 2;
    int bit = (qs[i / 8] >> (i % 8)) & 1;
    return bit ? +1 : -1;
}

/* Q2_0_g64 ([TR] III.5, [BH]): fp16 d first, then 16 bytes of 2-bit codes,     */
/* lowest bits first; weight i is code (qs[i/4] >> 2*(i%4)) & 3, value c - 1.   */
static int q2_0_weight(const uint8_t *block18, int i)
{
    const uint8_t *qs = block18 + 2;
    int c = (qs[i / 4] >> (2 * (i % 4))) & 3;
    return c - 1;
}

static uint16_t block_scale_bits(const uint8_t *block18)
{
    return (uint16_t)(block18[0] | ((uint16_t)block18[1] << 8));
}

/* ------------------------------------------------------------------------- */
/* Q1_0 x q8_0 and Q2_0_g64 x q8_0 products.                                   */
/*   blocks : [N][K/QK][18] source bytes (QK = 128 for Q1_0, 64 for Q2_0_g64)  */
/*   q, dx  : q8_0 activations of B tokens, [B][K] int8 and [B][K/32] fp16     */
/*   isum   : [B][N][K/32] per q8_0-block integer dot products (may be NULL)   */
/*   y_exact: [B][N] exact value in double                                     */
/*   y_chain: [B][N] binary32 chain of [TR] III.3 (may be NULL)                */
/*   mag    : [B][N] sum over blocks |d_w * d_x * isum| (may be NULL)          */
/* For a block b of row n and its q8_0 blocks j:                               */
/*   isum_j = sum_{i in j} w_i * q_i            (integer, exact)               */
/*   E     += d_w * d_x,j * isum_j              (double: every term is exact)  */
/*   chain: t = 0; t = fmaf(d_x,j, isum_j, t) for each j; y = fmaf(d_w, t, y)  */
/* ------------------------------------------------------------------------- */
static void q_product(int qk, const uint8_t *blocks, const int8_t *q,
                      const uint16_t *dx, int64_t N, int64_t K, int64_t B,
                      int32_t *isum, double *y_exact, float *y_chain, double *mag)
{
    int64_t nblk = K / qk;            /* weight blocks per row */
    int64_t nq8 = K / 32;             /* q8_0 blocks per token row */
    int per = qk / 32;                /* q8_0 blocks per weight block */
    for (int64_t b = 0; b < B; b++) {
        for (int64_t n = 0; n < N; n++) {
            double e = 0.0, m = 0.0;
            float chain = 0.0f;
            for (int64_t blk = 0; blk < nblk; blk++) {
                const uint8_t *block18 = blocks + (n * nblk + blk) * 18;
                float dw = oracle_f16_to_f32(block_scale_bits(block18));
                float t = 0.0f;
                for (int j = 0; j < per; j++) {
                    int64_t jj = blk * per + j;      /* q8_0 block index in the row */
                    int64_t s = 0;
                    for (int i = 0; i < 32; i++) {
                        int widx = j * 32 + i;       /* weight index inside the block */
                        int w = (qk == 128) ? q1_0_sign(block18, widx)
                                            : q2_0_weight(block18, widx);
                        s += (int64_t)w * (int64_t)q[b * K + blk * qk + widx];
                    }
                    float dxf = oracle_f16_to_f32(dx[b * nq8 + jj]);
                    if (isum)
                        isum[(b * N + n) * nq8 + jj] = (int32_t)s;
                    t = fmaf(dxf, (float)s, t);
                    double term = (double)dw * (double)dxf * (double)s; /* exact */
                    e += term;
                    m += fabs(term);
                }
                chain = fmaf(dw, t, chain);
            }
            y_exact[b * N + n] = e;
            if (y_chain)
                y_chain[b * N + n] = chain;
            if (mag)
                mag[b * N + n] = m;
        }
    }
}

ORACLE_API void oracle_q1_0_product(const uint8_t *blocks, const int8_t *q,
                                    const uint16_t *dx, int64_t N, int64_t K, int64_t B,
                                    int32_t *isum, double *y_exact, float *y_chain,
                                    double *mag)
{
    q_product(128, blocks, q, dx, N, K, B, isum, y_exact, y_chain, mag);
}

ORACLE_API void oracle_q2_0_g64_product(const uint8_t *blocks, const int8_t *q,
                                        const uint16_t *dx, int64_t N, int64_t K, int64_t B,
                                        int32_t *isum, double *y_exact, float *y_chain,
                                        double *mag)
{
    q_product(64, blocks, q, dx, N, K, B, isum, y_exact, y_chain, mag);
}

/* ------------------------------------------------------------------------- */
/* Planar ternary product ([TA] sections 1, 2, 4.1, 5).                         */
/*   planes : [N][K/64][2] u64, beat g of row r = {pos, neg}; bit c <-> column  */
/*            64g + c (reading R5)                                             */
/*   acc[b][r] = sum_{c: pos} q[b][c] - sum_{c: neg} q[b][c]   (int32)         */
/*   y[b][r]   = (float(acc) * x_scale[b]) * w_scale           (reading R6)    */
/* Returns 0; -1 if some beat has a column in both planes; -2 if an            */
/* accumulator leaves the int32 range.                                         */
/* ------------------------------------------------------------------------- */
ORACLE_API int oracle_trit_planes_product(const uint64_t *planes, float w_scale,
                                          const int8_t *q, const float *x_scale,
                                          int64_t N, int64_t K, int64_t B,
                                          int32_t *acc, float *y)
{
    int64_t nbeat = K / 64;
    for (int64_t b = 0; b < B; b++) {
        for (int64_t r = 0; r < N; r++) {
            int64_t a = 0;
            for (int64_t g = 0; g < nbeat; g++) {
                uint64_t pos = planes[(r * nbeat + g) * 2 + 0];
                uint64_t neg = planes[(r * nbeat + g) * 2 + 1];
                if (pos & neg)
                    return -1;
                for (int c = 0; c < 64; c++) {
                    int64_t x = q[b * K + g * 64 + c];
                    if ((pos >> c) & 1u)
                        a += x;         /* w = +1: add     */
                    else if ((neg >> c) & 1u)
                        a -= x;         /* w = -1: subtract */
                }                        /* w =  0: skip    */
            }
            if (a > INT32_MAX || a < INT32_MIN)
                return -2;
            acc[b * N + r] = (int32_t)a;
            float t = (float)a * x_scale[b];
            y[b * N + r] = t * w_scale;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* bf16 dense head (reading R8): y[b][n] = sum_k float(W[n][k]) * x[b][k].      */
/* y_exact accumulates in double (each product is exact in double), mag is     */
/* sum_k |w * x|.                                                              */
/* ------------------------------------------------------------------------- */
ORACLE_API void oracle_bf16_product(const uint16_t *w, const float *x,
                                    int64_t N, int64_t K, int64_t B,
                                    double *y_exact, double *mag)
{
    for (int64_t b = 0; b < B; b++) {
        for (int64_t n = 0; n < N; n++) {
            double s = 0.0, m = 0.0;
            for (int64_t k = 0; k < K; k++) {
                double p = (double)oracle_bf16_to_f32(w[n * K + k]) * (double)x[b * K + k];
                s += p;
                m += fabs(p);
            }
            y_exact[b * N + n] = s;
            mag[b * N + n] = m;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Load-time split of the 18-byte blocks into two planes (the repacked layout  */
/* consumed by the GPU library):                                               */
/*   S = nblk rounded up to a multiple of 8 (scale rows are 16-byte aligned)   */
/*   scales[n][blk]           = fp16 d of block (n, blk), blk < nblk           */
/*   scales[n][blk]           = 0 for nblk <= blk < S (padding)                */
/*   bits[n][blk*16 + i]      = data byte i of block (n, blk), i in 0..15      */
/* Bit order inside the data bytes is unchanged.                               */
/* ------------------------------------------------------------------------- */
ORACLE_API void oracle_repack(const uint8_t *blocks, int64_t N, int64_t nblk,
                              uint8_t *bits, uint16_t *scales)
{
    int64_t S = (nblk + 7) / 8 * 8;
    for (int64_t n = 0; n < N; n++) {
        for (int64_t blk = 0; blk < S; blk++) {
            if (blk >= nblk) {
                scales[n * S + blk] = 0;
                continue;
            }
            const uint8_t *src = blocks + (n * nblk + blk) * 18;
            scales[n * S + blk] = block_scale_bits(src);
            for (int i = 0; i < 16; i++)
                bits[(n * nblk + blk) * 16 + i] = src[2 + i];
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Dequantization to fp32 (w * d for every weight), [N][K].                    */
/* ------------------------------------------------------------------------- */
ORACLE_API void oracle_dequant(int qk, const uint8_t *blocks, int64_t N, int64_t K,
                               float *out)
{
    int64_t nblk = K / qk;
    for (int64_t n = 0; n < N; n++) {
        for (int64_t blk = 0; blk < nblk; blk++) {
            const uint8_t *block18 = blocks + (n * nblk + blk) * 18;
            float d = oracle_f16_to_f32(block_scale_bits(block18));
            for (int i = 0; i < qk; i++) {
                int w = (qk == 128) ? q1_0_sign(block18, i) : q2_0_weight(block18, i);
                out[n * K + blk * qk + i] = (float)w * d;
            }
        }
    }
}

/* ------------------------------------------------------------------------- */
/* binary32 -> bf16, round to nearest, ties to even (reading R10), from the    */
/* IEEE 754 layout: bf16 keeps the sign, the 8 exponent bits and the top 7     */
/* fraction bits of a binary32.  The 16 dropped bits decide the rounding: more */
/* than half an ulp rounds the magnitude up, exactly half rounds to the even   */
/* neighbour (a carry out of the fraction correctly bumps the exponent, up to  */
/* infinity).  NaN stays NaN (quiet bit set); infinities are exact.            */
/* ------------------------------------------------------------------------- */
ORACLE_API uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u = f32_bits(f);
    uint32_t keep = u >> 16;
    uint32_t drop = u & 0xFFFFu;
    if ((u & 0x7F800000u) == 0x7F800000u)          /* Inf or NaN */
        return (uint16_t)(drop ? (keep | 0x0040u) : keep);
    if (drop > 0x8000u || (drop == 0x8000u && (keep & 1u)))
        keep += 1u;
    return (uint16_t)keep;
}

ORACLE_API void oracle_f32_to_bf16_array(const float *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = oracle_f32_to_bf16(x[i]);
}

/* ------------------------------------------------------------------------- */
/* Planar dequantization (readings R5, R10): out[r][64g + c] = (float)w *       */
/* w_scale with w = +1 (pos bit), -1 (neg bit), 0 (neither).  Returns 0, or -1 */
/* if some beat has a column in both planes.                                   */
/* ------------------------------------------------------------------------- */
ORACLE_API int oracle_trit_planes_dequant(const uint64_t *planes, float w_scale, int64_t N,
                                          int64_t K, float *out)
{
    int64_t nbeat = K / 64;
    for (int64_t r = 0; r < N; r++) {
        for (int64_t g = 0; g < nbeat; g++) {
            const uint64_t *beat = planes + (r * nbeat + g) * 2;   /* {pos, neg} */
            uint64_t pos = beat[0], neg = beat[1];
            if (pos & neg)
                return -1;
            for (int c = 0; c < 64; c++) {
                int w = 0;
                if ((pos >> c) & 1u)
                    w = 1;
                else if ((neg >> c) & 1u)
                    w = -1;
                out[r * K + g * 64 + c] = (float)w * w_scale;
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Base-3 packing (reading R15): trits of a row -> bytes, from the planar      */
/* layout.  out is [N][ceil(K/80) * 16].  Returns 0, or -1 if a planar beat   */
/* has a column in both planes.                                               */
/* ------------------------------------------------------------------------- */
static int planar_trit(const uint64_t *planes, int64_t nbeat, int64_t r, int64_t col)
{
    uint64_t pos = planes[(r * nbeat + col / 64) * 2 + 0];
    uint64_t neg = planes[(r * nbeat + col / 64) * 2 + 1];
    int bit = (int)(col % 64);
    if ((pos >> bit) & (neg >> bit) & 1u)
        return 2;                                   /* invalid: both planes */
    if ((pos >> bit) & 1u)
        return 1;
    if ((neg >> bit) & 1u)
        return -1;
    return 0;
}

ORACLE_API int oracle_base3_pack(const uint64_t *planes, int64_t N, int64_t K, uint8_t *out)
{
    int64_t nbeat = K / 64;
    int64_t ngroup = (K + 79) / 80;
    for (int64_t r = 0; r < N; r++) {
        for (int64_t g = 0; g < ngroup; g++) {
            for (int j = 0; j < 16; j++) {
                int value = 0, place = 1;
                for (int i = 0; i < 5; i++) {
                    int64_t col = 80 * g + 5 * j + i;
                    int t = col < K ? planar_trit(planes, nbeat, r, col) : 0;
                    if (t == 2)
                        return -1;
                    value += (t + 1) * place;       /* digit i = trit + 1 */
                    place *= 3;
                }
                out[(r * ngroup + g) * 16 + j] = (uint8_t)value;
            }
        }
    }
    return 0;
}

/* Trit of column col of a base-3 packed row (reading R15): digit i of byte j  */
/* of group g, found by dividing by 3 i times.                                 */
static int base3_trit(const uint8_t *row, int64_t col)
{
    int64_t g = col / 80;
    int j = (int)((col % 80) / 5), i = (int)(col % 5);
    int value = row[g * 16 + j];
    for (int k = 0; k < i; k++)
        value /= 3;
    return value % 3 - 1;
}

/* ------------------------------------------------------------------------- */
/* Base-3 product (readings R6, R7, R15): the planar arithmetic on trits       */
/* decoded from the packed bytes.                                              */
/*   acc[b][r] = sum_c t(r, c) * q[b][c]  (int64, asserted to fit int32)       */
/*   y[b][r]   = (float(acc) * x_scale[b]) * w_scale                           */
/* Returns 0, -1 for a byte above 242 (not a base-3 byte), -2 on overflow.     */
/* ------------------------------------------------------------------------- */
ORACLE_API int oracle_base3_product(const uint8_t *packed, float w_scale, const int8_t *q,
                                    const float *x_scale, int64_t N, int64_t K, int64_t B,
                                    int32_t *acc, float *y)
{
    int64_t row_bytes = (K + 79) / 80 * 16;
    for (int64_t r = 0; r < N; r++)
        for (int64_t i = 0; i < row_bytes; i++)
            if (packed[r * row_bytes + i] > 242)
                return -1;
    for (int64_t b = 0; b < B; b++) {
        for (int64_t r = 0; r < N; r++) {
            const uint8_t *row = packed + r * row_bytes;
            int64_t a = 0;
            for (int64_t c = 0; c < K; c++) {
                int t = base3_trit(row, c);
                if (t == 1)
                    a += q[b * K + c];
                else if (t == -1)
                    a -= q[b * K + c];
            }
            if (a > INT32_MAX || a < INT32_MIN)
                return -2;
            acc[b * N + r] = (int32_t)a;
            float tt = (float)a * x_scale[b];
            y[b * N + r] = tt * w_scale;
        }
    }
    return 0;
}

/* Every trit of a base-3 packed matrix, [N][K] int8 (reading R15). */
ORACLE_API void oracle_base3_unpack(const uint8_t *packed, int64_t N, int64_t K, int8_t *out)
{
    int64_t row_bytes = (K + 79) / 80 * 16;
    for (int64_t r = 0; r < N; r++)
        for (int64_t c = 0; c < K; c++)
            out[r * K + c] = (int8_t)base3_trit(packed + r * row_bytes, c);
}
