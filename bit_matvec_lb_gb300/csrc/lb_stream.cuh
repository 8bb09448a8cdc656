// lb_stream.cuh -- persistent, TMA-fed decode GEMV over a group of weight matrices that share
// one activation (batch of B tokens).  Used for Q1_0, Q2_0_g64 and planar ternary weights.
//
// Arithmetic (integer block sums, then float scales):
//   Q1_0     -- "bankml: verified low-bit inference on commodity CPUs -- a technical report",
//               III.2 (128 sign bits + fp16 scale, signed sum against q8_0 activations) and III.3
//               (integer sum per q8_0 block, one multiply-add per q8_0 block then per weight
//               block).
//   Q2_0_g64 -- same report, III.5 (64 two-bit codes, code c means c - 1) and III.8 (offset
//               code: sum w*x = sum c*x - sum x).
//   planar   -- tritium.technology "Architecture", sections 1-2 (select-accumulate over {pos,
//               neg} bit planes), 4.1 (int32 accumulator, exact for x = -128) and 5 (w_scale and
//               x_scale applied as two separate multiplies).
//
// GPU design (the pages' kernels are CPU/RTL prior art; nothing here translates them):
//   * Decode GEMV streams every weight byte once: it is HBM-bound, and a single 4096x4096
//     projection is only a few microseconds of HBM time, less than the fixed cost of a launch.
//     So one launch walks a whole list of matrices (for example q|k|v, or gate|up, which read
//     the same activation), and the CTAs are persistent (at most two per SM).
//   * Each CTA has one producer warp and eight consumer warps.  The producer streams tiles of
//     TR = 8*RW consecutive rows into a ring of shared-memory stages with bulk asynchronous
//     copies (TMA, non-tensor form) whose completion is counted on an mbarrier per stage;
//     consumers release a stage through a second mbarrier.  A tile of whole rows is one
//     contiguous range of the weight plane and of the (16-byte padded) scale plane, so a stage
//     costs two copies; only very long rows are sliced into columns, one copy per row.  Weight
//     copies start before the grid-dependency wait: weights are read-only for the kernels that
//     may run before this one finishes (see pdl_wait()).
//   * The B activation rows are staged once per CTA in shared memory, re-laid-out so that a
//     mask (and, for sign bits, a left shift) of a weight word lines up with one activation word:
//       Q2_0_g64: field r of every byte is masked in place (value c*4^r); four independent dp4a
//                 accumulators per q8_0 block are recombined exactly (64a0 + 16a1 + 4a2 + a3);
//       Q1_0 / planar: bit k of every byte is moved to bit 7 (x128), two dp4a chains.
//     The image is XOR-swizzled per chunk so lanes' 16-byte reads do not conflict.  Per q8_0
//     block the stage holds {d / 64, -64 * sum q}: the integer result t = 64 * isum, and
//     (d / 64) * t == d * isum exactly.
//   * Consumer warp w owns rows w*RW .. w*RW+RW-1 of every tile; lane l owns 16-byte chunks
//     l, l+32, ... of those rows.  Row sums are finished with warp shuffles: no atomics, and the
//     results do not depend on the grid size.
//   * Every wait is bounded (about 2 s); a wait that gives up sets the device error word and the
//     kernel stops instead of hanging.
#pragma once
#include <type_traits>

#include "lb_common.cuh"

namespace lb {

constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kStreamThreads = kConsumerThreads + 32;
constexpr int kMaxGroup = 64;
constexpr int kMaxStages = 4;
constexpr int kBarBytes = 2 * kMaxStages * 8;

enum Fmt { kQ1 = 0, kQ2 = 1, kTrit = 2 };

// Activation columns consumed by one 16-byte weight chunk, and 16-byte quads per chunk.
template <int F> struct FmtInfo;
template <> struct FmtInfo<kQ1> { static constexpr int kCols = 128; static constexpr int kQuads = 8; };
template <> struct FmtInfo<kQ2> { static constexpr int kCols = 64; static constexpr int kQuads = 4; };
template <> struct FmtInfo<kTrit> { static constexpr int kCols = 64; static constexpr int kQuads = 4; };

// Physical 16-byte slot of logical quad u of chunk c (conflict-free for 8 consecutive chunks).
template <int F>
__device__ __forceinline__ int quad_slot(int c, int u) {
    if (FmtInfo<F>::kQuads == 8) return c * 8 + (u ^ (c & 7));
    return c * 4 + (u ^ ((c >> 1) & 3));
}

struct StreamMat {
    const uint8_t *w;        // [N][nchunk][16] bytes: sign bits, codes or planar beats
    const uint16_t *scales;  // [N][S] fp16 (Q formats), nullptr for planar
    float *y;                // [B][N]
    int32_t *aux;            // block sums [B][N][K/32] (Q) or accumulators [B][N] (planar)
    float w_scale;           // planar tensor scale
    int32_t N;
    int32_t unit0;           // index of this matrix's first row tile
    int32_t pad;
};

struct StreamParams {
    StreamMat m[kMaxGroup];
    const int8_t *q;          // [B][K]
    const uint16_t *d;        // [B][K/32] q8_0 scales (Q formats)
    const float *x_scale;     // [B] (planar)
    int *err;                 // device error word
    int64_t K;
    int32_t G, nunits, nct, KC, nchunk, S, stages, stage_bytes, act_bytes;
    int32_t fault;            // test hook: 0, or the consumers' wait limit in us (CTA 0 starves)
};

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // every wait gives up after about 2 s

// ------------------------------------------------------------------------------------------
// Activation staging (consumer threads only).  One thread per 32-value group.
//   Q2_0_g64 image : A[t][r] = (x[16t+r], x[16t+4+r], x[16t+8+r], x[16t+12+r]), r = 0..3,
//                    lines up with the 2-bit field r of every byte of code word t.
//   Q1_0 / planar  : A[t][k] = (x[32t+k], x[32t+8+k], x[32t+16+k], x[32t+24+k]), k = 0..7,
//                    lines up with bit k of every byte of sign word t.
//   st             : per q8_0 block {scale widened to fp32 / 64, -64 * sum of its 32 codes}.
// ------------------------------------------------------------------------------------------
template <int F>
__device__ __forceinline__ void stage_activations(const int8_t *__restrict__ q,
                                                  const uint16_t *__restrict__ d, int B,
                                                  int64_t K, uint4 *__restrict__ xp,
                                                  float2 *__restrict__ st, int tid, int nthr) {
    const int ngroups = (int)((int64_t)B * K / 32);
    const int per_token = (int)(K / 32);
    for (int i = tid; i < ngroups; i += nthr) {
        const uint4 *src = reinterpret_cast<const uint4 *>(q) + 2 * (int64_t)i;
        const uint4 lo = src[0], hi = src[1];
        const int b = i / per_token, j = i % per_token;
        uint4 o0, o1;
        if (F == kQ2) {
            transpose4x4(lo.x, lo.y, lo.z, lo.w, o0.x, o0.y, o0.z, o0.w);
            transpose4x4(hi.x, hi.y, hi.z, hi.w, o1.x, o1.y, o1.z, o1.w);
        } else {
            transpose4x4(lo.x, lo.z, hi.x, hi.z, o0.x, o0.y, o0.z, o0.w);  // k = 0..3
            transpose4x4(lo.y, lo.w, hi.y, hi.w, o1.x, o1.y, o1.z, o1.w);  // k = 4..7
        }
        const int c = j * 32 / FmtInfo<F>::kCols;
        const int u0 = ((j * 32) % FmtInfo<F>::kCols) / 16;
        uint4 *tok = xp + (int64_t)b * (K / 16);
        tok[quad_slot<F>(c, u0)] = o0;
        tok[quad_slot<F>(c, u0 + 1)] = o1;
        const int s = byte_sum_s8(lo.x) + byte_sum_s8(lo.y) + byte_sum_s8(lo.z) +
                      byte_sum_s8(lo.w) + byte_sum_s8(hi.x) + byte_sum_s8(hi.y) +
                      byte_sum_s8(hi.z) + byte_sum_s8(hi.w);
        st[i] = make_float2(F != kTrit ? f16_bits_to_float(d[i]) * 0.015625f : 0.0f,
                            __int_as_float(-64 * s));
    }
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int t) {
    return t == 0 ? v.x : (t == 1 ? v.y : (t == 2 ? v.z : v.w));
}

// init + 128 * sum over the 32 weights of sign word w of bit * q (bit k of byte j <-> A[k]
// byte j).  Left shifts are additions so they may use either integer pipe; two independent
// dp4a chains.
__device__ __forceinline__ int q1_word_dot(uint32_t w, const uint4 &a0, const uint4 &a1,
                                           int init) {
    const uint32_t H = 0x80808080u;
    const uint32_t w1 = w + w, w2 = w1 + w1, w3 = w2 + w2, w4 = w3 + w3, w5 = w4 + w4,
                   w6 = w5 + w5, w7 = w6 + w6;  // w << s: bit k reaches bit 7 at s = 7 - k
    int v0 = dp4a_us(w7 & H, a0.x, init);
    int v1 = dp4a_us(w6 & H, a0.y, 0);
    v0 = dp4a_us(w5 & H, a0.z, v0);
    v1 = dp4a_us(w4 & H, a0.w, v1);
    v0 = dp4a_us(w3 & H, a1.x, v0);
    v1 = dp4a_us(w2 & H, a1.y, v1);
    v0 = dp4a_us(w1 & H, a1.z, v0);
    v1 = dp4a_us(w & H, a1.w, v1);
    return v0 + v1;
}

// init + 64 * sum over the 32 weights of code words w0, w1 (one q8_0 block) of code * q.
// Field r of every byte is masked in place (value c * 4^r), giving four independent dp4a
// accumulators that are recombined exactly: 64 S = 64 a0 + 16 a1 + 4 a2 + a3.
__device__ __forceinline__ int q2_block_dot(uint32_t w0, uint32_t w1, const uint4 &av0,
                                            const uint4 &av1, int init) {
    int a0 = dp4a_us(w0 & 0x03030303u, av0.x, 0);
    int a1 = dp4a_us(w0 & 0x0C0C0C0Cu, av0.y, 0);
    int a2 = dp4a_us(w0 & 0x30303030u, av0.z, 0);
    int a3 = dp4a_us(w0 & 0xC0C0C0C0u, av0.w, init);
    a0 = dp4a_us(w1 & 0x03030303u, av1.x, a0);
    a1 = dp4a_us(w1 & 0x0C0C0C0Cu, av1.y, a1);
    a2 = dp4a_us(w1 & 0x30303030u, av1.z, a2);
    a3 = dp4a_us(w1 & 0xC0C0C0C0u, av1.w, a3);
    return a0 * 64 + (a1 * 16 + (a2 * 4 + a3));
}

// Adds init + 64 * sum over the 32 columns of pos word P / neg word Nn (bit c <-> column c) of
// c * q, c = 1 + p - n in {0, 1, 2}, into four field sums s[0..3].  The two bits of c are p
// (high) and u = not(p or n) (low), so with u formed once the 2-bit values of the even columns
// are ((P << 1) and odd bits) or (u and even bits), those of the odd columns (P and odd bits) or
// ((u >> 1) and even bits): field j of the even word is column 2j, of the odd word column 2j + 1,
// and field r of byte i (column 8i + 2r or 8i + 2r + 1) lines up with activation word 2r (even)
// or 2r + 1 (odd) of the Q1_0 image.  As in q2_block_dot, field r is masked in place (value
// c * 4^r) and dp4a-accumulated into s[r]; with one activation scale per token the sums stay
// apart for a whole row and trit_combine forms (64 s[0] + 16 s[1] + 4 s[2] + s[3]) / 64 once at
// its end.  init carries the offset -64 * sum q of the word (sum c*q - sum q = sum w*q).
__device__ __forceinline__ void trit_word_acc(uint32_t P, uint32_t Nn, const uint4 &a0,
                                              const uint4 &a1, int init, int (&s)[4]) {
    constexpr uint32_t E = 0x55555555u;  // bit 2j of every field
    const uint32_t u = nor_u32(P, Nn);
    const uint32_t fe = select_imm<E>(P << 1, u);
    const uint32_t fo = select_imm<E>(P, u >> 1);
    s[0] = dp4a_us(and_imm<0x03030303u>(fe), a0.x, s[0]);
    s[1] = dp4a_us(and_imm<0x0C0C0C0Cu>(fe), a0.z, s[1]);
    s[2] = dp4a_us(and_imm<0x30303030u>(fe), a1.x, s[2]);
    s[3] = dp4a_us(and_imm<0xC0C0C0C0u>(fe), a1.z, s[3] + init);
    s[0] = dp4a_us(and_imm<0x03030303u>(fo), a0.y, s[0]);
    s[1] = dp4a_us(and_imm<0x0C0C0C0Cu>(fo), a0.w, s[1]);
    s[2] = dp4a_us(and_imm<0x30303030u>(fo), a1.y, s[2]);
    s[3] = dp4a_us(and_imm<0xC0C0C0C0u>(fo), a1.w, s[3]);
}
// (the weighted sum is formed modulo 2^32: the terms may pass 2^31 while the result, 64 times a
// dot product of at most 2^17 columns of |q| <= 128, does not)
__device__ __forceinline__ int trit_combine(const int (&s)[4]) {
    const uint32_t t = (uint32_t)s[0] * 64u + (uint32_t)s[1] * 16u + (uint32_t)s[2] * 4u +
                       (uint32_t)s[3];
    return (int)t >> 6;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ int warp_sum_int(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Matrix that owns row tile u, starting the search at `mi` (a CTA visits tiles in increasing
// order, so the index only moves forward).
__device__ __forceinline__ int find_mat(const StreamParams &p, int u, int mi) {
    while (mi + 1 < p.G && p.m[mi + 1].unit0 <= u) mi++;
    return mi;
}

__device__ __forceinline__ void report(int *err) {
    if (err) atomicOr(err, 1);
}

template <int F, int B, int RW, bool AUX>
__global__ void __launch_bounds__(kStreamThreads, 2)
    stream_gemv_kernel(const __grid_constant__ StreamParams p) {
    constexpr int kCols = FmtInfo<F>::kCols;
    constexpr int kPer = kCols / 32;
    constexpr int TR = kConsumerWarps * RW;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kMaxStages;
    uint8_t *act = smem + kBarBytes;
    uint8_t *stages = act + p.act_bytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KC = p.KC;
    const int KCp = (KC + 7) & ~7;
    const int nq8 = (int)(p.K / 32);

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();
    // Test hook (lb_test_inject_wait_timeout): CTA 0's producer copies nothing, so its
    // consumers' first wait runs out after p.fault microseconds; they report and stop.
    const uint64_t wait_ns = p.fault ? (uint64_t)p.fault * 1000u : kWaitLimitNs;

    if (warp == kConsumerWarps) {
        if (p.fault && blockIdx.x == 0) return;
        // ---------------- producer warp: stream row tiles into the stage ring ----------------
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;
        bool ok = true;
        int mi = 0;
        for (int u = blockIdx.x; u < p.nunits && ok; u += gridDim.x) {
            mi = find_mat(p, u, mi);
            const StreamMat &M = p.m[mi];
            const int row0 = (u - M.unit0) * TR;
            const int rows = min(TR, M.N - row0);
            for (int ct = 0; ct < p.nct; ct++) {
                const int c0 = ct * KC;
                const int kc = min(KC, p.nchunk - c0);
                const int kcp = (kc + 7) & ~7;
                // every lane waits; the outcome is made warp-uniform before anyone acts on it
                if (!__all_sync(0xffffffffu, mbar_wait(&empty[stage], phase ^ 1))) {
                    ok = false;
                    break;
                }
                uint8_t *sb = stages + (size_t)stage * p.stage_bytes;
                if (p.nct == 1) {
                    // Whole rows: the tile is one contiguous range of each plane (scale rows are
                    // padded to S = KCp entries), so two bulk copies move the stage.
                    if (lane == 0) {
                        const uint32_t wb = (uint32_t)rows * kc * 16;
                        const uint32_t sbytes = F != kTrit ? (uint32_t)rows * kcp * 2 : 0u;
                        mbar_arrive_expect_tx(&full[stage], wb + sbytes);
                        bulk_g2s(sb, M.w + (int64_t)row0 * p.nchunk * 16, wb, &full[stage]);
                        if (F != kTrit)
                            bulk_g2s(sb + (size_t)TR * KC * 16, M.scales + (int64_t)row0 * p.S,
                                     sbytes, &full[stage]);
                    }
                } else {
                    // Column slice of long rows: one copy per row and plane.
                    if (lane == 0)
                        mbar_arrive_expect_tx(
                            &full[stage],
                            (uint32_t)(rows * (kc * 16 + (F != kTrit ? kcp * 2 : 0))));
                    __syncwarp();
                    for (int r = lane; r < rows; r += 32) {
                        const int64_t row = row0 + r;
                        bulk_g2s(sb + (size_t)r * KC * 16, M.w + (row * p.nchunk + c0) * 16,
                                 (uint32_t)kc * 16, &full[stage]);
                        if (F != kTrit)
                            bulk_g2s(sb + (size_t)TR * KC * 16 + (size_t)r * KCp * 2,
                                     M.scales + row * p.S + c0, (uint32_t)kcp * 2, &full[stage]);
                    }
                }
                issued++;
                if (++stage == p.stages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        if (!ok && lane == 0) report(p.err);
        // Let every copy this warp issued land before the CTA can retire (bounded).
        for (int i = max(0, issued - p.stages); i < issued; i++)
            mbar_wait(&full[i % p.stages], (uint32_t)((i / p.stages) & 1));
        return;
    }

    // ---------------- consumer warps ----------------
    pdl_wait();
    uint4 *xp = reinterpret_cast<uint4 *>(act);
    float2 *st = reinterpret_cast<float2 *>(act + (size_t)B * p.K);
    stage_activations<F>(p.q, p.d, B, p.K, xp, st, threadIdx.x, kConsumerThreads);
    named_sync(1, kConsumerThreads);

    int stage = 0;
    uint32_t phase = 0;
    int mi = 0;
    const int tok_quads = (int)(p.K / 16);
    for (int u = blockIdx.x; u < p.nunits; u += gridDim.x) {
        mi = find_mat(p, u, mi);
        const StreamMat &M = p.m[mi];
        const int row0 = (u - M.unit0) * TR;
        const int rows = min(TR, M.N - row0);
        typedef typename std::conditional<F == kTrit, int, float>::type Acc;
        Acc acc[RW][B];
        int fs[F == kTrit ? RW : 1][F == kTrit ? B : 1][4];  // planar field sums
#pragma unroll
        for (int rr = 0; rr < RW; rr++)
#pragma unroll
            for (int b = 0; b < B; b++) acc[rr][b] = 0;
        if (F == kTrit) {
#pragma unroll
            for (int rr = 0; rr < (F == kTrit ? RW : 1); rr++)
#pragma unroll
                for (int b = 0; b < (F == kTrit ? B : 1); b++)
#pragma unroll
                    for (int f = 0; f < 4; f++) fs[rr][b][f] = 0;
        }

        for (int ct = 0; ct < p.nct; ct++) {
            const int c0 = ct * KC;
            const int kc = min(KC, p.nchunk - c0);
            if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], phase, wait_ns))) {
                if (lane == 0) report(p.err);
                return;
            }
            const uint8_t *sb = stages + (size_t)stage * p.stage_bytes;
            const uint4 *sw = reinterpret_cast<const uint4 *>(sb) + warp * RW * KC;
            const uint16_t *ss =
                reinterpret_cast<const uint16_t *>(sb + (size_t)TR * KC * 16) + warp * RW * KCp;
            // one chunk of this lane (every lane takes chunks lane, lane + 32, ...)
            auto chunk = [&](const int c) {
                const int cg = c0 + c;  // chunk index within the row
                uint4 wv[RW];
                float dw[RW];
#pragma unroll
                for (int rr = 0; rr < RW; rr++) {
                    wv[rr] = sw[rr * KC + c];
                    dw[rr] = F != kTrit ? f16_bits_to_float(ss[rr * KCp + c]) : 0.0f;
                }
#pragma unroll
                for (int b = 0; b < B; b++) {
                    const uint4 *tok = xp + b * tok_quads;
                    if (F == kTrit) {
                        const float2 *stb = st + b * nq8 + cg * 2;
#pragma unroll
                        for (int h = 0; h < 2; h++) {  // columns 32h .. 32h+31 of the beat
                            const uint4 a0 = tok[quad_slot<F>(cg, 2 * h)];
                            const uint4 a1 = tok[quad_slot<F>(cg, 2 * h + 1)];
                            const int s64 = __float_as_int(stb[h].y);  // -64 * sum q
#pragma unroll
                            for (int rr = 0; rr < RW; rr++) {
                                const uint32_t pw = h ? wv[rr].y : wv[rr].x;
                                const uint32_t nw = h ? wv[rr].w : wv[rr].z;
                                // select-accumulate: + where pos, - where neg (x64, exact)
                                trit_word_acc(pw, nw, a0, a1, s64,
                                              fs[F == kTrit ? rr : 0][F == kTrit ? b : 0]);
                            }
                        }
                    } else {
                        const float2 *stb = st + b * nq8 + cg * kPer;
                        float t[RW];
#pragma unroll
                        for (int rr = 0; rr < RW; rr++) t[rr] = 0.0f;
#pragma unroll
                        for (int j = 0; j < kPer; j++) {
                            const float2 ds = stb[j];  // {d / 64, -64 * sum q}
                            const int s64 = __float_as_int(ds.y);
                            int a[RW];  // 64 * isum
                            if (F == kQ1) {
                                const uint4 a0 = tok[quad_slot<F>(cg, 2 * j)];
                                const uint4 a1 = tok[quad_slot<F>(cg, 2 * j + 1)];
#pragma unroll
                                for (int rr = 0; rr < RW; rr++)  // 128 sum b q - 64 sum q
                                    a[rr] = q1_word_dot(word_of(wv[rr], j), a0, a1, s64);
                            } else {
                                const uint4 av0 = tok[quad_slot<F>(cg, 2 * j)];
                                const uint4 av1 = tok[quad_slot<F>(cg, 2 * j + 1)];
#pragma unroll
                                for (int rr = 0; rr < RW; rr++)  // 64 sum c q - 64 sum q
                                    a[rr] = q2_block_dot(word_of(wv[rr], 2 * j),
                                                         word_of(wv[rr], 2 * j + 1), av0, av1,
                                                         s64);
                            }
#pragma unroll
                            for (int rr = 0; rr < RW; rr++) {
                                const int r = warp * RW + rr;
                                if (AUX && M.aux && r < rows)
                                    M.aux[((int64_t)b * M.N + row0 + r) * nq8 + cg * kPer + j] =
                                        a[rr] >> 6;
                                t[rr] = fmaf(ds.x, (float)a[rr], t[rr]);
                            }
                        }
#pragma unroll
                        for (int rr = 0; rr < RW; rr++)
                            acc[rr][b] = fmaf(dw[rr], t[rr], acc[rr][b]);
                    }
                }
            };
            if ((B == 1 && !AUX) && kc % 64 == 0) {
                // every lane has the same even number of chunks: two per pass, so that
                // the loads of one overlap the arithmetic of the other (at one token only;
                // more tokens would spill registers)
#pragma unroll 2
                for (int c = lane; c < kc; c += 32) chunk(c);
            } else {
                for (int c = lane; c < kc; c += 32) chunk(c);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == p.stages) {
                stage = 0;
                phase ^= 1;
            }
        }
        // finish the rows of this tile: the RW x B sums over the warp, one lane per result
        constexpr int V = RW * B;
        constexpr int kSpan = 32 / PowTwo<V>::value;  // lanes per result after the reduction
        Acc part[V];
#pragma unroll
        for (int rr = 0; rr < RW; rr++)
#pragma unroll
            for (int b = 0; b < B; b++)
                part[rr * B + b] =
                    F == kTrit ? (Acc)trit_combine(fs[F == kTrit ? rr : 0][F == kTrit ? b : 0])
                               : acc[rr][b];
        const Acc tot = warp_sum_many<V>(part, lane);
        const int vi = lane / kSpan;
        const int r = warp * RW + vi / B, b = vi % B;
        if (lane % kSpan == 0 && vi < V && r < rows) {
            const int64_t o = (int64_t)b * M.N + row0 + r;
            if (F == kTrit) {
                const int a = (int)tot;
                const float t = __fmul_rn((float)a, p.x_scale[b]);
                M.y[o] = __fmul_rn(t, M.w_scale);
                if (M.aux) M.aux[o] = a;
            } else {
                M.y[o] = (float)tot;
            }
        }
    }
}

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------
struct StreamPlan {
    int RW, KC, nct, stages, stage_bytes, act_bytes, smem;
};

// Tile geometry for a format and activation: rows per warp RW (largest power of two up to
// max_rw whose tile fits the stage budget), column slice KC (chunks; the whole row unless the
// row is too long, then a multiple of 8), and the stage count (at most four, at least two,
// aiming at two CTAs per SM).
inline StreamPlan plan_stream(int F, int B, int64_t K, int max_rw) {
    const int cols = F == kQ1 ? 128 : 64;
    const int nchunk = (int)(K / cols);
    const int scale_b = F == kTrit ? 0 : 2;
    const int budget = 40 * 1024;
    StreamPlan pl{};
    pl.act_bytes = (int)(((int64_t)B * K + (int64_t)B * (K / 32) * 8 + 127) / 128 * 128);
    int KC = nchunk;
    auto row_cost = [&](int kc) { return kc * 16 + ((kc + 7) & ~7) * scale_b; };
    int RW = 1;
    for (int rw = max_rw; rw >= 1; rw /= 2) {
        if (8 * rw * row_cost(KC) <= budget) {
            RW = rw;
            break;
        }
    }
    if (8 * RW * row_cost(KC) > budget) {  // very long rows: slice columns
        KC = budget / (8 * (16 + scale_b)) / 8 * 8;
        RW = 1;
    }
    pl.RW = RW;
    pl.KC = KC;
    pl.nct = (nchunk + KC - 1) / KC;
    const int TR = 8 * RW;
    pl.stage_bytes = (TR * KC * 16 + TR * ((KC + 7) & ~7) * scale_b + 127) / 128 * 128;
    const int per_cta = 113 * 1024;
    int stages = kMaxStages;
    while (stages > 2 && kBarBytes + pl.act_bytes + stages * pl.stage_bytes > per_cta) stages--;
    pl.stages = stages;
    pl.smem = kBarBytes + pl.act_bytes + stages * pl.stage_bytes;
    return pl;
}

template <int F, int B, int RW, bool AUX>
inline int launch_stream_cfg(StreamParams &p, const StreamPlan &pl, int sms, cudaStream_t st) {
    auto kern = stream_gemv_kernel<F, B, RW, AUX>;
    if (pl.RW != RW) return LB_ERR_LAUNCH;  // the tile geometry must match the kernel
    int bps = 0;
    if (int e = prepare_kernel(reinterpret_cast<const void *>(kern), kStreamThreads,
                               (size_t)pl.smem, &bps))
        return e;
    const int TR = 8 * RW;
    int units = 0;
    for (int i = 0; i < p.G; i++) {
        p.m[i].unit0 = units;
        units += (p.m[i].N + TR - 1) / TR;
    }
    p.nunits = units;
    p.nct = pl.nct;
    p.KC = pl.KC;
    p.stages = pl.stages;
    p.stage_bytes = pl.stage_bytes;
    p.act_bytes = pl.act_bytes;
    int64_t grid = (int64_t)sms * bps;
    if (grid > units) grid = units;
    if (grid < 1) grid = 1;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(kStreamThreads), (size_t)pl.smem, st, p);
}

// ------------------------------------------------------------------------------------------
// Batched variant (B >= 3): lane = weight row.
//
// At larger batch the activation reads, not the weights, bound the kernel above: every lane
// reads the activation words of its own chunk, once per token and row.  Here a warp takes 32
// rows, one per lane, and a contiguous range of the row's chunks, so for any chunk all 32 lanes
// read the same activation words -- shared-memory broadcasts -- and each weight chunk is read
// once.  A unit is 32 rows; the eight consumer warps split its chunks and add their partial sums
// through shared memory at the end of the unit.  Rows are staged one bulk copy per row (one per
// producer lane) with a 16-byte pad, so the lanes' 16-byte weight reads do not conflict.
// Calls with few rows use RG = 2 or 4 row groups per warp: a unit is then 32 / RG rows, lane
// (row r, group g) takes every RG-th chunk of the warp's range starting at g, and the groups'
// partial sums meet by warp shuffles -- RG times as many units, so small matrices fill the GPU.
// The RG groups read RG consecutive chunks of the activation image at once (distinct banks).
// ------------------------------------------------------------------------------------------
constexpr int kRowsPerUnit = 32;

template <int F, int B, int RG>
__global__ void __launch_bounds__(kStreamThreads, 2)
    stream_rows_kernel(const __grid_constant__ StreamParams p) {
    constexpr int kCols = FmtInfo<F>::kCols;
    constexpr int kPer = kCols / 32;
    constexpr int TR = kRowsPerUnit / RG;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kMaxStages;
    uint8_t *act = smem + kBarBytes;
    uint8_t *stages = act + p.act_bytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KC = p.KC;                  // chunks per stage (a multiple of 8, or the whole row)
    const int KCp = (KC + 7) & ~7;
    const int wpitch = (KC + 1) * 16;     // padded row pitch of the weight slice
    const int spitch = KCp * 2;           // row pitch of the scale slice
    const int nq8 = (int)(p.K / 32);
    float *red = reinterpret_cast<float *>(stages + (size_t)p.stages * p.stage_bytes);

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();
    // Test hook, as in stream_gemv_kernel.
    const uint64_t wait_ns = p.fault ? (uint64_t)p.fault * 1000u : kWaitLimitNs;

    if (warp == kConsumerWarps) {
        if (p.fault && blockIdx.x == 0) return;
        // ---------------- producer warp: lane r copies row r of every stage ----------------
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;
        bool ok = true;
        int mi = 0;
        for (int u = blockIdx.x; u < p.nunits && ok; u += gridDim.x) {
            mi = find_mat(p, u, mi);
            const StreamMat &M = p.m[mi];
            const int row0 = (u - M.unit0) * TR;
            const int rows = min(TR, M.N - row0);
            for (int ct = 0; ct < p.nct; ct++) {
                const int c0 = ct * KC;
                const int kc = min(KC, p.nchunk - c0);
                const int kcp = (kc + 7) & ~7;
                if (!__all_sync(0xffffffffu, mbar_wait(&empty[stage], phase ^ 1))) {
                    ok = false;
                    break;
                }
                uint8_t *sb = stages + (size_t)stage * p.stage_bytes;
                if (lane == 0)
                    mbar_arrive_expect_tx(
                        &full[stage], (uint32_t)(rows * (kc * 16 + (F != kTrit ? kcp * 2 : 0))));
                __syncwarp();
                if (lane < rows) {
                    const int64_t row = row0 + lane;
                    bulk_g2s(sb + (size_t)lane * wpitch, M.w + (row * p.nchunk + c0) * 16,
                             (uint32_t)kc * 16, &full[stage]);
                    if (F != kTrit)
                        bulk_g2s(sb + (size_t)TR * wpitch + (size_t)lane * spitch,
                                 M.scales + row * p.S + c0, (uint32_t)kcp * 2, &full[stage]);
                }
                issued++;
                if (++stage == p.stages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        if (!ok && lane == 0) report(p.err);
        for (int i = max(0, issued - p.stages); i < issued; i++)
            mbar_wait(&full[i % p.stages], (uint32_t)((i / p.stages) & 1));
        return;
    }

    // ---------------- consumer warps ----------------
    pdl_wait();
    uint4 *xp = reinterpret_cast<uint4 *>(act);
    float2 *st = reinterpret_cast<float2 *>(act + (size_t)B * p.K);
    stage_activations<F>(p.q, p.d, B, p.K, xp, st, threadIdx.x, kConsumerThreads);
    named_sync(1, kConsumerThreads);

    int stage = 0;
    uint32_t phase = 0;
    int mi = 0;
    const int tok_quads = (int)(p.K / 16);
    for (int u = blockIdx.x; u < p.nunits; u += gridDim.x) {
        mi = find_mat(p, u, mi);
        const StreamMat &M = p.m[mi];
        const int row0 = (u - M.unit0) * TR;
        const int rows = min(TR, M.N - row0);
        typedef typename std::conditional<F == kTrit, int, float>::type Acc;
        Acc acc[B];
        int fs[F == kTrit ? B : 1][4];  // planar field sums
#pragma unroll
        for (int b = 0; b < B; b++) acc[b] = 0;
        if (F == kTrit) {
#pragma unroll
            for (int b = 0; b < (F == kTrit ? B : 1); b++)
#pragma unroll
                for (int f = 0; f < 4; f++) fs[b][f] = 0;
        }

        for (int ct = 0; ct < p.nct; ct++) {
            const int c0 = ct * KC;
            const int kc = min(KC, p.nchunk - c0);
            if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], phase, wait_ns))) {
                if (lane == 0) report(p.err);
                return;
            }
            const uint8_t *sb = stages + (size_t)stage * p.stage_bytes;
            const int lr = lane % TR, lg = lane / TR;  // row of the unit, chunk group
            const uint8_t *wrow = sb + (size_t)lr * wpitch;
            const uint16_t *srow =
                reinterpret_cast<const uint16_t *>(sb + (size_t)TR * wpitch + (size_t)lr * spitch);
            // this warp's chunks of the stage: a contiguous eighth (rounded up)
            const int per = (kc + kConsumerWarps - 1) / kConsumerWarps;
            const int cb = warp * per, ce = min(kc, cb + per);
            for (int c = cb + lg; c < ce; c += RG) {
                const int cg = c0 + c;
                const uint4 wv = *reinterpret_cast<const uint4 *>(wrow + (size_t)c * 16);
                const float dw = F != kTrit ? f16_bits_to_float(srow[c]) : 0.0f;
#pragma unroll
                for (int b = 0; b < B; b++) {
                    const uint4 *tok = xp + b * tok_quads;
                    if (F == kTrit) {
                        const float2 *stb = st + b * nq8 + cg * 2;
#pragma unroll
                        for (int h = 0; h < 2; h++) {
                            const uint4 a0 = tok[quad_slot<F>(cg, 2 * h)];
                            const uint4 a1 = tok[quad_slot<F>(cg, 2 * h + 1)];
                            const int s64 = __float_as_int(stb[h].y);  // -64 * sum q
                            trit_word_acc(h ? wv.y : wv.x, h ? wv.w : wv.z, a0, a1, s64,
                                          fs[F == kTrit ? b : 0]);
                        }
                    } else {
                        const float2 *stb = st + b * nq8 + cg * kPer;
                        float t = 0.0f;
#pragma unroll
                        for (int j = 0; j < kPer; j++) {
                            const float2 ds = stb[j];  // {d / 64, -64 * sum q}
                            const int s64 = __float_as_int(ds.y);
                            const uint4 av0 = tok[quad_slot<F>(cg, 2 * j)];
                            const uint4 av1 = tok[quad_slot<F>(cg, 2 * j + 1)];
                            const int a = F == kQ1
                                              ? q1_word_dot(word_of(wv, j), av0, av1, s64)
                                              : q2_block_dot(word_of(wv, 2 * j),
                                                             word_of(wv, 2 * j + 1), av0, av1,
                                                             s64);
                            t = fmaf(ds.x, (float)a, t);
                        }
                        acc[b] = fmaf(dw, t, acc[b]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == p.stages) {
                stage = 0;
                phase ^= 1;
            }
        }
        if (F == kTrit) {
#pragma unroll
            for (int b = 0; b < B; b++) acc[b] = (Acc)trit_combine(fs[F == kTrit ? b : 0]);
        }
        // add the row groups' partial sums (shuffles), then the eight warps' (shared memory)
#pragma unroll
        for (int o = TR; o < 32; o <<= 1)
#pragma unroll
            for (int b = 0; b < B; b++) acc[b] += __shfl_xor_sync(0xffffffffu, acc[b], o);
        if (lane < TR) {
#pragma unroll
            for (int b = 0; b < B; b++)
                red[(warp * B + b) * TR + lane] = F == kTrit ? __int_as_float((int)acc[b])
                                                             : (float)acc[b];
        }
        named_sync(1, kConsumerThreads);
        for (int i = threadIdx.x; i < B * TR; i += kConsumerThreads) {
            const int b = i / TR, r = i % TR;
            if (r < rows) {
                const int64_t o = (int64_t)b * M.N + row0 + r;
                if (F == kTrit) {
                    int a = 0;
#pragma unroll
                    for (int w = 0; w < kConsumerWarps; w++)
                        a += __float_as_int(red[(w * B + b) * TR + r]);
                    const float t = __fmul_rn((float)a, p.x_scale[b]);
                    M.y[o] = __fmul_rn(t, M.w_scale);
                    if (M.aux) M.aux[o] = a;
                } else {
                    float v = 0.0f;
#pragma unroll
                    for (int w = 0; w < kConsumerWarps; w++) v += red[(w * B + b) * TR + r];
                    M.y[o] = v;
                }
            }
        }
        named_sync(1, kConsumerThreads);
    }
}

// Geometry of the batched variant for units of `tr` rows: chunks per stage (whole row, or a
// multiple of 8 within a 40 KB stage), stage count for two CTAs per SM where possible.
inline StreamPlan plan_rows(int F, int B, int64_t K, int tr) {
    const int cols = F == kQ1 ? 128 : 64;
    const int nchunk = (int)(K / cols);
    const int scale_b = F == kTrit ? 0 : 2;
    StreamPlan pl{};
    pl.act_bytes = (int)(((int64_t)B * K + (int64_t)B * (K / 32) * 8 + 127) / 128 * 128);
    auto stage_cost = [&](int kc) { return tr * ((kc + 1) * 16 + ((kc + 7) & ~7) * scale_b); };
    const int red_b = kConsumerWarps * B * tr * 4;
    // Stage budget: two stages next to the activation image should still let two CTAs share
    // an SM (up to 40 KB per stage, at least 8 KB).
    int budget = (113 * 1024 - kBarBytes - pl.act_bytes - red_b) / 2;
    if (budget < 8 * 1024) budget = 40 * 1024;  // one CTA per SM anyway: large stages
    if (budget > 40 * 1024) budget = 40 * 1024;
    int KC = nchunk;
    if (stage_cost(KC) > budget) KC = (budget / tr - 16) / (16 + scale_b) / 8 * 8;
    pl.RW = 0;
    pl.KC = KC;
    pl.nct = (nchunk + KC - 1) / KC;
    pl.stage_bytes = (stage_cost(KC) + 127) / 128 * 128;
    const int per_cta = 113 * 1024;
    int stages = kMaxStages;
    while (stages > 2 && kBarBytes + pl.act_bytes + stages * pl.stage_bytes + red_b > per_cta)
        stages--;
    pl.stages = stages;
    pl.smem = kBarBytes + pl.act_bytes + stages * pl.stage_bytes + red_b;
    return pl;
}

template <int F, int B, int RG>
inline int launch_rows_cfg(StreamParams &p, int sms, cudaStream_t st) {
    constexpr int TR = kRowsPerUnit / RG;
    const StreamPlan pl = plan_rows(F, B, p.K, TR);
    auto kern = stream_rows_kernel<F, B, RG>;
    int bps = 0;
    if (int e = prepare_kernel(reinterpret_cast<const void *>(kern), kStreamThreads,
                               (size_t)pl.smem, &bps))
        return e;
    int units = 0;
    for (int i = 0; i < p.G; i++) {
        p.m[i].unit0 = units;
        units += (p.m[i].N + TR - 1) / TR;
    }
    p.nunits = units;
    p.nct = pl.nct;
    p.KC = pl.KC;
    p.stages = pl.stages;
    p.stage_bytes = pl.stage_bytes;
    p.act_bytes = pl.act_bytes;
    int64_t grid = (int64_t)sms * bps;
    if (grid > units) grid = units;
    if (grid < 1) grid = 1;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(kStreamThreads), (size_t)pl.smem, st, p);
}

// Row groups per warp: as many (1, 2 or 4) as keep the call's units within two CTAs per SM,
// with an eighth of slack (measured, 8 tokens, 2560 x 6912 planar: 320 units of 8 rows on 304
// CTA slots 10.8 us, 160 units of 16 rows 12.2 us, 80 units of 32 rows 17.2 us).
template <int F, int B>
inline int launch_rows(StreamParams &p, int sms, cudaStream_t st) {
    int64_t units32 = 0;
    for (int i = 0; i < p.G; i++) units32 += (p.m[i].N + kRowsPerUnit - 1) / kRowsPerUnit;
    const int64_t slots = 2 * (int64_t)sms;
    if (4 * units32 <= slots + slots / 8) return launch_rows_cfg<F, B, 4>(p, sms, st);
    if (2 * units32 <= slots) return launch_rows_cfg<F, B, 2>(p, sms, st);
    return launch_rows_cfg<F, B, 1>(p, sms, st);
}

template <int F, int B>
inline int launch_stream(StreamParams &p, bool aux, int sms, cudaStream_t st) {
    if (aux) return launch_stream_cfg<F, B, 1, true>(p, plan_stream(F, B, p.K, 1), sms, st);
    if constexpr (B > 2) {
        return launch_rows<F, B>(p, sms, st);
    } else {
        // Q1_0 rows are short (a chunk is 128 weights): eight rows per warp cut the fixed cost
        // per row (stage hand-off, reduction, activation loads) at one token; a 64-row tile
        // then costs about 7/4 of a 32-row one.  Taken where that wins over whole waves of
        // tiles on the CTA slots (two per SM).
        int max_rw = 4;
        if (F == kQ1 && B == 1) {
            int64_t t8 = 0, t4 = 0;
            for (int i = 0; i < p.G; i++) {
                t8 += (p.m[i].N + 63) / 64;
                t4 += (p.m[i].N + 31) / 32;
            }
            const int64_t slots = 2 * (int64_t)sms;
            if ((t8 + slots - 1) / slots * 7 < (t4 + slots - 1) / slots * 4) max_rw = 8;
        }
        const StreamPlan pl = plan_stream(F, B, p.K, max_rw);
        if constexpr (F == kQ1 && B == 1) {
            if (pl.RW == 8) return launch_stream_cfg<F, B, 8, false>(p, pl, sms, st);
        }
        if (pl.RW == 4) return launch_stream_cfg<F, B, 4, false>(p, pl, sms, st);
        if (pl.RW == 2) return launch_stream_cfg<F, B, 2, false>(p, pl, sms, st);
        return launch_stream_cfg<F, B, 1, false>(p, pl, sms, st);
    }
}

template <int F, int B>
inline int launch_tc_gemv(StreamParams &p, int sms, cudaStream_t st);

// Fewest 128-row units for which the tensor-core variant beats the lane-per-row kernel: one of
// its CTAs walks a unit's K in dependent steps of ~0.6 us, so a call with few units is latency-
// bound there (measured at 8 tokens: 32 units 16.7 us vs 9.3 us lane-per-row, 108 units 11.7 vs
// 15.4 us, 128 units 1107 vs 1058 GB/s).
constexpr int64_t kTcMinUnits = 64;

template <int F>
inline int dispatch_stream(StreamParams &p, int B, bool aux, int sms, cudaStream_t st) {
    p.fault = 0;
    // Five or more tokens (four for Q2_0_g64): the tensor-core variant (lb_tcgemv.cuh) when K
    // is a multiple of its 256-column step, its activation operand (16 K bytes) fits in shared
    // memory and the call has at least kTcMinUnits row units; the block-sum hook stays on the
    // streaming kernels.  Below that the lane-per-row kernel is faster (64 x 4096^2 at 3 tokens:
    // Q2_0 2373 vs 2134 GB/s, Q1_0 1416 vs 1169, planar 2842 vs 1820; at 4 tokens Q1_0 1289 vs
    // 1141, planar 2379 vs 1886, Q2_0 2075 vs 2118).
    int64_t tc_units = 0;
    for (int i = 0; i < p.G; i++) tc_units += (p.m[i].N + 127) / 128;
    const int tc_min_tokens = F == kQ2 ? 4 : 5;
    if (B >= tc_min_tokens && !aux && p.K % 256 == 0 && p.K <= 4096 &&
        tc_units >= kTcMinUnits) {
        switch (B) {
            case 4: return launch_tc_gemv<F, 4>(p, sms, st);
            case 5: return launch_tc_gemv<F, 5>(p, sms, st);
            case 6: return launch_tc_gemv<F, 6>(p, sms, st);
            case 7: return launch_tc_gemv<F, 7>(p, sms, st);
            case 8: return launch_tc_gemv<F, 8>(p, sms, st);
        }
    }
    p.fault = take_injected_wait_fault();  // only the streaming kernels honor the test hook
    switch (B) {
        case 1: return launch_stream<F, 1>(p, aux, sms, st);
        case 2: return launch_stream<F, 2>(p, aux, sms, st);
        case 3: return launch_stream<F, 3>(p, aux, sms, st);
        case 4: return launch_stream<F, 4>(p, aux, sms, st);
        case 5: return launch_stream<F, 5>(p, aux, sms, st);
        case 6: return launch_stream<F, 6>(p, aux, sms, st);
        case 7: return launch_stream<F, 7>(p, aux, sms, st);
        case 8: return launch_stream<F, 8>(p, aux, sms, st);
    }
    return LB_ERR_BATCH;
}

inline int64_t scale_stride(int64_t K, int qk) { return (K / qk + 7) / 8 * 8; }

}  // namespace lb

#include "lb_tcgemv.cuh"
