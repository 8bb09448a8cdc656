// lb_gemv.cu -- decode GEMVs for Q1_0, Q2_0_g64 and the planar ternary layout (batch 1..8).
//
// Arithmetic (integer block sums, then float scales):
//   Q1_0     -- "bankml: verified low-bit inference on commodity CPUs -- a technical report",
//               III.2 (128 sign bits + fp16 scale, signed sum, q8_0 activations) and III.3
//               (integer sum per q8_0 block, then one multiply-add per q8_0 block and per
//               weight block).
//   Q2_0_g64 -- same report, III.5 (64 two-bit codes, code c means c - 1) and III.8 (offset
//               code: sum w*x = sum c*x - sum x).
//   planar   -- tritium.technology "Architecture", sections 1-2 (select-accumulate over
//               {pos, neg} bit planes), 4.1 (int32 accumulator, exact for x = -128) and 5
//               (w_scale and x_scale applied as two separate multiplies).
//
// GPU design (the pages' kernels are CPU/RTL prior art; this is not a translation):
//   * Weights are streamed once from HBM with 128-bit loads that bypass L1 (each lane owns one
//     16-byte chunk per row: a Q1_0 block, a Q2_0_g64 block or one planar beat), so one warp
//     request covers 512 contiguous bytes of a row.
//   * The activations of all B tokens are staged once per CTA in shared memory, already
//     re-laid-out so that a shift and a mask of a weight word lines up with one activation word
//     (the weights are never shuffled; bankml's report permutes the activation for the same
//     reason). The shared image is XOR-swizzled per chunk so the lanes' 16-byte reads are
//     bank-conflict free.
//   * Sign bits and codes are expanded in registers to bytes and consumed by dp4a; integer sums
//     per q8_0 block are exact, so any lane order gives the same block sums.
//   * Each warp keeps R rows in flight; partial row sums are combined with warp shuffles.
//     No atomics: results are deterministic run to run.
#include "lb_common.cuh"

namespace lb {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

enum Fmt { kQ1 = 0, kQ2 = 1, kTrit = 2 };

// Bytes of activations consumed by one 16-byte weight chunk, and 16-byte quads per chunk.
template <int F> struct FmtInfo;
template <> struct FmtInfo<kQ1> { static constexpr int kCols = 128; static constexpr int kQuads = 8; };
template <> struct FmtInfo<kQ2> { static constexpr int kCols = 64; static constexpr int kQuads = 4; };
template <> struct FmtInfo<kTrit> { static constexpr int kCols = 64; static constexpr int kQuads = 4; };

// Physical 16-byte slot of logical quad u of chunk c (conflict-free for 8 consecutive chunks).
template <int F>
__device__ __forceinline__ int64_t quad_slot(int64_t c, int u) {
    if (FmtInfo<F>::kQuads == 8) return c * 8 + (u ^ (int)(c & 7));
    return c * 4 + (u ^ (int)((c >> 1) & 3));
}

// ------------------------------------------------------------------------------------------
// Activation staging.  One thread per 32-value group (one q8_0 block, or half a planar beat).
//   Q2_0_g64 image : for each 16 activations x[16t .. 16t+15] the words
//                    A[t][r] = (x[16t+r], x[16t+4+r], x[16t+8+r], x[16t+12+r]), r = 0..3,
//                    which line up with ((code word t) >> 2r) & 0x03030303.
//   Q1_0 / planar  : for each 32 activations x[32t .. 32t+31] the words
//                    A[t][k] = (x[32t+k], x[32t+8+k], x[32t+16+k], x[32t+24+k]), k = 0..7,
//                    which line up with ((sign word t) >> k) & 0x01010101.
//   dxf / sq       : q8_0 scale widened to fp32 and the sum of the 32 codes of each block.
// ------------------------------------------------------------------------------------------
template <int F>
__device__ void stage_activations(const int8_t *__restrict__ q, const uint16_t *__restrict__ d,
                                  int B, int64_t K, uint4 *__restrict__ xp,
                                  float *__restrict__ dxf, int *__restrict__ sq) {
    const int64_t ngroups = (int64_t)B * K / 32;
    const int64_t per_token = K / 32;
    for (int64_t i = threadIdx.x; i < ngroups; i += blockDim.x) {
        const uint4 *src = reinterpret_cast<const uint4 *>(q) + 2 * i;
        uint4 lo = src[0], hi = src[1];
        const int64_t b = i / per_token, j = i % per_token;
        uint4 o0, o1;
        if (F == kQ2) {
            transpose4x4(lo.x, lo.y, lo.z, lo.w, o0.x, o0.y, o0.z, o0.w);
            transpose4x4(hi.x, hi.y, hi.z, hi.w, o1.x, o1.y, o1.z, o1.w);
        } else {
            transpose4x4(lo.x, lo.z, hi.x, hi.z, o0.x, o0.y, o0.z, o0.w);  // k = 0..3
            transpose4x4(lo.y, lo.w, hi.y, hi.w, o1.x, o1.y, o1.z, o1.w);  // k = 4..7
        }
        const int64_t c = j * 32 / FmtInfo<F>::kCols;              // chunk within the token
        const int u0 = (int)((j * 32) % FmtInfo<F>::kCols) / 16;   // first quad of the group
        uint4 *tok = xp + b * (K / 16);
        tok[quad_slot<F>(c, u0)] = o0;
        tok[quad_slot<F>(c, u0 + 1)] = o1;
        if (F != kTrit) {
            int s = byte_sum_s8(lo.x) + byte_sum_s8(lo.y) + byte_sum_s8(lo.z) + byte_sum_s8(lo.w) +
                    byte_sum_s8(hi.x) + byte_sum_s8(hi.y) + byte_sum_s8(hi.z) + byte_sum_s8(hi.w);
            sq[i] = s;
            dxf[i] = f16_bits_to_float(d[i]);
        }
    }
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int t) {
    return t == 0 ? v.x : (t == 1 ? v.y : (t == 2 ? v.z : v.w));
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

// ------------------------------------------------------------------------------------------
// Q1_0 / Q2_0_g64 GEMV
// ------------------------------------------------------------------------------------------
template <int F, int B, int R, bool ISUM>
__global__ void __launch_bounds__(kThreads)
    gemv_q_kernel(const uint8_t *__restrict__ bits, const uint16_t *__restrict__ scales,
                  const int8_t *__restrict__ q, const uint16_t *__restrict__ d,
                  float *__restrict__ y, int32_t *__restrict__ isum, int64_t N, int64_t K) {
    constexpr int kCols = FmtInfo<F>::kCols;
    constexpr int kPer = kCols / 32;  // q8_0 blocks per weight block
    extern __shared__ uint4 smem[];
    const int64_t nq8 = K / 32;
    uint4 *xp = smem;
    float *dxf = reinterpret_cast<float *>(xp + (int64_t)B * K / 16);
    int *sq = reinterpret_cast<int *>(dxf + (int64_t)B * nq8);
    stage_activations<F>(q, d, B, K, xp, dxf, sq);
    __syncthreads();

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t nchunk = K / kCols;
    const int64_t ngroups = (N + R - 1) / R;
    for (int64_t g = (int64_t)blockIdx.x * kWarps + warp; g < ngroups;
         g += (int64_t)gridDim.x * kWarps) {
        const int64_t r0 = g * R;
        float acc[R][B];
#pragma unroll
        for (int rr = 0; rr < R; rr++)
#pragma unroll
            for (int b = 0; b < B; b++) acc[rr][b] = 0.0f;

        for (int64_t c = lane; c < nchunk; c += 32) {
            uint4 wv[R];
            float dw[R];
#pragma unroll
            for (int rr = 0; rr < R; rr++) {
                const int64_t row = r0 + rr;
                if (row < N) {
                    wv[rr] = ldg_stream(bits + (row * nchunk + c) * 16);
                    dw[rr] = f16_bits_to_float(scales[row * nchunk + c]);
                } else {
                    wv[rr] = make_uint4(0, 0, 0, 0);
                    dw[rr] = 0.0f;
                }
            }
#pragma unroll
            for (int b = 0; b < B; b++) {
                const uint4 *tok = xp + (int64_t)b * (K / 16);
                const float *dxb = dxf + b * nq8 + c * kPer;
                const int *sqb = sq + b * nq8 + c * kPer;
                float t[R];
#pragma unroll
                for (int rr = 0; rr < R; rr++) t[rr] = 0.0f;
#pragma unroll
                for (int j = 0; j < kPer; j++) {  // q8_0 block j of this weight block
                    const float dx = dxb[j];
                    const int s = sqb[j];
                    int a[R];
#pragma unroll
                    for (int rr = 0; rr < R; rr++) a[rr] = 0;
                    if (F == kQ1) {
                        // word j of the chunk holds the 32 sign bits of q8_0 block j
                        const uint4 a0 = tok[quad_slot<F>(c, 2 * j)];
                        const uint4 a1 = tok[quad_slot<F>(c, 2 * j + 1)];
#pragma unroll
                        for (int rr = 0; rr < R; rr++) {
                            const uint32_t w = word_of(wv[rr], j);
                            int v = 0;
                            v = dp4a_us(w & 0x01010101u, a0.x, v);
                            v = dp4a_us((w >> 1) & 0x01010101u, a0.y, v);
                            v = dp4a_us((w >> 2) & 0x01010101u, a0.z, v);
                            v = dp4a_us((w >> 3) & 0x01010101u, a0.w, v);
                            v = dp4a_us((w >> 4) & 0x01010101u, a1.x, v);
                            v = dp4a_us((w >> 5) & 0x01010101u, a1.y, v);
                            v = dp4a_us((w >> 6) & 0x01010101u, a1.z, v);
                            v = dp4a_us((w >> 7) & 0x01010101u, a1.w, v);
                            a[rr] = 2 * v - s;  // sum s_i q_i = 2 sum b_i q_i - sum q_i
                        }
                    } else {
                        // words 2j, 2j+1 of the chunk hold the 32 codes of q8_0 block j
#pragma unroll
                        for (int h = 0; h < 2; h++) {
                            const uint4 av = tok[quad_slot<F>(c, 2 * j + h)];
#pragma unroll
                            for (int rr = 0; rr < R; rr++) {
                                const uint32_t w = word_of(wv[rr], 2 * j + h);
                                int v = a[rr];
                                v = dp4a_us(w & 0x03030303u, av.x, v);
                                v = dp4a_us((w >> 2) & 0x03030303u, av.y, v);
                                v = dp4a_us((w >> 4) & 0x03030303u, av.z, v);
                                v = dp4a_us((w >> 6) & 0x03030303u, av.w, v);
                                a[rr] = v;
                            }
                        }
#pragma unroll
                        for (int rr = 0; rr < R; rr++) a[rr] -= s;  // offset code: - sum q
                    }
#pragma unroll
                    for (int rr = 0; rr < R; rr++) {
                        if (ISUM && r0 + rr < N)
                            isum[((int64_t)b * N + r0 + rr) * nq8 + c * kPer + j] = a[rr];
                        t[rr] = fmaf(dx, (float)a[rr], t[rr]);
                    }
                }
#pragma unroll
                for (int rr = 0; rr < R; rr++) acc[rr][b] = fmaf(dw[rr], t[rr], acc[rr][b]);
            }
        }
#pragma unroll
        for (int rr = 0; rr < R; rr++)
#pragma unroll
            for (int b = 0; b < B; b++) {
                const float v = warp_sum(acc[rr][b]);
                if (lane == 0 && r0 + rr < N) y[(int64_t)b * N + r0 + rr] = v;
            }
    }
}

// ------------------------------------------------------------------------------------------
// planar ternary GEMV
// ------------------------------------------------------------------------------------------
template <int B, int R>
__global__ void __launch_bounds__(kThreads)
    gemv_trit_kernel(const uint64_t *__restrict__ planes, float w_scale,
                     const int8_t *__restrict__ q, const float *__restrict__ x_scale,
                     float *__restrict__ y, int32_t *__restrict__ acc_out, int64_t N,
                     int64_t K) {
    extern __shared__ uint4 smem[];
    uint4 *xp = smem;
    stage_activations<kTrit>(q, nullptr, B, K, xp, nullptr, nullptr);
    __syncthreads();

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t nbeat = K / 64;
    const int64_t ngroups = (N + R - 1) / R;
    for (int64_t g = (int64_t)blockIdx.x * kWarps + warp; g < ngroups;
         g += (int64_t)gridDim.x * kWarps) {
        const int64_t r0 = g * R;
        int acc[R][B];
#pragma unroll
        for (int rr = 0; rr < R; rr++)
#pragma unroll
            for (int b = 0; b < B; b++) acc[rr][b] = 0;
        for (int64_t c = lane; c < nbeat; c += 32) {
            uint4 wv[R];  // {pos lo, pos hi, neg lo, neg hi}
#pragma unroll
            for (int rr = 0; rr < R; rr++) {
                const int64_t row = r0 + rr;
                wv[rr] = row < N ? ldg_stream(planes + (row * nbeat + c) * 2)
                                 : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int b = 0; b < B; b++) {
                const uint4 *tok = xp + (int64_t)b * (K / 16);
#pragma unroll
                for (int h = 0; h < 2; h++) {  // columns 32h .. 32h+31 of the beat
                    const uint4 a0 = tok[quad_slot<kTrit>(c, 2 * h)];
                    const uint4 a1 = tok[quad_slot<kTrit>(c, 2 * h + 1)];
#pragma unroll
                    for (int rr = 0; rr < R; rr++) {
                        const uint32_t p = h ? wv[rr].y : wv[rr].x;
                        const uint32_t n = h ? wv[rr].w : wv[rr].z;
                        int vp = 0, vn = 0;
                        vp = dp4a_us(p & 0x01010101u, a0.x, vp);
                        vn = dp4a_us(n & 0x01010101u, a0.x, vn);
                        vp = dp4a_us((p >> 1) & 0x01010101u, a0.y, vp);
                        vn = dp4a_us((n >> 1) & 0x01010101u, a0.y, vn);
                        vp = dp4a_us((p >> 2) & 0x01010101u, a0.z, vp);
                        vn = dp4a_us((n >> 2) & 0x01010101u, a0.z, vn);
                        vp = dp4a_us((p >> 3) & 0x01010101u, a0.w, vp);
                        vn = dp4a_us((n >> 3) & 0x01010101u, a0.w, vn);
                        vp = dp4a_us((p >> 4) & 0x01010101u, a1.x, vp);
                        vn = dp4a_us((n >> 4) & 0x01010101u, a1.x, vn);
                        vp = dp4a_us((p >> 5) & 0x01010101u, a1.y, vp);
                        vn = dp4a_us((n >> 5) & 0x01010101u, a1.y, vn);
                        vp = dp4a_us((p >> 6) & 0x01010101u, a1.z, vp);
                        vn = dp4a_us((n >> 6) & 0x01010101u, a1.z, vn);
                        vp = dp4a_us((p >> 7) & 0x01010101u, a1.w, vp);
                        vn = dp4a_us((n >> 7) & 0x01010101u, a1.w, vn);
                        acc[rr][b] += vp - vn;  // select-accumulate: + where pos, - where neg
                    }
                }
            }
        }
#pragma unroll
        for (int rr = 0; rr < R; rr++)
#pragma unroll
            for (int b = 0; b < B; b++) {
                const int a = warp_sum_int(acc[rr][b]);
                const int64_t row = r0 + rr;
                if (lane == 0 && row < N) {
                    const float t = __fmul_rn((float)a, x_scale[b]);
                    y[(int64_t)b * N + row] = __fmul_rn(t, w_scale);
                    if (acc_out) acc_out[(int64_t)b * N + row] = a;
                }
            }
    }
}

// ------------------------------------------------------------------------------------------
// launch helpers
// ------------------------------------------------------------------------------------------
template <int B> struct RowsFor { static constexpr int R = B <= 2 ? 4 : (B <= 4 ? 2 : 1); };

static int grid_rows(int64_t ngroups, int sms, int blocks_per_sm) {
    int64_t want = (ngroups + kWarps - 1) / kWarps;
    int64_t cap = (int64_t)sms * (blocks_per_sm > 0 ? blocks_per_sm : 1);
    if (want > cap) want = cap;
    return (int)(want < 1 ? 1 : want);
}

template <typename KernelT>
static int prepare(KernelT kernel, size_t smem, int *blocks_per_sm) {
    return prepare_kernel(reinterpret_cast<const void *>(kernel), kThreads, smem, blocks_per_sm);
}

template <int F, int B>
static int launch_q(const uint8_t *bits, const uint16_t *scales, const int8_t *q,
                    const uint16_t *d, float *y, int32_t *isum, int64_t N, int64_t K, int sms,
                    cudaStream_t st) {
    constexpr int R = RowsFor<B>::R;
    const size_t smem = (size_t)B * K + (size_t)B * (K / 32) * 8;
    int bps = 0;
    if (isum) {
        auto kern = gemv_q_kernel<F, B, R, true>;
        if (int e = prepare(kern, smem, &bps)) return e;
        kern<<<grid_rows((N + R - 1) / R, sms, bps), kThreads, smem, st>>>(bits, scales, q, d,
                                                                           y, isum, N, K);
    } else {
        auto kern = gemv_q_kernel<F, B, R, false>;
        if (int e = prepare(kern, smem, &bps)) return e;
        kern<<<grid_rows((N + R - 1) / R, sms, bps), kThreads, smem, st>>>(bits, scales, q, d,
                                                                           y, nullptr, N, K);
    }
    return launch_status();
}

template <int F>
static int dispatch_q(const uint8_t *bits, const uint16_t *scales, const int8_t *q,
                      const uint16_t *d, float *y, int32_t *isum, int64_t N, int64_t K, int B,
                      int sms, cudaStream_t st) {
    switch (B) {
        case 1: return launch_q<F, 1>(bits, scales, q, d, y, isum, N, K, sms, st);
        case 2: return launch_q<F, 2>(bits, scales, q, d, y, isum, N, K, sms, st);
        case 3: return launch_q<F, 3>(bits, scales, q, d, y, isum, N, K, sms, st);
        case 4: return launch_q<F, 4>(bits, scales, q, d, y, isum, N, K, sms, st);
        case 5: return launch_q<F, 5>(bits, scales, q, d, y, isum, N, K, sms, st);
        case 6: return launch_q<F, 6>(bits, scales, q, d, y, isum, N, K, sms, st);
        case 7: return launch_q<F, 7>(bits, scales, q, d, y, isum, N, K, sms, st);
        case 8: return launch_q<F, 8>(bits, scales, q, d, y, isum, N, K, sms, st);
    }
    return LB_ERR_BATCH;
}

template <int B>
static int launch_trit(const uint64_t *planes, float w_scale, const int8_t *q,
                       const float *x_scale, float *y, int32_t *acc, int64_t N, int64_t K,
                       int sms, cudaStream_t st) {
    constexpr int R = RowsFor<B>::R;
    const size_t smem = (size_t)B * K;
    int bps = 0;
    auto kern = gemv_trit_kernel<B, R>;
    if (int e = prepare(kern, smem, &bps)) return e;
    kern<<<grid_rows((N + R - 1) / R, sms, bps), kThreads, smem, st>>>(planes, w_scale, q,
                                                                       x_scale, y, acc, N, K);
    return launch_status();
}

static int q_args_ok(const void *bits, const void *scales, const void *q, const void *d,
                     const void *y, const void *isum, int64_t N, int64_t K, int B, int qk) {
    if (!bits || !scales || !q || !d || !y) return LB_ERR_NULL;
    if (!aligned16(bits) || !aligned16(scales) || !aligned16(q) || !aligned16(d) ||
        !aligned16(y) || (isum && !aligned16(isum)))
        return LB_ERR_ALIGN;
    if (N < 1 || K < qk || K % qk != 0) return LB_ERR_SHAPE;
    if (B < 1 || B > 8) return LB_ERR_BATCH;
    return LB_OK;
}

}  // namespace lb

using namespace lb;

LB_EXPORT int lb_gemv_q1_0(const uint8_t *bits, const uint16_t *scales, const int8_t *q,
                           const uint16_t *d, float *y, int32_t *isum_opt, int64_t N, int64_t K,
                           int B, void *stream) {
    if (int e = q_args_ok(bits, scales, q, d, y, isum_opt, N, K, B, 128)) return e;
    DeviceInfo di;
    if (int st = current_device_info(&di)) return st;
    return dispatch_q<kQ1>(bits, scales, q, d, y, isum_opt, N, K, B, di.sms, as_stream(stream));
}

LB_EXPORT int lb_gemv_q2_0_g64(const uint8_t *codes, const uint16_t *scales, const int8_t *q,
                               const uint16_t *d, float *y, int32_t *isum_opt, int64_t N,
                               int64_t K, int B, void *stream) {
    if (int e = q_args_ok(codes, scales, q, d, y, isum_opt, N, K, B, 64)) return e;
    DeviceInfo di;
    if (int st = current_device_info(&di)) return st;
    return dispatch_q<kQ2>(codes, scales, q, d, y, isum_opt, N, K, B, di.sms, as_stream(stream));
}

LB_EXPORT int lb_gemv_trit_planes(const uint64_t *planes, float w_scale, const int8_t *q,
                                  const float *x_scale, float *y, int32_t *acc_opt, int64_t N,
                                  int64_t K, int B, void *stream) {
    if (!planes || !q || !x_scale || !y) return LB_ERR_NULL;
    if (!aligned16(planes) || !aligned16(q) || !aligned16(x_scale) || !aligned16(y) ||
        (acc_opt && !aligned16(acc_opt)))
        return LB_ERR_ALIGN;
    if (N < 1 || K < 64 || K % 64 != 0 || K > (1 << 24) / 128) return LB_ERR_SHAPE;
    if (B < 1 || B > 8) return LB_ERR_BATCH;
    DeviceInfo di;
    if (int st = current_device_info(&di)) return st;
    cudaStream_t st = as_stream(stream);
    switch (B) {
        case 1: return launch_trit<1>(planes, w_scale, q, x_scale, y, acc_opt, N, K, di.sms, st);
        case 2: return launch_trit<2>(planes, w_scale, q, x_scale, y, acc_opt, N, K, di.sms, st);
        case 3: return launch_trit<3>(planes, w_scale, q, x_scale, y, acc_opt, N, K, di.sms, st);
        case 4: return launch_trit<4>(planes, w_scale, q, x_scale, y, acc_opt, N, K, di.sms, st);
        case 5: return launch_trit<5>(planes, w_scale, q, x_scale, y, acc_opt, N, K, di.sms, st);
        case 6: return launch_trit<6>(planes, w_scale, q, x_scale, y, acc_opt, N, K, di.sms, st);
        case 7: return launch_trit<7>(planes, w_scale, q, x_scale, y, acc_opt, N, K, di.sms, st);
        case 8: return launch_trit<8>(planes, w_scale, q, x_scale, y, acc_opt, N, K, di.sms, st);
    }
    return LB_ERR_BATCH;
}
