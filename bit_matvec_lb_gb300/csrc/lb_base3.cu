// lb_base3.cu -- base-3 packed ternary weights: five trits per byte, and the decode GEMV on them.
//
// "bankml: verified low-bit inference on commodity CPUs -- a technical report", III.8: a trit
// carries log2(3) bits and, since 3^5 = 243 <= 256, five trits fit in one byte (1.6 bits per
// trit, within 1 % of the bound); tritium.technology "Architecture", open questions: base-3
// packing saves about 20 % of the ternary body's bytes against an unpack cost.  This file is that
// experiment on the GPU.  Layout (the pages fix none; the plainest reading): byte j of 16-byte
// group g of a row holds columns 80g + 5j + i, i = 0..4, as sum_i (t + 1) * 3^i (the lowest
// column in the lowest digit); a row is ceil(K/80) groups and columns past K hold trit 0.  The
// product is the planar one (sections 1, 4.1, 5): acc = sum_{t=+1} q - sum_{t=-1} q (int32,
// exact), y = (float(acc) * x_scale) * w_scale, so it equals lb_gemv_trit_planes bit for bit.
//
// GEMV design.  Warp per weight row (two rows in flight per warp), lane per 16-byte group of
// the row (coalesced 512-byte warp loads).  A byte is decoded by one lookup in a 256-entry table
// in shared memory (byte -> trits 0..3 as int8x4 and trit 4; bytes above 242 read as zero
// trits), replicated 16 times so the lanes of a half-warp never share a bank.  The activation image of every token is staged once per CTA,
// permuted per 80-column group so that the table's int8x4 of byte j lines up with one activation
// word (columns 5j .. 5j+3) and the fifth trits of four bytes, gathered by byte permutes, with a
// second word; dp4a accumulates.  Row sums by warp shuffles.
#include <algorithm>

#include "lb_common.cuh"

namespace lb {

constexpr int kB3Threads = 256;
constexpr int kB3Warps = kB3Threads / 32;
constexpr int kB3Rep = 16;                         // table copies (one per half-warp lane)
constexpr int kB3LutBytes = 256 * kB3Rep * 8;      // uint2 entries, every byte value
constexpr int kB3RowsPerWarp = 2;                  // rows in flight per warp
constexpr int kB3GroupsPerLane = 4;                // groups of one row loaded per batch

__host__ __device__ constexpr int64_t b3_groups(int64_t K) { return (K + 79) / 80; }

// ------------------------------------------------------------------------------------------
// Packing from the planar layout: one thread per output byte.  Writes weights, so it never
// lets the next kernel start early (see pdl_wait()).
// ------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) pack_base3_kernel(const uint64_t *__restrict__ planes,
                                                         uint8_t *__restrict__ out, int64_t N,
                                                         int64_t K) {
    pdl_wait();
    const int64_t G = b3_groups(K), nbeat = K / 64;
    const int64_t total = N * G * 16;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t r = i / (G * 16), rem = i % (G * 16);
        const int64_t c0 = (rem / 16) * 80 + (rem % 16) * 5;
        int value = 0, place = 1;
#pragma unroll
        for (int d = 0; d < 5; d++) {
            const int64_t c = c0 + d;
            int t = 0;
            if (c < K) {
                const uint64_t *beat = planes + (r * nbeat + c / 64) * 2;
                const int bit = (int)(c & 63);
                t = (int)((beat[0] >> bit) & 1u) - (int)((beat[1] >> bit) & 1u);
            }
            value += (t + 1) * place;
            place *= 3;
        }
        out[i] = (uint8_t)value;
    }
}

// ------------------------------------------------------------------------------------------
// GEMV
// ------------------------------------------------------------------------------------------
struct B3Params {
    const uint8_t *w;        // [N][G * 16]
    const int8_t *q;         // [B][K]
    const float *x_scale;    // [B]
    float *y;                // [B][N]
    int32_t *acc;            // [B][N] or NULL
    float w_scale;
    int64_t N, K;
    int G;
};

__device__ __forceinline__ uint32_t b3_word(const uint4 &v, int t) {
    return t == 0 ? v.x : (t == 1 ? v.y : (t == 2 ? v.z : v.w));
}

// Fifth trits (byte 0 of h[k], int8) of four consecutive bytes as one int8x4 word.
__device__ __forceinline__ uint32_t gather4(uint32_t h0, uint32_t h1, uint32_t h2, uint32_t h3) {
    return prmt(prmt(h0, h1, 0x0040u), prmt(h2, h3, 0x0040u), 0x5410u);
}

template <int B>
__global__ void __launch_bounds__(kB3Threads) gemv_base3_kernel(const __grid_constant__ B3Params p) {
    extern __shared__ __align__(16) uint8_t b3sm[];
    uint2 *lut = reinterpret_cast<uint2 *>(b3sm);                  // [256][kB3Rep]
    uint4 *img = reinterpret_cast<uint4 *>(b3sm + kB3LutBytes);    // [B][G][5]
    pdl_launch_dependents();
    // decoding table: byte value -> trits 0..3 (int8x4) and trit 4 (byte 0); values above 242
    // are not base-3 bytes and decode as zero trits (so every lookup stays in the table)
    for (int e = threadIdx.x; e < 256 * kB3Rep; e += blockDim.x) {
        int v = e / kB3Rep;
        if (v > 242) v = 121;
        uint32_t lo = 0;
#pragma unroll
        for (int d = 0; d < 4; d++) {
            lo |= (uint32_t)(uint8_t)(int8_t)(v % 3 - 1) << (8 * d);
            v /= 3;
        }
        lut[e] = make_uint2(lo, (uint32_t)(uint8_t)(int8_t)(v % 3 - 1));
    }
    pdl_wait();
    // activation image: uint4 u < 4 of group g holds words 4u..4u+3, word j = columns 5j..5j+3;
    // uint4 4 holds word v = columns 5(4v+k)+4, k = 0..3.  Columns past K are zero.
    const int G = p.G;
    for (int i = threadIdx.x; i < B * G; i += blockDim.x) {
        const int b = i / G, g = i % G;
        const int8_t *src = p.q + (int64_t)b * p.K + (int64_t)g * 80;
        const int64_t left = p.K - (int64_t)g * 80;
        uint8_t x[80];
        if (left >= 80) {
#pragma unroll
            for (int u = 0; u < 5; u++) {
                const uint4 v = reinterpret_cast<const uint4 *>(src)[u];
                const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int k = 0; k < 16; k++) x[16 * u + k] = (uint8_t)(wv[k / 4] >> (8 * (k % 4)));
            }
        } else {
#pragma unroll
            for (int k = 0; k < 80; k++) x[k] = k < left ? (uint8_t)src[k] : 0;
        }
        uint32_t wd[20];
#pragma unroll
        for (int j = 0; j < 16; j++)
            wd[j] = (uint32_t)x[5 * j] | ((uint32_t)x[5 * j + 1] << 8) |
                    ((uint32_t)x[5 * j + 2] << 16) | ((uint32_t)x[5 * j + 3] << 24);
#pragma unroll
        for (int v = 0; v < 4; v++)
            wd[16 + v] = (uint32_t)x[20 * v + 4] | ((uint32_t)x[20 * v + 9] << 8) |
                         ((uint32_t)x[20 * v + 14] << 16) | ((uint32_t)x[20 * v + 19] << 24);
        uint4 *dst = img + (int64_t)i * 5;
#pragma unroll
        for (int u = 0; u < 5; u++)
            dst[u] = make_uint4(wd[4 * u], wd[4 * u + 1], wd[4 * u + 2], wd[4 * u + 3]);
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint2 *mylut = lut + (lane & (kB3Rep - 1));
    const int64_t row_bytes = (int64_t)G * 16;
    const int64_t nwarps = (int64_t)gridDim.x * kB3Warps;
    float xs[B];
#pragma unroll
    for (int b = 0; b < B; b++) xs[b] = p.x_scale[b];

    for (int64_t r0 = ((int64_t)blockIdx.x * kB3Warps + warp) * kB3RowsPerWarp; r0 < p.N;
         r0 += nwarps * kB3RowsPerWarp) {
        // NA independent partial sums per row and token (at 1-2 tokens the dp4a chains of one
        // row would otherwise be a single serial dependence)
        constexpr int NA = B <= 2 ? 4 : 1;
        int acc[kB3RowsPerWarp][B][NA];
#pragma unroll
        for (int rr = 0; rr < kB3RowsPerWarp; rr++)
#pragma unroll
            for (int b = 0; b < B; b++)
#pragma unroll
                for (int c = 0; c < NA; c++) acc[rr][b][c] = 0;
        for (int g0 = 0; g0 < G; g0 += 32 * kB3GroupsPerLane) {
            uint4 wv[kB3RowsPerWarp][kB3GroupsPerLane];
            // every load of the batch first (rows past N and groups past G read nothing)
#pragma unroll
            for (int rr = 0; rr < kB3RowsPerWarp; rr++)
#pragma unroll
                for (int k = 0; k < kB3GroupsPerLane; k++) {
                    const int g = g0 + 32 * k + lane;
                    const int64_t r = r0 + rr;
                    wv[rr][k] = (r < p.N && g < G)
                                    ? ldg_stream(p.w + r * row_bytes + (int64_t)g * 16)
                                    : make_uint4(0x79797979u, 0x79797979u, 0x79797979u,
                                                 0x79797979u);  // byte 121: five zero trits
                }
#pragma unroll
            for (int k = 0; k < kB3GroupsPerLane; k++) {
                const int g = g0 + 32 * k + lane;
                if (g >= G) break;
                const uint4 *a = img + (int64_t)g * 5;
#pragma unroll
                for (int rr = 0; rr < kB3RowsPerWarp; rr++) {
                    const uint32_t words[4] = {wv[rr][k].x, wv[rr][k].y, wv[rr][k].z,
                                               wv[rr][k].w};
#pragma unroll
                    for (int u = 0; u < 4; u++) {
                        uint2 e[4];
#pragma unroll
                        for (int k2 = 0; k2 < 4; k2++)
                            e[k2] = mylut[((words[u] >> (8 * k2)) & 0xFFu) * kB3Rep];
                        const uint32_t w4 = gather4(e[0].y, e[1].y, e[2].y, e[3].y);
#pragma unroll
                        for (int b = 0; b < B; b++) {
                            const uint4 av = a[(int64_t)b * G * 5 + u];
                            const uint32_t a5 = b3_word(a[(int64_t)b * G * 5 + 4], u);
                            int s = acc[rr][b][u % NA];
                            s = dp4a_ss(e[0].x, av.x, s);
                            s = dp4a_ss(e[1].x, av.y, s);
                            s = dp4a_ss(e[2].x, av.z, s);
                            s = dp4a_ss(e[3].x, av.w, s);
                            acc[rr][b][u % NA] = dp4a_ss(w4, a5, s);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int rr = 0; rr < kB3RowsPerWarp; rr++) {
#pragma unroll
            for (int b = 0; b < B; b++) {
                int s = acc[rr][b][0];
#pragma unroll
                for (int c = 1; c < NA; c++) s += acc[rr][b][c];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                acc[rr][b][0] = s;
            }
            const int64_t r = r0 + rr;
            if (lane == 0 && r < p.N) {
#pragma unroll
                for (int b = 0; b < B; b++) {
                    const float f = (float)acc[rr][b][0];
                    p.y[(int64_t)b * p.N + r] = __fmul_rn(__fmul_rn(f, xs[b]), p.w_scale);
                    if (p.acc) p.acc[(int64_t)b * p.N + r] = acc[rr][b][0];
                }
            }
        }
    }
}

template <int B>
static int launch_base3(const B3Params &p, size_t smem, int sms, cudaStream_t st) {
    auto kern = gemv_base3_kernel<B>;
    int bps = 0;
    if (int e = prepare_kernel(reinterpret_cast<const void *>(kern), kB3Threads, smem, &bps))
        return e;
    if (bps < 1) return LB_ERR_SHAPE;
    const int64_t warps_needed = (p.N + kB3RowsPerWarp - 1) / kB3RowsPerWarp;
    int64_t grid = (warps_needed + kB3Warps - 1) / kB3Warps;
    grid = std::min<int64_t>(grid, (int64_t)sms * bps);
    return launch_pdl(kern, dim3((unsigned)grid), dim3(kB3Threads), smem, st, p);
}

}  // namespace lb

using namespace lb;

LB_EXPORT int lb_pack_base3(const uint64_t *planes, int64_t N, int64_t K, uint8_t *packed,
                            void *stream) {
    if (!planes || !packed) return LB_ERR_NULL;
    if (!aligned16(planes) || !aligned16(packed)) return LB_ERR_ALIGN;
    if (N < 1 || N > (1ll << 30) || K < 64 || K % 64 != 0 || K > (1 << 24) / 128)
        return LB_ERR_SHAPE;
    DeviceInfo di;
    if (int st = current_device_info(&di)) return st;
    const int64_t total = N * b3_groups(K) * 16;
    int64_t grid = (total + 255) / 256;
    if (grid > (int64_t)di.sms * 16) grid = (int64_t)di.sms * 16;
    return launch_pdl(pack_base3_kernel, dim3((unsigned)grid), dim3(256), 0, as_stream(stream),
                      planes, packed, N, K);
}

LB_EXPORT int lb_gemv_base3(const uint8_t *packed, float w_scale, const int8_t *q,
                            const float *x_scale, float *y, int32_t *acc_opt, int64_t N,
                            int64_t K, int B, void *stream) {
    if (!packed || !q || !x_scale || !y) return LB_ERR_NULL;
    if (!aligned16(packed) || !aligned16(q) || !aligned16(x_scale) || !aligned16(y) ||
        (acc_opt && !aligned16(acc_opt)))
        return LB_ERR_ALIGN;
    if (N < 1 || N > (1ll << 30) || K < 64 || K % 64 != 0 || K > (1 << 24) / 128)
        return LB_ERR_SHAPE;
    if (B < 1 || B > 8) return LB_ERR_BATCH;
    const int64_t G = b3_groups(K);
    const size_t smem = (size_t)kB3LutBytes + (size_t)B * (size_t)G * 80;
    if (smem > 200 * 1024) return LB_ERR_SHAPE;
    DeviceInfo di;
    if (int st = current_device_info(&di)) return st;
    B3Params p{packed, q, x_scale, y, acc_opt, w_scale, N, K, (int)G};
    cudaStream_t st = as_stream(stream);
    switch (B) {
        case 1: return launch_base3<1>(p, smem, di.sms, st);
        case 2: return launch_base3<2>(p, smem, di.sms, st);
        case 3: return launch_base3<3>(p, smem, di.sms, st);
        case 4: return launch_base3<4>(p, smem, di.sms, st);
        case 5: return launch_base3<5>(p, smem, di.sms, st);
        case 6: return launch_base3<6>(p, smem, di.sms, st);
        case 7: return launch_base3<7>(p, smem, di.sms, st);
        default: return launch_base3<8>(p, smem, di.sms, st);
    }
}
