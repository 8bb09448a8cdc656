// lb_bf16.cu -- dense bf16 head GEMV: y[b][n] = sum_k float(W[n][k]) * x[b][k].
//
// tritium.technology "Architecture", section 3: the dense head of a tied-embedding model is
// the largest single weight stream of a token; it is stored bf16 (the checkpoint's precision)
// and widened exactly for an f32 product.  Widening bf16 is a 16-bit left shift.
//
// GPU design: each lane streams 16-byte chunks (8 weights) of R rows (8 at one or two tokens,
// 4 otherwise: every activation read from shared memory serves R rows) with L1-bypassing loads;
// the B activation rows sit in shared memory (fp32, swizzled per 16 bytes so 8 consecutive
// lanes read distinct banks) and are reused for the R rows; fp32 FMAs accumulate per lane, and
// at 4 and 8 tokens one multi-value warp reduction finishes the R x B sums of a row group (a
// tree per sum otherwise).
#include "lb_common.cuh"

namespace lb {

constexpr int kBfThreads = 256;
constexpr int kBfWarps = kBfThreads / 32;

__device__ __forceinline__ int64_t bf_slot(int64_t c, int h) {
    return 2 * c + (h ^ (int)((c >> 2) & 1));
}

template <int B, int R>
__global__ void __launch_bounds__(kBfThreads)
    gemv_bf16_kernel(const uint16_t *__restrict__ w, const float *__restrict__ x,
                     float *__restrict__ y, int64_t N, int64_t K) {
    extern __shared__ float4 xs[];  // [B][K/4] float4, swizzled in pairs
    const int64_t nchunk = K / 8;
    pdl_launch_dependents();
    pdl_wait();
    for (int64_t i = threadIdx.x; i < (int64_t)B * nchunk * 2; i += blockDim.x) {
        const int64_t b = i / (nchunk * 2), rem = i % (nchunk * 2);
        const int64_t c = rem >> 1;
        const int h = (int)(rem & 1);
        xs[b * nchunk * 2 + bf_slot(c, h)] = reinterpret_cast<const float4 *>(x + b * K)[rem];
    }
    __syncthreads();

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t ngroups = (N + R - 1) / R;
    for (int64_t g = (int64_t)blockIdx.x * kBfWarps + warp; g < ngroups;
         g += (int64_t)gridDim.x * kBfWarps) {
        const int64_t r0 = g * R;
        float acc[R][B];
#pragma unroll
        for (int rr = 0; rr < R; rr++)
#pragma unroll
            for (int b = 0; b < B; b++) acc[rr][b] = 0.0f;
        for (int64_t c = lane; c < nchunk; c += 32) {
            float wf[R][8];
#pragma unroll
            for (int rr = 0; rr < R; rr++) {
                const int64_t row = r0 + rr;
                uint4 v = row < N ? ldg_stream(w + (row * nchunk + c) * 8) : make_uint4(0, 0, 0, 0);
                const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    wf[rr][2 * j] = __uint_as_float(u[j] << 16);
                    wf[rr][2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
                }
            }
#pragma unroll
            for (int b = 0; b < B; b++) {
                const float4 x0 = xs[b * nchunk * 2 + bf_slot(c, 0)];
                const float4 x1 = xs[b * nchunk * 2 + bf_slot(c, 1)];
                const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                for (int rr = 0; rr < R; rr++)
#pragma unroll
                    for (int j = 0; j < 8; j++) acc[rr][b] = fmaf(wf[rr][j], xv[j], acc[rr][b]);
            }
        }
        constexpr int V = R * B;
        if constexpr (B >= 4 && (V & (V - 1)) == 0) {
            // the R x B sums over the warp in one multi-value reduction, one lane per result
            constexpr int kSpan = 32 / PowTwo<V>::value;
            float part[V];
#pragma unroll
            for (int rr = 0; rr < R; rr++)
#pragma unroll
                for (int b = 0; b < B; b++) part[rr * B + b] = acc[rr][b];
            const float tot = warp_sum_many<V>(part, lane);
            const int vi = lane / kSpan, rr = vi / B, b = vi % B;
            if (lane % kSpan == 0 && r0 + rr < N) y[(int64_t)b * N + r0 + rr] = tot;
        } else {
            // one tree per sum (padding to a power of two would cost registers; at one token the
            // multi-value form measured slower: 6.06 -> 4.29 TB/s on the BitNet head)
#pragma unroll
            for (int rr = 0; rr < R; rr++)
#pragma unroll
                for (int b = 0; b < B; b++) {
                    float v = acc[rr][b];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    if (lane == 0 && r0 + rr < N) y[(int64_t)b * N + r0 + rr] = v;
                }
        }
    }
}

template <int B>
static int launch_bf16(const uint16_t *w, const float *x, float *y, int64_t N, int64_t K,
                       int sms, cudaStream_t st) {
    constexpr int R = B <= 2 ? 8 : 4;
    const size_t smem = (size_t)B * K * 4;
    auto kern = gemv_bf16_kernel<B, R>;
    int bps = 0;
    if (int e = prepare_kernel(reinterpret_cast<const void *>(kern), kBfThreads, smem, &bps))
        return e;
    int64_t want = ((N + R - 1) / R + kBfWarps - 1) / kBfWarps;
    int64_t cap = (int64_t)sms * bps;
    int grid = (int)(want < cap ? (want < 1 ? 1 : want) : cap);
    return launch_pdl(kern, dim3(grid), dim3(kBfThreads), smem, st, w, x, y, N, K);
}

}  // namespace lb

using namespace lb;

LB_EXPORT int lb_gemv_bf16(const uint16_t *w, const float *x, float *y, int64_t N, int64_t K,
                           int B, void *stream) {
    if (!w || !x || !y) return LB_ERR_NULL;
    if (!aligned16(w) || !aligned16(x) || !aligned16(y)) return LB_ERR_ALIGN;
    if (N < 1 || K < 8 || K % 8 != 0) return LB_ERR_SHAPE;
    if (B < 1 || B > 8) return LB_ERR_BATCH;
    DeviceInfo di;
    if (int s = current_device_info(&di)) return s;
    cudaStream_t st = as_stream(stream);
    switch (B) {
        case 1: return launch_bf16<1>(w, x, y, N, K, di.sms, st);
        case 2: return launch_bf16<2>(w, x, y, N, K, di.sms, st);
        case 3: return launch_bf16<3>(w, x, y, N, K, di.sms, st);
        case 4: return launch_bf16<4>(w, x, y, N, K, di.sms, st);
        case 5: return launch_bf16<5>(w, x, y, N, K, di.sms, st);
        case 6: return launch_bf16<6>(w, x, y, N, K, di.sms, st);
        case 7: return launch_bf16<7>(w, x, y, N, K, di.sms, st);
        case 8: return launch_bf16<8>(w, x, y, N, K, di.sms, st);
    }
    return LB_ERR_BATCH;
}
