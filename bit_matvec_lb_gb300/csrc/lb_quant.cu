// lb_quant.cu -- activation quantizers and the load-time weight repack.
//
// q8_0 follows "bankml: verified low-bit inference on commodity CPUs -- a technical report",
// section III.2 (blocks of 32 signed bytes with their own fp16 scale, scale from 127 / max|x|,
// round half to even) and bankml BUILD_HISTORY.md, ledger item P2 ("AVX2 quantizer: 127/amax,
// round-half-even").  Every step is binary32 with IEEE division (no fast-math), so the codes
// and scales are bit-identical to a scalar evaluation of the same formula.
#include "lb_common.cuh"

namespace lb {

// One q8_0 block of 32 values is handled by 8 consecutive lanes, 4 values (one float4) each.
__global__ void __launch_bounds__(256) quantize_q8_0_kernel(const float4 *__restrict__ x,
                                                            uint32_t *__restrict__ q,
                                                            uint16_t *__restrict__ d,
                                                            int64_t nquads) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int lane = threadIdx.x & 31;
    // The loop condition is warp-uniform so every lane reaches the shuffles; nquads is a
    // multiple of 8, so a group of 8 lanes (one q8_0 block) is either wholly valid or not.
    for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31); i0 < nquads;
         i0 += stride) {
        const int64_t i = i0 + lane;
        const bool ok = i < nquads;
        float4 v = ok ? x[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        float a = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
        const float amax = a;
        const float id = (amax != 0.0f) ? __fdiv_rn(127.0f, amax) : 0.0f;
        const int q0 = __float2int_rn(__fmul_rn(v.x, id));
        const int q1 = __float2int_rn(__fmul_rn(v.y, id));
        const int q2 = __float2int_rn(__fmul_rn(v.z, id));
        const int q3 = __float2int_rn(__fmul_rn(v.w, id));
        if (!ok) continue;
        q[i] = (uint32_t)(q0 & 0xFF) | ((uint32_t)(q1 & 0xFF) << 8) |
               ((uint32_t)(q2 & 0xFF) << 16) | ((uint32_t)(q3 & 0xFF) << 24);
        if ((lane & 7) == 0)
            d[i >> 3] = __half_as_ushort(__float2half_rn(__fdiv_rn(amax, 127.0f)));
    }
}

// Per-token absmax int8: one CTA per token.  The first kHold float4 of each thread stay in
// registers between the absmax pass and the quantize pass (one read of the row up to
// K = 512 * 4 * kHold); the rest of a longer row is read twice.
constexpr int kHold = 4;

__global__ void __launch_bounds__(512) quantize_i8_absmax_kernel(const float *__restrict__ x,
                                                                 int8_t *__restrict__ q,
                                                                 float *__restrict__ x_scale,
                                                                 int64_t K) {
    __shared__ float red[32];
    pdl_launch_dependents();
    pdl_wait();
    const int64_t b = blockIdx.x;
    const float4 *xb = reinterpret_cast<const float4 *>(x + b * K);
    const int64_t nq = K / 4;
    float a = 0.0f;
    float4 held[kHold];
#pragma unroll
    for (int r = 0; r < kHold; r++) {
        const int64_t i = threadIdx.x + (int64_t)r * blockDim.x;
        held[r] = i < nq ? xb[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 v = held[r];
        a = fmaxf(a, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    for (int64_t i = threadIdx.x + (int64_t)kHold * blockDim.x; i < nq; i += blockDim.x) {
        float4 v = xb[i];
        a = fmaxf(a, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
    __syncthreads();
    if (threadIdx.x < 32) {
        a = (threadIdx.x < (blockDim.x >> 5)) ? red[threadIdx.x] : 0.0f;
        for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        if (threadIdx.x == 0) red[0] = a;
    }
    __syncthreads();
    const float amax = red[0];
    const float s = (amax != 0.0f) ? __fdiv_rn(127.0f, amax) : 0.0f;
    if (threadIdx.x == 0) x_scale[b] = __fdiv_rn(amax, 127.0f);
    uint32_t *qb = reinterpret_cast<uint32_t *>(q + b * K);
#pragma unroll
    for (int r = 0; r < kHold; r++) {
        const int64_t i = threadIdx.x + (int64_t)r * blockDim.x;
        if (i < nq) qb[i] = quantize_i8_word(held[r], s);
    }
    for (int64_t i = threadIdx.x + (int64_t)kHold * blockDim.x; i < nq; i += blockDim.x)
        qb[i] = quantize_i8_word(xb[i], s);
}

// One thread per scale slot (n, j), j < S: block j of row n when j < nblk (fp16 scale to
// `scales`, 16 data bytes to `bits`), a zero padding scale otherwise.
__global__ void __launch_bounds__(256) repack_kernel(const uint8_t *__restrict__ blocks,
                                                     uint4 *__restrict__ bits,
                                                     uint16_t *__restrict__ scales, int64_t N,
                                                     int64_t nblk, int64_t S) {
    // No early trigger here: repack WRITES weights, and the GEMVs read weights before their
    // grid-dependency wait, so a kernel launched after a repack must start only once the repack
    // has completed.
    pdl_wait();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < N * S; i += stride) {
        const int64_t n = i / S, j = i % S;
        if (j >= nblk) {
            scales[i] = 0;
            continue;
        }
        const int64_t b = n * nblk + j;
        const uint8_t *src = blocks + b * 18;
        scales[i] = (uint16_t)(src[0] | ((uint16_t)src[1] << 8));
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; k++)
            w[k] = (uint32_t)src[2 + 4 * k] | ((uint32_t)src[3 + 4 * k] << 8) |
                   ((uint32_t)src[4 + 4 * k] << 16) | ((uint32_t)src[5 + 4 * k] << 24);
        bits[b] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

static int grid_for(int64_t work, int threads, int sms) {
    int64_t g = (work + threads - 1) / threads;
    int64_t cap = (int64_t)sms * 16;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return (int)g;
}

}  // namespace lb

using namespace lb;

LB_EXPORT int lb_quantize_q8_0(const float *x, int8_t *q, uint16_t *d, int64_t B, int64_t K,
                               void *stream) {
    if (!x || !q || !d) return LB_ERR_NULL;
    if (!aligned16(x) || !aligned16(q) || !aligned16(d)) return LB_ERR_ALIGN;
    if (B < 1 || K < 32 || K % 32 != 0) return LB_ERR_SHAPE;
    DeviceInfo di;
    if (int st = current_device_info(&di)) return st;
    const int64_t nquads = B * K / 4;
    return launch_pdl(quantize_q8_0_kernel, dim3(grid_for(nquads, 256, di.sms)), dim3(256), 0,
                      as_stream(stream), reinterpret_cast<const float4 *>(x),
                      reinterpret_cast<uint32_t *>(q), d, nquads);
}

LB_EXPORT int lb_quantize_i8_absmax(const float *x, int8_t *q, float *x_scale, int64_t B,
                                    int64_t K, void *stream) {
    if (!x || !q || !x_scale) return LB_ERR_NULL;
    if (!aligned16(x) || !aligned16(q) || !aligned16(x_scale)) return LB_ERR_ALIGN;
    if (B < 1 || B > 0x7fffffff || K < 16 || K % 16 != 0) return LB_ERR_SHAPE;
    DeviceInfo di;
    if (int st = current_device_info(&di)) return st;
    return launch_pdl(quantize_i8_absmax_kernel, dim3((unsigned)B), dim3(512), 0,
                      as_stream(stream), x, q, x_scale, K);
}

static int repack_common(const void *blocks18, int64_t N, int64_t K, int qk, uint8_t *bits,
                         uint16_t *scales, void *stream) {
    if (!blocks18 || !bits || !scales) return LB_ERR_NULL;
    if (!aligned16(bits) || !aligned16(scales)) return LB_ERR_ALIGN;
    if (N < 1 || K < qk || K % qk != 0) return LB_ERR_SHAPE;
    DeviceInfo di;
    if (int st = current_device_info(&di)) return st;
    const int64_t nblk = K / qk, S = (nblk + 7) / 8 * 8;
    return launch_pdl(repack_kernel, dim3(grid_for(N * S, 256, di.sms)), dim3(256), 0,
                      as_stream(stream), reinterpret_cast<const uint8_t *>(blocks18),
                      reinterpret_cast<uint4 *>(bits), scales, N, nblk, S);
}

LB_EXPORT int lb_repack_q1_0(const void *blocks18, int64_t N, int64_t K, uint8_t *bits,
                             uint16_t *scales, void *stream) {
    return repack_common(blocks18, N, K, 128, bits, scales, stream);
}

LB_EXPORT int lb_repack_q2_0_g64(const void *blocks18, int64_t N, int64_t K, uint8_t *codes,
                                 uint16_t *scales, void *stream) {
    return repack_common(blocks18, N, K, 64, codes, scales, stream);
}
