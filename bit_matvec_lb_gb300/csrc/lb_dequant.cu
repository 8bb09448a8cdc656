// lb_dequant.cu -- dequantization of packed weights: every weight as the binary32 product
// (float)w * d, stored as fp32 or rounded to bf16.
//
// "bankml: verified low-bit inference on commodity CPUs -- a technical report": III.4 and IV.2
// (every weight of every tensor dequantizes bit-identically to the reference's floats), III.2
// (Q1_0: w = +1 for a set bit, -1 otherwise), III.5 (Q2_0_g64: w = code - 1).  Planar weights
// (tritium.technology "Architecture", section 2) dequantize to w * w_scale, w in {+1, -1, 0}.
//
// HBM-bound streaming kernel: a group of 8 threads (4 for bf16) takes one 32-column group of one
// row (the packed word is read once per group and broadcast), each thread writes one 16-byte
// vector of consecutive outputs, so every warp stores 512 contiguous bytes; every thread keeps
// several groups' loads in flight.  Blocks take whole rows, so indices need no division.
#include <cuda_bf16.h>

#include <algorithm>

#include "lb_common.cuh"

namespace lb {

enum DqFmt { kDqQ1 = 0, kDqQ2 = 1, kDqTrit = 2 };

// The packed word of (row n, 32-column group g) and its scale.
template <int F>
struct DqIn {
    uint4 w;
    float d;
};

template <int F>
__device__ __forceinline__ DqIn<F> dq_load(const uint8_t *__restrict__ w,
                                           const uint16_t *__restrict__ scales, float w_scale,
                                           int64_t n, int64_t g, int64_t K, int S) {
    DqIn<F> r;
    if (F == kDqQ1) {
        // block g / 4 of the row: 16 sign bytes; this group is its 4-byte word g % 4
        r.w = make_uint4(*reinterpret_cast<const uint32_t *>(w + n * (K / 8) + g * 4), 0, 0, 0);
        r.d = f16_bits_to_float(scales[n * S + g / 4]);
    } else if (F == kDqQ2) {
        // block g / 2 of the row: 16 code bytes; this group is its 8-byte half g % 2
        const uint2 c = *reinterpret_cast<const uint2 *>(w + n * (K / 4) + g * 8);
        r.w = make_uint4(c.x, c.y, 0, 0);
        r.d = f16_bits_to_float(scales[n * S + g / 2]);
    } else {
        // beat g / 2 of the row: {pos lo, pos hi, neg lo, neg hi}; this group is half g % 2
        const uint4 b = *reinterpret_cast<const uint4 *>(w + (n * (K / 64) + g / 2) * 16);
        r.w = (g & 1) ? make_uint4(b.y, b.w, 0, 0) : make_uint4(b.x, b.z, 0, 0);
        r.d = w_scale;
    }
    return r;
}

// Columns 4 part .. 4 part + 3 of the group as (float)w * d.
template <int F>
__device__ __forceinline__ void dq_values(const DqIn<F> &in, int part, float (&v)[4]) {
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const int c = 4 * part + j;
        int wt;
        if (F == kDqQ1)
            wt = ((in.w.x >> c) & 1u) ? 1 : -1;
        else if (F == kDqQ2)
            wt = (int)(((c < 16 ? in.w.x : in.w.y) >> (2 * (c & 15))) & 3u) - 1;
        else
            wt = (int)((in.w.x >> c) & 1u) - (int)((in.w.y >> c) & 1u);
        v[j] = (float)wt * in.d;
    }
}

// A block takes whole rows (rows blockIdx.x, blockIdx.x + gridDim.x, ...).  Within a row, slot t
// = TPG g + part writes columns OUT part .. OUT part + OUT - 1 of group g (TPG threads per
// 32-column group, OUT = 32 / TPG outputs each: 4 fp32 or 8 bf16, one 16-byte store), so no
// index needs a division; each thread takes kU slots per iteration, their loads issued before
// any conversion.
constexpr int kU = 4;

template <int F, bool BF16>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t *__restrict__ w,
                                                      const uint16_t *__restrict__ scales,
                                                      float w_scale, void *__restrict__ out,
                                                      int64_t N, int64_t K, int S) {
    constexpr int TPG = BF16 ? 4 : 8;
    constexpr int LOG_TPG = BF16 ? 2 : 3;
    pdl_launch_dependents();
    pdl_wait();
    const int slots = (int)(K / 32) * TPG;
    for (int64_t n = blockIdx.x; n < N; n += gridDim.x) {
        for (int t0 = threadIdx.x; t0 < slots; t0 += kU * blockDim.x) {
            DqIn<F> in[kU];
#pragma unroll
            for (int u = 0; u < kU; u++) {
                const int t = t0 + u * (int)blockDim.x;
                if (t < slots) in[u] = dq_load<F>(w, scales, w_scale, n, t >> LOG_TPG, K, S);
            }
#pragma unroll
            for (int u = 0; u < kU; u++) {
                const int t = t0 + u * (int)blockDim.x;
                if (t >= slots) break;
                const int part = t & (TPG - 1);
                const int64_t o = n * K + (int64_t)(t >> LOG_TPG) * 32 + (32 / TPG) * part;
                if (BF16) {
                    float v0[4], v1[4];
                    dq_values<F>(in[u], 2 * part, v0);
                    dq_values<F>(in[u], 2 * part + 1, v1);
                    __nv_bfloat162 h[4] = {__floats2bfloat162_rn(v0[0], v0[1]),
                                           __floats2bfloat162_rn(v0[2], v0[3]),
                                           __floats2bfloat162_rn(v1[0], v1[1]),
                                           __floats2bfloat162_rn(v1[2], v1[3])};
                    *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + o) =
                        make_uint4(*reinterpret_cast<uint32_t *>(&h[0]),
                                   *reinterpret_cast<uint32_t *>(&h[1]),
                                   *reinterpret_cast<uint32_t *>(&h[2]),
                                   *reinterpret_cast<uint32_t *>(&h[3]));
                } else {
                    float v[4];
                    dq_values<F>(in[u], part, v);
                    *reinterpret_cast<float4 *>(static_cast<float *>(out) + o) =
                        make_float4(v[0], v[1], v[2], v[3]);
                }
            }
        }
    }
}

template <int F>
static int dequant(const void *w, const uint16_t *scales, float w_scale, int64_t N, int64_t K,
                   int out_format, void *out, void *stream) {
    const int64_t qk = F == kDqQ1 ? 128 : 64;
    if (!w || !out || (F != kDqTrit && !scales)) return LB_ERR_NULL;
    if (!aligned16(w) || !aligned16(out) || (scales && !aligned16(scales))) return LB_ERR_ALIGN;
    if (N < 1 || N > (1ll << 30) || K < qk || K % qk != 0 || K > (1ll << 26)) return LB_ERR_SHAPE;
    if (out_format != LB_OUT_F32 && out_format != LB_OUT_BF16) return LB_ERR_SHAPE;
    DeviceInfo di;
    if (int st = current_device_info(&di)) return st;
    // whole rows per block: enough blocks for 8 resident per SM (fewer for few rows)
    int64_t grid = std::min<int64_t>(N, (int64_t)di.sms * 8);
    const int S = (int)((K / qk + 7) / 8 * 8);
    const uint8_t *wb = static_cast<const uint8_t *>(w);
    cudaStream_t st = as_stream(stream);
    if (out_format == LB_OUT_BF16)
        return launch_pdl(dequant_kernel<F, true>, dim3((unsigned)grid), dim3(256), 0, st, wb,
                          scales, w_scale, out, N, K, S);
    return launch_pdl(dequant_kernel<F, false>, dim3((unsigned)grid), dim3(256), 0, st, wb,
                      scales, w_scale, out, N, K, S);
}

}  // namespace lb

using namespace lb;

LB_EXPORT int lb_dequantize_q1_0(const uint8_t *bits, const uint16_t *scales, int64_t N,
                                 int64_t K, int out_format, void *out, void *stream) {
    return dequant<kDqQ1>(bits, scales, 0.f, N, K, out_format, out, stream);
}

LB_EXPORT int lb_dequantize_q2_0_g64(const uint8_t *codes, const uint16_t *scales, int64_t N,
                                     int64_t K, int out_format, void *out, void *stream) {
    return dequant<kDqQ2>(codes, scales, 0.f, N, K, out_format, out, stream);
}

LB_EXPORT int lb_dequantize_trit_planes(const uint64_t *planes, float w_scale, int64_t N,
                                        int64_t K, int out_format, void *out, void *stream) {
    return dequant<kDqTrit>(planes, nullptr, w_scale, N, K, out_format, out, stream);
}
