// lb_gemv_q.cuh -- argument checks and launch of the Q1_0 / Q2_0_g64 x q8_0 decode GEMVs
// (single matrix and grouped); the kernel is the streaming GEMV of lb_stream.cuh.  Each format's
// entry points live in their own translation unit so the two sets of kernel instances compile
// in parallel.
#pragma once
#include "lb_stream.cuh"

namespace lb {

template <int F>
inline int gemv_q_grouped(const lb_q_matrix *mats, int G, const int8_t *q, const uint16_t *d,
                          int64_t K, int B, void *stream) {
    const int qk = F == kQ1 ? 128 : 64;
    if (!mats || !q || !d) return LB_ERR_NULL;
    if (G < 1 || G > kMaxGroup) return LB_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(d)) return LB_ERR_ALIGN;
    if (K < qk || K % qk != 0 || K > (1ll << 24)) return LB_ERR_SHAPE;
    if (B < 1 || B > 8) return LB_ERR_BATCH;
    bool aux = false;
    for (int i = 0; i < G; i++) {
        const lb_q_matrix &m = mats[i];
        if (!m.bits || !m.scales || !m.y) return LB_ERR_NULL;
        if (!aligned16(m.bits) || !aligned16(m.scales) || !aligned16(m.y) ||
            (m.isum_opt && !aligned16(m.isum_opt)))
            return LB_ERR_ALIGN;
        if (m.N < 1 || m.N > (1ll << 30)) return LB_ERR_SHAPE;
        aux = aux || m.isum_opt != nullptr;
    }
    DeviceInfo di;
    if (int st = current_device_info(&di)) return st;
    StreamParams p = {};
    for (int i = 0; i < G; i++) {
        p.m[i].w = mats[i].bits;
        p.m[i].scales = mats[i].scales;
        p.m[i].y = mats[i].y;
        p.m[i].aux = mats[i].isum_opt;
        p.m[i].N = (int32_t)mats[i].N;
    }
    p.G = G;
    p.q = q;
    p.d = d;
    p.err = device_error_word();
    if (!p.err) return LB_ERR_LAUNCH;
    p.K = K;
    p.nchunk = (int32_t)(K / qk);
    p.S = (int32_t)scale_stride(K, qk);
    return dispatch_stream<F>(p, B, aux, di.sms, as_stream(stream));
}

}  // namespace lb
