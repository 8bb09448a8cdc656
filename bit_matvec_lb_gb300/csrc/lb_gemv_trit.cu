// lb_gemv_trit.cu -- entry points of the planar ternary decode GEMV (single matrix and
// grouped); the kernel is the streaming GEMV of lb_stream.cuh.
#include "lb_stream.cuh"

using namespace lb;

LB_EXPORT int lb_gemv_trit_planes_grouped(const lb_trit_matrix *mats, int G, const int8_t *q,
                                          const float *x_scale, int64_t K, int B,
                                          void *stream) {
    if (!mats || !q || !x_scale) return LB_ERR_NULL;
    if (G < 1 || G > kMaxGroup) return LB_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(x_scale)) return LB_ERR_ALIGN;
    if (K < 64 || K % 64 != 0 || K > (1 << 24) / 128) return LB_ERR_SHAPE;
    if (B < 1 || B > 8) return LB_ERR_BATCH;
    for (int i = 0; i < G; i++) {
        const lb_trit_matrix &m = mats[i];
        if (!m.planes || !m.y) return LB_ERR_NULL;
        if (!aligned16(m.planes) || !aligned16(m.y) || (m.acc_opt && !aligned16(m.acc_opt)))
            return LB_ERR_ALIGN;
        if (m.N < 1 || m.N > (1ll << 30)) return LB_ERR_SHAPE;
    }
    DeviceInfo di;
    if (int st = current_device_info(&di)) return st;
    StreamParams p = {};
    for (int i = 0; i < G; i++) {
        p.m[i].w = reinterpret_cast<const uint8_t *>(mats[i].planes);
        p.m[i].scales = nullptr;
        p.m[i].y = mats[i].y;
        p.m[i].aux = mats[i].acc_opt;  // written by the epilogue of every configuration
        p.m[i].w_scale = mats[i].w_scale;
        p.m[i].N = (int32_t)mats[i].N;
    }
    p.G = G;
    p.q = q;
    p.x_scale = x_scale;
    p.err = device_error_word();
    if (!p.err) return LB_ERR_LAUNCH;
    p.K = K;
    p.nchunk = (int32_t)(K / 64);
    p.S = 0;
    return dispatch_stream<kTrit>(p, B, false, di.sms, as_stream(stream));
}

LB_EXPORT int lb_gemv_trit_planes(const uint64_t *planes, float w_scale, const int8_t *q,
                                  const float *x_scale, float *y, int32_t *acc_opt, int64_t N,
                                  int64_t K, int B, void *stream) {
    const lb_trit_matrix m = {planes, w_scale, y, acc_opt, N};
    return lb_gemv_trit_planes_grouped(&m, 1, q, x_scale, K, B, stream);
}
