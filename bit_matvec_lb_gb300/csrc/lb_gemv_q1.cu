// lb_gemv_q1.cu -- entry points of the Q1_0 x q8_0 decode GEMVs (single matrix and grouped).
#include "lb_gemv_q.cuh"

using namespace lb;

LB_EXPORT int lb_gemv_q1_0_grouped(const lb_q_matrix *mats, int G, const int8_t *q,
                                   const uint16_t *d, int64_t K, int B, void *stream) {
    return gemv_q_grouped<kQ1>(mats, G, q, d, K, B, stream);
}

LB_EXPORT int lb_gemv_q1_0(const uint8_t *bits, const uint16_t *scales, const int8_t *q,
                           const uint16_t *d, float *y, int32_t *isum_opt, int64_t N, int64_t K,
                           int B, void *stream) {
    const lb_q_matrix m = {bits, scales, y, isum_opt, N};
    return gemv_q_grouped<kQ1>(&m, 1, q, d, K, B, stream);
}
