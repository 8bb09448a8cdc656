// lb_noalloc.cu -- Q2_0_g64 prefill GEMM whose activation scratch is a fixed device array of
// this library instead of caller memory.  The call allocates nothing: the scratch is a
// file-scope __device__ array, located once per device with cudaGetSymbolAddress.
#include "lb_common.cuh"

#include <mutex>

namespace lb {

int gemm_q_with_workspace(int q2, const uint8_t *bits, const uint16_t *scales, const int8_t *q,
                          const uint16_t *d, float *y, int64_t M, int64_t N, int64_t K,
                          void *workspace, size_t workspace_bytes, void *stream);

// Scratch for the converted activation tiles: round_up(M, 128) * K * 2 bytes.  Nothing in it has
// to start at zero -- the GEMM's prologue writes every byte the main kernel reads.
static __device__ __align__(256) uint8_t g_noalloc_scratch[LB_NOALLOC_SCRATCH_BYTES];

static constexpr int kMaxDev = 64;
static void *g_scratch_addr[kMaxDev];
static std::mutex g_scratch_mutex;

// Device address of the scratch on the current device (looked up on the first call per device).
static int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
        cudaGetLastError();
        return LB_ERR_ARCH;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            record_cuda_error(e);
            return LB_ERR_LAUNCH;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return LB_OK;
}

}  // namespace lb

using namespace lb;

LB_EXPORT int lb_gemm_q2_0_g64_noalloc(const uint8_t *codes, const uint16_t *scales,
                                       const int8_t *q, const uint16_t *d, float *y, int64_t M,
                                       int64_t N, int64_t K, void *stream) {
    if (!codes || !scales || !q || !d || !y) return LB_ERR_NULL;
    if (M < 1 || K < 1) return LB_ERR_SHAPE;
    // Refuse before any device work when the converted activations would not fit.
    const int64_t rows = (M + 127) / 128 * 128;
    if (M > (1 << 30) || K > (1 << 24) ||
        (uint64_t)rows * (uint64_t)K * 2u > (uint64_t)LB_NOALLOC_SCRATCH_BYTES)
        return LB_ERR_SHAPE;
    DeviceInfo di;
    if (int st = current_device_info(&di)) return st;
    void *ws = nullptr;
    if (int st = scratch_address(&ws)) return st;
    return gemm_q_with_workspace(1, codes, scales, q, d, y, M, N, K, ws,
                                 (size_t)LB_NOALLOC_SCRATCH_BYTES, stream);
}
