// lb_probe.cu -- instruction-rate probes for the roofline denominators of the prefill GEMMs
// (a measurement library beside liblb.so, loaded by the bench only).
//
// The exact GEMMs run on kind::f16 tensor-core MMAs because the integer kinds are not available
// on this architecture; these probes measure, on the GPU the bench runs on, the dense rates of
// the candidate instruction forms so that the choice and the denominator rest on a measurement:
//   0  tcgen05.mma kind::f16     M128 N256 K16, f16 x f16 -> f32 (tensor memory)
//   1  tcgen05.mma kind::f8f6f4  M128 N256 K32, e4m3 x e4m3 -> f32
//   2  mma.sync m16n8k16 f16 x f16 -> f32 (registers; the legacy warp-level path)
//   3  mma.sync m16n8k32 s8 x s8 -> s32
// Each runs one CTA per SM with its operands resident in shared memory or registers (zeros),
// issuing back-to-back MMAs, and reports dense FLOP/s (2 M N K per MMA) over the whole GPU.
#include <cuda_runtime.h>

#include "lb_tc.cuh"

namespace lbp {

using namespace lb;

constexpr int kTcReps = 16384;   // MMAs per CTA (tcgen05)
constexpr int kSyncReps = 8192;  // loop trips per warp (mma.sync, 4 independent MMAs each)
constexpr int kSyncWarps = 16;

// One thread issues kTcReps MMAs into one 256-column accumulator, then waits for them.
template <bool kF8>
__global__ void __launch_bounds__(128, 1) tc_rate_kernel(int *err) {
    __shared__ __align__(1024) uint8_t ops[16384 + 8192];
    __shared__ __align__(8) uint64_t done;
    __shared__ uint32_t slot;
    for (int i = threadIdx.x; i < (int)sizeof(ops) / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(ops)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        mbar_init(&done, 1);
        fence_mbar_init();
    }
    if (threadIdx.x < 32) tmem_alloc(&slot, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = slot;
    if (threadIdx.x == 0) {
        const uint32_t a = smem_u32(ops), b = a + 8192;
        if (kF8) {
            constexpr uint32_t idesc = (1u << 4) | ((256u >> 3) << 17) | ((128u >> 4) << 24);
            const uint64_t ad = smem_desc8(a), bd = smem_desc8(b);
            for (int i = 0; i < kTcReps; i++) mma_f8(tmem, ad, bd, idesc);
        } else {
            constexpr uint32_t idesc = idesc_f16(128, 256);
            const uint64_t ad = smem_desc(a), bd = smem_desc(b);
            for (int i = 0; i < kTcReps; i++) mma_f16(tmem, ad, bd, idesc, i ? 1u : 0u);
        }
        mma_commit(&done);
        if (!mbar_wait(&done, 0) && err) atomicOr(err, 1);
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// Each warp keeps four independent accumulators in registers.
template <bool kS8>
__global__ void __launch_bounds__(kSyncWarps * 32, 1) sync_rate_kernel(float *sink) {
    const uint32_t a0 = threadIdx.x & 1, a1 = 0, a2 = 0, a3 = 0, b0 = 0, b1 = 0;
    float f[4][4] = {};
    int s[4][4] = {};
    for (int i = 0; i < kSyncReps; i++) {
#pragma unroll
        for (int j = 0; j < 4; j++) {
            if (kS8)
                asm volatile(
                    "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, "
                    "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                    : "+r"(s[j][0]), "+r"(s[j][1]), "+r"(s[j][2]), "+r"(s[j][3])
                    : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
            else
                asm volatile(
                    "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, "
                    "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                    : "+f"(f[j][0]), "+f"(f[j][1]), "+f"(f[j][2]), "+f"(f[j][3])
                    : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
        }
    }
    float t = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; j++)
#pragma unroll
        for (int e = 0; e < 4; e++) t += f[j][e] + (float)s[j][e];
    if (t != 0.0f) sink[threadIdx.x] = t;  // zeros in, zeros out: never written
}

}  // namespace lbp

using namespace lbp;

// Measures the four rates on the current device; rates[i] receives dense FLOP/s of probe i (in
// the order of the header), or 0 if it could not run.  Returns 0, or -6 on a launch error, -7
// if a tensor-core wait ran out.  Synchronizes the device.
extern "C" __attribute__((visibility("default"))) int lbp_tensor_rates(double *rates) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -6;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return -6;
    int *err = nullptr;
    float *sink = nullptr;
    if (cudaMalloc(&err, sizeof(int)) != cudaSuccess) return -6;
    if (cudaMalloc(&sink, kSyncWarps * 32 * sizeof(float)) != cudaSuccess) {
        cudaFree(err);
        return -6;
    }
    cudaMemset(err, 0, sizeof(int));
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    int status = 0;
    for (int k = 0; k < 4; k++) {
        double flop = 0.0;
        float best = 0.0f;
        for (int rep = 0; rep < 3; rep++) {  // best of three (the first also warms up)
            cudaEventRecord(e0);
            if (k == 0) {
                tc_rate_kernel<false><<<sms, 128>>>(err);
                flop = 2.0 * 128 * 256 * 16 * (double)kTcReps * sms;
            } else if (k == 1) {
                tc_rate_kernel<true><<<sms, 128>>>(err);
                flop = 2.0 * 128 * 256 * 32 * (double)kTcReps * sms;
            } else if (k == 2) {
                sync_rate_kernel<false><<<sms, kSyncWarps * 32>>>(sink);
                flop = 2.0 * 16 * 8 * 16 * 4.0 * kSyncReps * kSyncWarps * sms;
            } else {
                sync_rate_kernel<true><<<sms, kSyncWarps * 32>>>(sink);
                flop = 2.0 * 16 * 8 * 32 * 4.0 * kSyncReps * kSyncWarps * sms;
            }
            cudaEventRecord(e1);
            if (cudaEventSynchronize(e1) != cudaSuccess || cudaGetLastError() != cudaSuccess) {
                status = -6;
                break;
            }
            float ms = 0.0f;
            cudaEventElapsedTime(&ms, e0, e1);
            if (rep == 0 || ms < best) best = ms;
        }
        rates[k] = (status == 0 && best > 0.0f) ? flop / (best * 1e-3) : 0.0;
        if (status) break;
    }
    int h = 0;
    cudaMemcpy(&h, err, sizeof(int), cudaMemcpyDeviceToHost);
    if (h && !status) status = -7;
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    cudaFree(err);
    cudaFree(sink);
    return status;
}
