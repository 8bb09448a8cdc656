// lb_common.cuh -- shared host checks and device helpers of the GB300 low-bit library.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "lb.h"

#define LB_EXPORT extern "C" __attribute__((visibility("default")))

namespace lb {

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device checks: compute capability 10.3 (GB300) and its SM count, cached per device.
struct DeviceInfo {
    int sms = 0;
    int ok = -1;  // -1 unknown, 0 refused, 1 sm_103
};

int current_device_info(DeviceInfo *out);  // LB_OK or LB_ERR_ARCH

inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

// Per-kernel launch preparation, cached: raise the dynamic shared-memory limit once and
// remember the occupancy for the last shared-memory size used.  LB_OK, or LB_ERR_SHAPE when
// the requested shared memory cannot be resident, or LB_ERR_LAUNCH.
int prepare_kernel(const void *kernel, int threads, size_t smem, int *blocks_per_sm);

inline int launch_status() {
    cudaError_t e = cudaPeekAtLastError();
    return e == cudaSuccess ? LB_OK : LB_ERR_LAUNCH;
}

// ------------------------------------------------------------------------------------------
// device side
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    // Streamed weights: read once, do not keep in L1.
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// dp4a with unsigned bytes in a and signed bytes in b: sum_i a_i * b_i + c.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ float f16_bits_to_float(uint16_t h) {
    return __half2float(__ushort_as_half(h));
}

// Byte permute: result byte i = byte sel_i of {b, a} (a = bytes 0..3, b = bytes 4..7).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Transpose a 4x4 byte matrix held as 4 words (row i = word i): out word j holds byte j of
// every input word, in input-word order.
__device__ __forceinline__ void transpose4x4(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3,
                                             uint32_t &o0, uint32_t &o1, uint32_t &o2,
                                             uint32_t &o3) {
    uint32_t t01l = prmt(w0, w1, 0x5140);  // w0.b0 w1.b0 w0.b1 w1.b1
    uint32_t t01h = prmt(w0, w1, 0x7362);  // w0.b2 w1.b2 w0.b3 w1.b3
    uint32_t t23l = prmt(w2, w3, 0x5140);
    uint32_t t23h = prmt(w2, w3, 0x7362);
    o0 = prmt(t01l, t23l, 0x5410);  // w0.b0 w1.b0 w2.b0 w3.b0
    o1 = prmt(t01l, t23l, 0x7632);  // w0.b1 w1.b1 w2.b1 w3.b1
    o2 = prmt(t01h, t23h, 0x5410);
    o3 = prmt(t01h, t23h, 0x7632);
}

__device__ __forceinline__ int byte_sum_s8(uint32_t w) { return dp4a_ss(w, 0x01010101u, 0); }

}  // namespace lb
