// lb_common.cuh -- shared host checks and device helpers of the GB300 low-bit library.
#pragma once

#include <cuda.h>
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

// Address (device pointer) of the current device's error word: kernels that give up on a
// bounded wait set it; lb_device_status() reads and clears it.
int *device_error_word();

// Per-kernel launch preparation, cached: raise the dynamic shared-memory limit once and
// remember the occupancy for the last shared-memory size used.  LB_OK, LB_ERR_SHAPE when the
// requested shared memory cannot be resident, or LB_ERR_LAUNCH.
int prepare_kernel(const void *kernel, int threads, size_t smem, int *blocks_per_sm);

inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

// Tensor map (TMA descriptor) of a row-major byte matrix [rows][row_bytes] whose copies are
// boxes of box_rows x box_bytes; rows past the end read as zero.  `swizzle_bytes` 0 (none), 32
// or 64: the 16-byte chunks of each box row are XOR-permuted by the hardware's 32 B / 64 B
// pattern.  LB_OK or LB_ERR_LAUNCH.
int encode_rows_map(CUtensorMap *map, const void *base, uint64_t row_bytes, uint64_t rows,
                    uint32_t box_bytes, uint32_t box_rows, int swizzle_bytes = 0);

// Test hook: the wait limit in microseconds set by lb_test_inject_wait_timeout (then cleared),
// or 0.  A streaming GEMV launch that takes a non-zero value makes CTA 0 copy no weights, so
// that CTA's consumers give up after that many microseconds and report through the error word.
int take_injected_wait_fault();

// Remember a failed CUDA call's error for lb_last_cuda_error() (calling thread) and clear it
// from the runtime's last-error slot.
void record_cuda_error(cudaError_t e);

// Launch `kernel` with programmatic stream serialization allowed (see pdl_wait()).
template <typename... KArgs, typename... Args>
inline int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                      cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
    if (e == cudaSuccess) return LB_OK;
    record_cuda_error(e);
    return LB_ERR_LAUNCH;
}

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

// Logic operations as single PTX instructions.  The mask-in-place word dots need one logic
// operation per mask; written in C++ the compiler may distribute a mask over the operation that
// formed its operand (one operation becomes two), which costs the decode loops about 10 %.
template <uint32_t M>
__device__ __forceinline__ uint32_t and_imm(uint32_t a) {
    uint32_t d;
    asm("and.b32 %0, %1, %2;" : "=r"(d) : "r"(a), "n"(M));
    return d;
}
// (a and not m) or (b and m)
template <uint32_t M>
__device__ __forceinline__ uint32_t select_imm(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xD8;" : "=r"(d) : "r"(a), "r"(b), "n"(M));
    return d;
}
// not (a or b)
__device__ __forceinline__ uint32_t nor_u32(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, 0, 0x03;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Per-token int8 quantization of four values: rne(v * s) clamped to [-128, 127], packed
// little-endian (shared by lb_quantize_i8_absmax and its operand-writing variant).
__device__ __forceinline__ uint32_t quantize_i8_word(float4 v, float s) {
    const int c[4] = {__float2int_rn(__fmul_rn(v.x, s)), __float2int_rn(__fmul_rn(v.y, s)),
                      __float2int_rn(__fmul_rn(v.z, s)), __float2int_rn(__fmul_rn(v.w, s))};
    uint32_t w = 0;
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const int t = c[j] > 127 ? 127 : (c[j] < -128 ? -128 : c[j]);
        w |= (uint32_t)(t & 0xFF) << (8 * j);
    }
    return w;
}

// Sums each of V per-lane values over the warp with VP - 1 + 5 - log2(VP) shuffles instead of
// 5 V (VP = V rounded up to a power of two, at most 32).  At the step with lane distance o the
// lanes with bit o set keep the upper half of the values still held, the others the lower half,
// and each adds its partner's copy of the half it keeps; then the one value left is summed over
// the remaining lane bits.  Lane l with l % (32 / VP) == 0 ends with the total of value
// l / (32 / VP), which the return value carries (values >= V are zero).
template <int V>
struct PowTwo {
    static constexpr int value = V <= 1 ? 1 : V <= 2 ? 2 : V <= 4 ? 4 : V <= 8 ? 8 : V <= 16 ? 16 : 32;
    static constexpr int log2 = V <= 1 ? 0 : V <= 2 ? 1 : V <= 4 ? 2 : V <= 8 ? 3 : V <= 16 ? 4 : 5;
};
template <int V, typename T>
__device__ __forceinline__ T warp_sum_many(const T (&in)[V], int lane) {
    static_assert(V >= 1 && V <= 32, "at most 32 values");
    constexpr int VP = PowTwo<V>::value;
    T v[VP];
#pragma unroll
    for (int i = 0; i < VP; i++) v[i] = i < V ? in[i] : T(0);
#pragma unroll
    for (int k = 0; k < PowTwo<V>::log2; k++) {
        const int o = 16 >> k, n = VP >> k;
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; i++) {
            const T send = up ? v[i] : v[i + n / 2];
            const T keep = up ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
#pragma unroll
    for (int o = 16 >> PowTwo<V>::log2; o > 0; o >>= 1)
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
    return v[0];
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

// Programmatic dependent launch.  Every kernel of the library is launched so that the next
// kernel in the stream may start once all of its CTAs have called pdl_launch_dependents(); each
// kernel calls pdl_wait() -- which returns when the previous kernel in the stream has completed
// and its memory is visible -- before it reads or writes any buffer another kernel may touch.
// Only reads of weights happen before pdl_wait().  The one kernel of the library that writes
// weights (the load-time repack) never triggers early, so a kernel launched after it starts
// only once it has completed; kernels of other libraries (torch, copies) never trigger early
// either.  Without a programmatic predecessor both instructions are no-ops.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------------------------------------
// mbarrier + bulk-copy (TMA, non-tensor) primitives, CTA scope.
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(
                     smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Bounded wait on the phase with the given parity: true once it completes, false after about
// `limit_ns` (the caller then reports through the error word and stops instead of hanging).
// The first test is inline; the timed loop is a separate function so that the common case (the
// phase has already completed) costs one try_wait and a branch.
// try_wait that lets the hardware suspend the thread for up to `hint_ns` while the phase is
// incomplete (it resumes as soon as the phase completes), so waiting warps do not take issue
// slots from working ones.
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t *bar, uint32_t parity,
                                                   uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
__device__ __noinline__ static bool mbar_wait_slow(uint64_t *bar, uint32_t parity,
                                                   uint64_t limit_ns) {
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; i++) {
        if (mbar_try_wait_hint(bar, parity, 1000u)) return true;
        if ((i & 15u) == 0 && global_ns() - t0 > limit_ns) return false;
    }
}
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          uint64_t limit_ns = 2000000000ull) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, limit_ns);
}
// 2-D tensor copy (box at column byte x, row y) global -> this CTA's shared memory, counted on
// `bar`.  x must be a multiple of 16.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
        "{%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
// Bulk copy global -> this CTA's shared memory; completion is counted on `bar` (tx bytes).
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
        "[%3];" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// Named barrier over `count` threads (id 0 is __syncthreads).
__device__ __forceinline__ void named_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace lb
