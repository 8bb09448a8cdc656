// lb_tc.cuh -- 5th-generation tensor core (tcgen05) helpers: tensor-memory allocation, MMA
// issue, commit, tensor-memory loads, and the shared-memory / instruction descriptors.
//
// Operand layout used throughout: K-major, no swizzle.  A [rows][32] f16 tile is stored as core
// matrices of 8 rows x 16 bytes (8 f16 of K):
//     byte offset(r, k) = (r / 8) * 512 + (k / 8) * 128 + (r % 8) * 16 + (k % 8) * 2
// i.e. leading-dimension byte offset (between K-adjacent core matrices) 128 and stride byte
// offset (between 8-row groups) 512; one 16-deep MMA step reads two K-adjacent core matrices,
// the second step starts 256 bytes further.
#pragma once
#include "lb_common.cuh"

namespace lb {

constexpr int kCoreLBO = 128;
constexpr int kCoreSBO = 512;

__device__ __forceinline__ int canon_offset(int r, int k) {
    return (r >> 3) * kCoreSBO + (k >> 3) * kCoreLBO + (r & 7) * 16 + (k & 7) * 2;
}

// Eight f16 of K for one row of an activation operand tile from two words of int8 codes x, y:
// x0 y0 x1 y1 x2 y2 x3 y3 (f16x2 number i pairs byte i of x with byte i of y).  Exact: each code
// is biased by +128 into the mantissa of 1024 (exponent byte 0x64) and 1152 is subtracted.
__device__ __forceinline__ uint4 int8_pair_f16(uint32_t x, uint32_t y) {
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    const uint32_t lo = prmt(x, y, 0x5140) ^ 0x80808080u;  // x0 y0 x1 y1, biased +128
    const uint32_t hi = prmt(x, y, 0x7362) ^ 0x80808080u;  // x2 y2 x3 y3
    uint32_t h[4] = {prmt(lo, 0x64646464u, 0x5140), prmt(lo, 0x64646464u, 0x7362),
                     prmt(hi, 0x64646464u, 0x5140), prmt(hi, 0x64646464u, 0x7362)};
#pragma unroll
    for (int e = 0; e < 4; e++) {
        __half2 v = __hsub2(*reinterpret_cast<__half2 *>(&h[e]), bias);
        h[e] = *reinterpret_cast<uint32_t *>(&v);
    }
    return make_uint4(h[0], h[1], h[2], h[3]);
}

// Shared-memory matrix descriptor: start address, LBO, SBO (all >> 4), version 1, no swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((kCoreLBO >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((kCoreSBO >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// Shared-memory matrix descriptor for 8-bit operands whose rows are 32 bytes (one 32-deep
// block): K-adjacent core matrices 128 B apart, 8-row groups 256 B apart.
__device__ __forceinline__ uint64_t smem_desc8(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)(128 >> 4) << 16;
    d |= (uint64_t)(256 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// Instruction descriptor, kind::f16: D f32, A and B f16, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Bulk copy this CTA's shared memory -> global, in the issuing thread's bulk group.  dst, src
// and bytes must be multiples of 16; the source must be written before a proxy fence.
__device__ __forceinline__ void bulk_s2g(void *dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_u32(src)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until this thread's bulk groups have read their shared-memory sources ...
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// ... or have completed their writes.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// D[tmem] (+)= A[desc] * B[desc]^T, cta_group::1, kind::f16.
__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] = A[desc] * B[desc]^T, cta_group::1, kind::f8f6f4 (formats in the instruction
// descriptor), D overwritten.
__device__ __forceinline__ void mma_f8(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, 0, 0; "
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p; }" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc)
        : "memory");
}

// Arrive once on `bar` when every MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}
// 32 consecutive columns of the calling warp's 32 lanes (lane quarter = warp id % 4).  The load
// and its completion wait are one asm statement, so no use of r can be scheduled before the
// data has arrived.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// The same load, returned as 16 pairs of columns (2c, 2c + 1) in 64-bit registers (column 2c in
// the low half), ready for paired f32x2 arithmetic without register moves.
__device__ __forceinline__ void tmem_ld32_pairs(uint32_t taddr, uint64_t (&p)[16]) {
    asm volatile(
        "{ .reg .b32 r<32>;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {r0,r1,r2,r3,r4,r5,r6,r7,r8,r9,r10,r11,r12,r13,"
        "r14,r15,r16,r17,r18,r19,r20,r21,r22,r23,r24,r25,r26,r27,r28,r29,r30,r31}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t"
        "mov.b64 %0, {r0, r1}; mov.b64 %1, {r2, r3}; mov.b64 %2, {r4, r5};\n\t"
        "mov.b64 %3, {r6, r7}; mov.b64 %4, {r8, r9}; mov.b64 %5, {r10, r11};\n\t"
        "mov.b64 %6, {r12, r13}; mov.b64 %7, {r14, r15}; mov.b64 %8, {r16, r17};\n\t"
        "mov.b64 %9, {r18, r19}; mov.b64 %10, {r20, r21}; mov.b64 %11, {r22, r23};\n\t"
        "mov.b64 %12, {r24, r25}; mov.b64 %13, {r26, r27}; mov.b64 %14, {r28, r29};\n\t"
        "mov.b64 %15, {r30, r31}; }"
        : "=l"(p[0]), "=l"(p[1]), "=l"(p[2]), "=l"(p[3]), "=l"(p[4]), "=l"(p[5]), "=l"(p[6]),
          "=l"(p[7]), "=l"(p[8]), "=l"(p[9]), "=l"(p[10]), "=l"(p[11]), "=l"(p[12]),
          "=l"(p[13]), "=l"(p[14]), "=l"(p[15])
        : "r"(taddr)
        : "memory");
}

// Half of that load: 16 consecutive columns as 8 pairs.
__device__ __forceinline__ void tmem_ld16_pairs(uint32_t taddr, uint64_t (&p)[8]) {
    asm volatile(
        "{ .reg .b32 r<16>;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {r0,r1,r2,r3,r4,r5,r6,r7,r8,r9,r10,r11,r12,r13,"
        "r14,r15}, [%8];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t"
        "mov.b64 %0, {r0, r1}; mov.b64 %1, {r2, r3}; mov.b64 %2, {r4, r5};\n\t"
        "mov.b64 %3, {r6, r7}; mov.b64 %4, {r8, r9}; mov.b64 %5, {r10, r11};\n\t"
        "mov.b64 %6, {r12, r13}; mov.b64 %7, {r14, r15}; }"
        : "=l"(p[0]), "=l"(p[1]), "=l"(p[2]), "=l"(p[3]), "=l"(p[4]), "=l"(p[5]), "=l"(p[6]),
          "=l"(p[7])
        : "r"(taddr)
        : "memory");
}

// acc += a * {s, s} on pairs of binary32 (element 0 in the low half), each element rounded once
// as by fmaf.
__device__ __forceinline__ void ffma2p(uint64_t &acc, uint64_t a, uint64_t s2) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(s2));
}

// acc (two binary32 in one 64-bit register, element 0 in the low half) += {a0, a1} * {s, s},
// each element rounded once as by fmaf.
__device__ __forceinline__ void ffma2(uint64_t &acc, uint32_t a0, uint32_t a1, uint64_t s2) {
    asm("{ .reg .b64 t; mov.b64 t, {%1, %2}; fma.rn.f32x2 %0, t, %3, %0; }"
        : "+l"(acc)
        : "r"(a0), "r"(a1), "l"(s2));
}

}  // namespace lb
