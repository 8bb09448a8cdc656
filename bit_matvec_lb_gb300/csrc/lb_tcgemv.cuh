// lb_tcgemv.cuh -- batched decode GEMV (3 to 8 tokens) on the 5th-generation tensor cores, for
// Q1_0, Q2_0_g64 and planar ternary weights.  Same arithmetic as lb_stream.cuh (integer block
// sums, then the fp16/fp32 scales), computed exactly with fp8 operands:
//   * weights: every weight is -1, 0, +1 or +2, exact in e4m3;
//   * activations: an int8 code q is split as q = 16 * hi + lo with hi in [-8, 7] and lo in
//     [0, 15], both exact in e4m3.  The eight tokens' hi parts and lo parts are the 16 columns of
//     the MMA's N dimension, so one 128 x 16 x 32 MMA per q8_0 block gives, per weight row and
//     token, S_hi and S_lo with |S| <= 32 * 2 * 15 (exact in fp32), and isum = 16 S_hi + S_lo is
//     exact too.
//   * The scales are applied as in the streaming GEMV: t = sum over the weight block of
//     d_x * isum, then acc = fma(d_w, t, acc) (planar: the integer sum -- accumulated in binary32,
//     exact below 2^24 -- then the two multiplies).
// Why: at 8 tokens the dp4a formulation costs about four instructions per weight and cannot keep
// up with HBM; here a weight costs about half an instruction to decode and the products run on
// the tensor cores.
//
// CTA (persistent, one per SM) = 16 warps working on units of 128 weight rows x all of K, in
// steps of 8 q8_0 blocks (256 columns).  The activation operand (hi/lo e4m3 tiles of all of K,
// 16 K bytes) and the activation scales as binary32 are built once per CTA by warps 1-15 and
// stay resident; then:
//   warp 0      producer: one 2-D tensor copy of 128 rows x one step of packed weights per step
//               into a 4-stage ring;
//   warps 1-3   issue the MMAs of every third step (one thread each); warp 2 owns tensor memory;
//   warps 4-11  weight decoders: thread = (row, half of the step); packed word -> e4m3 bytes by
//               a byte lookup (prmt) -> operand tiles (K-major core matrices, no swizzle);
//   warps 12-15 drain: thread = row = accumulator lane; tcgen05.ld, scales, outputs.
// Four 128-column accumulators (8 blocks x 16 columns) let the MMAs run ahead of the drain.
// Every wait is bounded and reports through the device error word.
#pragma once
#include "lb_stream.cuh"
#include "lb_tc.cuh"

namespace lb {

constexpr int kTgThreads = 512;
constexpr int kTgRows = 128;                    // rows per unit (accumulator lanes)
constexpr int kTgBlocks = 8;                    // q8_0 blocks per step
constexpr int kTgCols = kTgBlocks * 32;         // columns per step
constexpr int kTgAStages = 3;                   // weight operand stages
constexpr int kTgPStages = 4;                   // packed-weight stages
constexpr int kTgMaxK = 4096;                   // K up to which the activation operand is resident
constexpr int kTgAccBufs = 4;                   // 128-column accumulators
constexpr int kTgIssuers = 3;                   // MMA-issuing warps (1-3)
// An issuer waits on the operand stage and accumulator of its own step; with fewer stages or
// accumulators than issuers, two issuers would wait on phases of one barrier two apart, which a
// parity wait cannot tell apart.
static_assert(kTgAStages >= kTgIssuers && kTgAccBufs >= kTgIssuers, "stages per issuer");
constexpr uint64_t kSixteen2 = 0x4180000041800000ull;  // {16.0f, 16.0f}
constexpr uint64_t kOne2 = 0x3F8000003F800000ull;      // {1.0f, 1.0f}
constexpr int kTgWTile = kTgRows * 32;          // one block's weight operand, e4m3: 4 KB
constexpr int kTgXTile = 16 * 32;               // one block's activation operand: 512 B
constexpr int kTgWStage = kTgBlocks * kTgWTile; // 32 KB
constexpr int kTgXStage = kTgBlocks * kTgXTile; // 4 KB

// Packed bytes of one row for one step, and the row pitch in the packed stage (dense: one
// tensor copy per step lands the 128 rows back to back, with the hardware swizzle of a row's
// size, 64 B or 32 B, so the decoders' 16-byte reads of 32 consecutive rows do not conflict).
template <int F> struct TgFmt;
template <> struct TgFmt<kQ1> { static constexpr int kBytes = kTgCols / 8; static constexpr int kPitch = kBytes; };
template <> struct TgFmt<kQ2> { static constexpr int kBytes = kTgCols / 4; static constexpr int kPitch = kBytes; };
template <> struct TgFmt<kTrit> { static constexpr int kBytes = kTgCols / 4; static constexpr int kPitch = kBytes; };

// One tensor map per matrix of the group: the packed weight plane as [N][row bytes], copied in
// boxes of 128 rows x one step.
struct TgMaps {
    CUtensorMap m[kMaxGroup];
};

template <int F>
constexpr int tg_smem_bytes() {
    return kTgAStages * kTgWStage + kTgPStages * kTgRows * TgFmt<F>::kPitch +
           (kTgMaxK / 32) * kTgXTile + (kTgMaxK / 32) * 8 * 4 + 512 + 1024;
}

// Column permutation inside a 32-column block shared by the weight decode and the activation
// builder: operand column p holds weight / activation column tg_col<F>(p) of the block.
template <int F>
__host__ __device__ constexpr int tg_col(int p) {
    // Q2_0_g64: byte lookups of (w >> 2s) & 0x33333333 give columns (2i + s) and (8 + 2i + s);
    // Q1_0 / planar: lookups of (w >> s) & 0x11111111 give columns (4i + s) and (16 + 4i + s).
    return F == kQ2 ? 16 * (p >> 4) + 8 * ((p >> 2) & 1) + 2 * (p & 3) + ((p >> 3) & 1)
                    : 16 * (p >> 4) + 4 * (p & 3) + ((p >> 2) & 3);
}

// Offset of byte (row r, column kb) in a K-major, no-swizzle operand tile of 32 bytes per row
// (core matrices of 8 rows x 16 bytes; K-adjacent ones 128 B apart, 8-row groups 256 B apart).
__device__ __forceinline__ int tg_off(int r, int kb) {
    return (r >> 3) * 256 + (kb >> 4) * 128 + (r & 7) * 16 + (kb & 15);
}

// e4m3 byte pair of two small integers (|v| <= 16 is exact): lo in bits 0-7, hi in 8-15.
__device__ __forceinline__ uint32_t e4m3x2(int lo, int hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"((float)hi), "f"((float)lo));
    return r;
}

// Weight decode of one 32-column block into its two 16-byte operand chunks (columns 0-15 and
// 16-31 of the permuted order).
__device__ __forceinline__ void tg_decode_q2(uint32_t w0, uint32_t w1, uint4 &c0, uint4 &c1) {
    constexpr uint32_t T = 0x403800B8u;  // code 0..3 -> e4m3 of -1, 0, +1, +2
    const uint32_t x0 = w0 & 0x33333333u, y0 = (w0 >> 2) & 0x33333333u;
    const uint32_t x1 = w1 & 0x33333333u, y1 = (w1 >> 2) & 0x33333333u;
    c0 = make_uint4(prmt(T, 0, x0), prmt(T, 0, x0 >> 16), prmt(T, 0, y0), prmt(T, 0, y0 >> 16));
    c1 = make_uint4(prmt(T, 0, x1), prmt(T, 0, x1 >> 16), prmt(T, 0, y1), prmt(T, 0, y1 >> 16));
}
__device__ __forceinline__ void tg_decode_q1(uint32_t w, uint4 &c0, uint4 &c1) {
    constexpr uint32_t T = 0x000038B8u;  // bit 0 -> -1, bit 1 -> +1
    uint32_t lo[4], hi[4];
#pragma unroll
    for (int s = 0; s < 4; s++) {
        const uint32_t x = (w >> s) & 0x11111111u;
        lo[s] = prmt(T, 0, x);
        hi[s] = prmt(T, 0, x >> 16);
    }
    c0 = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    c1 = make_uint4(hi[0], hi[1], hi[2], hi[3]);
}
__device__ __forceinline__ void tg_decode_trit(uint32_t pos, uint32_t neg, uint4 &c0, uint4 &c1) {
    constexpr uint32_t T = 0x00B83800u;  // index pos + 2 neg: 0 -> 0, 1 -> +1, 2 -> -1
    uint32_t lo[4], hi[4];
#pragma unroll
    for (int s = 0; s < 4; s++) {
        const uint32_t x = ((pos >> s) & 0x11111111u) | (((neg >> s) & 0x11111111u) << 1);
        lo[s] = prmt(T, 0, x);
        hi[s] = prmt(T, 0, x >> 16);
    }
    c0 = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    c1 = make_uint4(hi[0], hi[1], hi[2], hi[3]);
}

__device__ __forceinline__ bool wait_or_report_tg(uint64_t *bar, uint32_t parity, int *err) {
    if (mbar_wait(bar, parity)) return true;
    report(err);
    return false;
}

template <int F, int B>
__global__ void __launch_bounds__(kTgThreads, 1)
    tc_gemv_kernel(const __grid_constant__ StreamParams p, const __grid_constant__ TgMaps maps) {
    constexpr int kPB = TgFmt<F>::kBytes, kPP = TgFmt<F>::kPitch;
    constexpr int kBlkPerW = F == kQ1 ? 4 : 2;          // q8_0 blocks per weight block (Q)
    extern __shared__ uint8_t tg_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(tg_raw) + 1023) &
                                              ~(uintptr_t)1023);
    uint8_t *wst = sm;                                            // weight operand stages
    uint8_t *pst = wst + kTgAStages * kTgWStage;                  // packed weight stages
    uint8_t *xop = pst + kTgPStages * kTgRows * kPP;              // activation operand, all K
    // activation scales d_x as binary32, [q8_0 block][token] (tokens past B unused)
    float *dxf = reinterpret_cast<float *>(xop + (kTgMaxK / 32) * kTgXTile);
    uint16_t *lut = reinterpret_cast<uint16_t *>(dxf + (kTgMaxK / 32) * 8);  // q -> e4m3 hi, lo
    __shared__ __align__(8) uint64_t pk_full[kTgPStages], pk_empty[kTgPStages], a_full[kTgAStages],
        a_empty[kTgAStages], t_full[kTgAccBufs], t_empty[kTgAccBufs], mma_done;
    __shared__ uint32_t tmem_slot;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nsteps = (int)(p.K / kTgCols);
    const int nq8 = (int)(p.K / 32);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kTgPStages; s++) {
            mbar_init(&pk_full[s], 1);
            mbar_init(&pk_empty[s], 8);
        }
        for (int s = 0; s < kTgAStages; s++) {
            mbar_init(&a_full[s], 8);  // eight decoder warps
            mbar_init(&a_empty[s], 1);
        }
        for (int b = 0; b < kTgAccBufs; b++) {
            mbar_init(&t_full[b], 1);
            mbar_init(&t_empty[b], 4);
        }
        mbar_init(&mma_done, kTgIssuers);
        fence_mbar_init();
    }
    // byte lookup: int8 code -> {e4m3(code >> 4), e4m3(code & 15)}
    if (threadIdx.x < 256) {
        const int v = (int)(int8_t)(uint8_t)threadIdx.x;
        lut[threadIdx.x] = (uint16_t)(e4m3x2(v >> 4, 0) | (e4m3x2(v & 15, 0) << 8));
    }
    if (warp == 2) tmem_alloc(&tmem_slot, kTgAccBufs * 128);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    pdl_launch_dependents();

    if (warp != 0) {
        // ---------------- activation operand, built once for all of K (warps 1-11) ----------------
        // Tile j (512 B) holds q8_0 block j as 16 rows: hi parts of tokens 0..7, then lo parts,
        // absent tokens zero; columns in the weight decode's order.  The weights of the first
        // steps stream in meanwhile (the producer does not wait for the activations).
        pdl_wait();
        const int items = nq8 * 8 * 2;  // (block, token, half)
        for (int it = threadIdx.x - 32; it < items; it += kTgThreads - 32) {
            const int h = it & 1, b = (it >> 1) & 7, j = it >> 4;
            uint32_t hw[4] = {0, 0, 0, 0}, lw[4] = {0, 0, 0, 0};
            if (b < B) {
                const uint4 qv = *reinterpret_cast<const uint4 *>(p.q + (int64_t)b * p.K + j * 32 + 16 * h);
                const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
                auto enc = [&](int c) { return (uint32_t)lut[(qw[c >> 2] >> (8 * (c & 3))) & 0xFF]; };
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    // operand columns 16h + 4i .. +3 hold block columns tg_col(...) - 16h
                    const int p0 = 16 * h + 4 * i;
                    const uint32_t e01 = enc(tg_col<F>(p0) - 16 * h) | (enc(tg_col<F>(p0 + 1) - 16 * h) << 16);
                    const uint32_t e23 = enc(tg_col<F>(p0 + 2) - 16 * h) | (enc(tg_col<F>(p0 + 3) - 16 * h) << 16);
                    hw[i] = prmt(e01, e23, 0x6420);
                    lw[i] = prmt(e01, e23, 0x7531);
                }
            }
            if (F != kTrit && h == 0)
                dxf[j * 8 + b] = b < B ? f16_bits_to_float(p.d[(int64_t)b * nq8 + j]) : 0.0f;
            uint8_t *tile = xop + j * kTgXTile;
            *reinterpret_cast<uint4 *>(tile + tg_off(b, 16 * h)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4 *>(tile + tg_off(8 + b, 16 * h)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        fence_proxy_async_smem();
        named_sync(1, kTgThreads - 32);
    }

    if (warp == 0) {
        // ---------------- producer: packed weights, one tensor copy per step ----------------
        int pi = 0;
        uint32_t ph = 0;
        int issued = 0;
        bool ok = true;
        int mi = 0;
        if (lane == 0) {
            for (int u = blockIdx.x; u < p.nunits && ok; u += gridDim.x) {
                mi = find_mat(p, u, mi);
                const StreamMat &M = p.m[mi];
                const int row0 = (u - M.unit0) * kTgRows;
                for (int s = 0; s < nsteps; s++) {
                    if (!mbar_wait(&pk_empty[pi], ph ^ 1)) {
                        ok = false;
                        break;
                    }
                    // the box always holds 128 rows (rows past N read as zero)
                    mbar_arrive_expect_tx(&pk_full[pi], (uint32_t)(kTgRows * kPB));
                    tma_load_2d(pst + pi * kTgRows * kPP, &maps.m[mi], s * kPB, row0, &pk_full[pi]);
                    issued++;
                    if (++pi == kTgPStages) {
                        pi = 0;
                        ph ^= 1;
                    }
                }
            }
        }
        if (!ok && lane == 0) report(p.err);
        for (int i = max(0, issued - kTgPStages); i < issued; i++)
            mbar_wait(&pk_full[i % kTgPStages], (uint32_t)((i / kTgPStages) & 1));

    } else if (warp >= 1 && warp <= kTgIssuers) {
        // ---------------- MMA issue: warp 1 + i issues the steps g = i (mod 3) ----------------
        // (one thread each)
        if (lane == 0) {
            constexpr uint32_t idesc = (1u << 4) | ((16u >> 3) << 17) | ((128u >> 4) << 24);
            const int total = p.nunits <= (int)blockIdx.x
                                  ? 0
                                  : ((p.nunits - 1 - (int)blockIdx.x) / (int)gridDim.x + 1) * nsteps;
            const uint32_t wbase = smem_u32(wst), xbase = smem_u32(xop);
            for (int g = warp - 1; g < total; g += kTgIssuers) {
                const int ai = g % kTgAStages, tb = g % kTgAccBufs;
                if (!wait_or_report_tg(&a_full[ai], (uint32_t)((g / kTgAStages) & 1), p.err)) break;
                if (!wait_or_report_tg(&t_empty[tb], (uint32_t)(((g / kTgAccBufs) & 1) ^ 1), p.err))
                    break;
                tc_fence_after();
                // descriptors of the step's first block; the others follow by adding the tile
                // offsets to the start-address field (smem addresses stay below 2^18, so the
                // 14-bit field of addr >> 4 cannot carry into the next field)
                const uint64_t ad0 = smem_desc8(wbase + ai * kTgWStage);
                const uint64_t bd0 = smem_desc8(xbase + (g % nsteps) * kTgBlocks * kTgXTile);
                const uint32_t d0 = tmem + (uint32_t)(tb * 128);
#pragma unroll
                for (int jb = 0; jb < kTgBlocks; jb++)
                    mma_f8(d0 + (uint32_t)(jb * 16), ad0 + (uint64_t)((jb * kTgWTile) >> 4),
                           bd0 + (uint64_t)((jb * kTgXTile) >> 4), idesc);
                mma_commit(&a_empty[ai]);
                mma_commit(&t_full[tb]);
            }
            mma_commit(&mma_done);
            wait_or_report_tg(&mma_done, 0, p.err);
        }
    } else if (warp >= 4 && warp < 12) {
        // ---------------- weight decoders: thread = (row, half of the step's blocks) ----------------
        const int r = (threadIdx.x - 128) & (kTgRows - 1);
        const int hh = (threadIdx.x - 128) >> 7;  // warps 4-7: blocks 0-3, warps 8-11: blocks 4-7
        int pi = 0, ai = 0;
        uint32_t pph = 0, aph = 0;
        bool ok = true;
        const int total = p.nunits <= (int)blockIdx.x
                              ? 0
                              : ((p.nunits - 1 - (int)blockIdx.x) / (int)gridDim.x + 1) * nsteps;
        const int woff = (r >> 3) * 256 + (r & 7) * 16;
        for (int g = 0; g < total && ok; g++) {
            if (!__all_sync(0xffffffffu, mbar_wait(&pk_full[pi], pph)) ||
                !__all_sync(0xffffffffu, mbar_wait(&a_empty[ai], aph ^ 1))) {
                if (lane == 0) report(p.err);
                ok = false;
                break;
            }
            const uint4 *src = reinterpret_cast<const uint4 *>(pst + pi * kTgRows * kPP + r * kPP);
            // 16-byte chunk v of this row sits at chunk v ^ sw (the swizzle of the tensor copy)
            const int sw = kPB == 64 ? ((r >> 1) & 3) : ((r >> 2) & 1);
            uint8_t *dst = wst + ai * kTgWStage + woff;
            if (F == kQ1) {
#pragma unroll
                for (int vv = 0; vv < kPB / 32; vv++) {
                    const int v = hh * (kPB / 32) + vv;
                    const uint4 c = src[v ^ sw];
                    const uint32_t ws[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
                    for (int t = 0; t < 4; t++) {
                        uint4 c0, c1;
                        tg_decode_q1(ws[t], c0, c1);
                        uint8_t *tile = dst + (4 * v + t) * kTgWTile;
                        *reinterpret_cast<uint4 *>(tile) = c0;
                        *reinterpret_cast<uint4 *>(tile + 128) = c1;
                    }
                }
            } else {
#pragma unroll
                for (int vv = 0; vv < kPB / 32; vv++) {
                    const int v = hh * (kPB / 32) + vv;
                    const uint4 c = src[v ^ sw];  // Q2: blocks 2v, 2v+1; planar: one 64-column beat
                    uint4 c0, c1;
                    if (F == kQ2) {
                        tg_decode_q2(c.x, c.y, c0, c1);
                        *reinterpret_cast<uint4 *>(dst + (2 * v) * kTgWTile) = c0;
                        *reinterpret_cast<uint4 *>(dst + (2 * v) * kTgWTile + 128) = c1;
                        tg_decode_q2(c.z, c.w, c0, c1);
                        *reinterpret_cast<uint4 *>(dst + (2 * v + 1) * kTgWTile) = c0;
                        *reinterpret_cast<uint4 *>(dst + (2 * v + 1) * kTgWTile + 128) = c1;
                    } else {
                        tg_decode_trit(c.x, c.z, c0, c1);  // columns 0-31: pos lo, neg lo
                        *reinterpret_cast<uint4 *>(dst + (2 * v) * kTgWTile) = c0;
                        *reinterpret_cast<uint4 *>(dst + (2 * v) * kTgWTile + 128) = c1;
                        tg_decode_trit(c.y, c.w, c0, c1);  // columns 32-63: pos hi, neg hi
                        *reinterpret_cast<uint4 *>(dst + (2 * v + 1) * kTgWTile) = c0;
                        *reinterpret_cast<uint4 *>(dst + (2 * v + 1) * kTgWTile + 128) = c1;
                    }
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&a_full[ai]);
                mbar_arrive(&pk_empty[pi]);
            }
            if (++pi == kTgPStages) {
                pi = 0;
                pph ^= 1;
            }
            if (++ai == kTgAStages) {
                ai = 0;
                aph ^= 1;
            }
        }
    } else if (warp >= 12) {
        // ---------------- drain: thread = row = accumulator lane ----------------
        // d_x comes from the shared table built in the prologue; d_w (the lane's row) from
        // global memory, two steps ahead of its use.
        const int r = threadIdx.x - 384;
        const int lq = warp & 3;
        int tb = 0;
        uint32_t tph = 0;
        bool ok = true;
        int mi = 0;
        for (int u = blockIdx.x; u < p.nunits && ok; u += gridDim.x) {
            mi = find_mat(p, u, mi);
            const StreamMat &M = p.m[mi];
            const int row0 = (u - M.unit0) * kTgRows;
            const bool rv = r < M.N - row0;
            const int64_t row = row0 + (rv ? r : 0);
            // Planar sums accumulate in binary32 too: every partial is an integer below
            // 128 * K < 2^24, so they are exact and the final integer conversion is too.
            typedef float Acc;
            // 5+ tokens: two tokens per f32x2 instruction (the scalar form, with fewer live
            // registers, is faster at 3-4 tokens, where the paired form spills)
            constexpr bool kPairs = B >= 5;
            constexpr int NP = (B + 1) / 2;  // token pairs
            Acc acc[B];
            float tq[B];
            uint64_t acc2[NP], tq2[NP];      // binary32 pairs: token 2k low, 2k + 1 high
#pragma unroll
            for (int b = 0; b < B; b++) {
                acc[b] = 0;
                tq[b] = 0.0f;
            }
#pragma unroll
            for (int k = 0; k < NP; k++) acc2[k] = tq2[k] = 0;
            // Weight scales two steps ahead in two fixed register slots (the loop is unrolled by
            // two so that no register move waits for the newest load; they come from HBM).
            auto dload = [&](int ss) {
                uint2 v = make_uint2(0u, 0u);
                if (F != kTrit && ss < nsteps) {
                    if (F == kQ2)
                        v = *reinterpret_cast<const uint2 *>(M.scales + row * p.S + ss * (kTgBlocks / 2));
                    else
                        v.x = *reinterpret_cast<const uint32_t *>(M.scales + row * p.S + ss * (kTgBlocks / 4));
                }
                return v;
            };
            uint2 dslot[2] = {dload(0), dload(1)};
            for (int s0 = 0; s0 < nsteps && ok; s0 += 2) {
#pragma unroll
                for (int hs = 0; hs < 2; hs++) {
                    const int s = s0 + hs;
                    if (s >= nsteps) break;
                    const int j0 = s * kTgBlocks;
                    const uint32_t dwp[2] = {dslot[hs].x, dslot[hs].y};
                    if (!__all_sync(0xffffffffu, mbar_wait(&t_full[tb], tph))) {
                        if (lane == 0) report(p.err);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int pb = 0; pb < kTgBlocks / 2; pb++) {
                        const uint32_t taddr =
                            tmem + ((uint32_t)(lq * 32) << 16) + (uint32_t)(tb * 128 + pb * 32);
                        if constexpr (!kPairs) {
                            uint32_t v[32];
                            tmem_ld32(taddr, v);
                            if (pb == kTgBlocks / 2 - 1) {
                                tc_fence_before();
                                __syncwarp();
                                if (lane == 0) mbar_arrive(&t_empty[tb]);
                            }
#pragma unroll
                            for (int t = 0; t < 2; t++) {
                                const int jb = 2 * pb + t;
#pragma unroll
                                for (int b = 0; b < B; b++) {
                                    // isum = 16 S_hi + S_lo, exact
                                    const float is = fmaf(16.0f, __uint_as_float(v[16 * t + b]),
                                                          __uint_as_float(v[16 * t + 8 + b]));
                                    if (F == kTrit)
                                        acc[b] += is;
                                    else
                                        tq[b] = fmaf(dxf[(j0 + jb) * 8 + b], is, tq[b]);
                                }
                                if (F != kTrit && (jb % kBlkPerW) == kBlkPerW - 1) {
                                    const int wb = jb / kBlkPerW;  // weight block within the step
                                    const uint32_t dwb = F == kQ2 ? (wb < 2 ? dwp[0] : dwp[1]) : dwp[0];
                                    const float dw = f16_bits_to_float((uint16_t)((wb & 1) ? (dwb >> 16) : dwb));
#pragma unroll
                                    for (int b = 0; b < B; b++) {
                                        acc[b] = (Acc)fmaf(dw, tq[b], (float)acc[b]);
                                        tq[b] = 0.0f;
                                    }
                                }
                            }
                        } else {
                            // token pairs (2k, 2k + 1): column pair 8t + k holds their S_hi, pair
                            // 8t + 4 + k their S_lo; two tokens per f32x2 instruction
                            // 7-8 tokens: one block's 16 columns per load (the 32-column
                            // load left too few registers there); 5-6 tokens: both blocks at once
                            constexpr bool kHalf = B >= 7;
                            uint64_t pw[kHalf ? 8 : 16];
                            if (!kHalf) tmem_ld32_pairs(taddr, reinterpret_cast<uint64_t (&)[16]>(pw));
#pragma unroll
                            for (int t = 0; t < 2; t++) {
                                uint64_t pr[8];
                                if (kHalf) {
                                    tmem_ld16_pairs(taddr + 16 * t, reinterpret_cast<uint64_t (&)[8]>(pw));
#pragma unroll
                                    for (int i = 0; i < 8; i++) pr[i] = pw[i];
                                } else {
#pragma unroll
                                    for (int i = 0; i < 8; i++) pr[i] = pw[8 * t + i];
                                }
                                if (pb == kTgBlocks / 2 - 1 && (kHalf ? t == 1 : t == 0)) {
                                    tc_fence_before();
                                    __syncwarp();
                                    if (lane == 0) mbar_arrive(&t_empty[tb]);
                                }
                                const int jb = 2 * pb + t;
                                const uint64_t *dxq = reinterpret_cast<const uint64_t *>(dxf + (j0 + jb) * 8);
#pragma unroll
                                for (int k = 0; k < NP; k++) {
                                    uint64_t is2 = pr[4 + k];
                                    ffma2p(is2, pr[k], kSixteen2);  // 16 S_hi + S_lo, exact
                                    if (F == kTrit)
                                        ffma2p(acc2[k], is2, kOne2);        // acc += isum, exact
                                    else
                                        ffma2p(tq2[k], is2, dxq[k]);        // t += d_x * isum
                                }
                                if (F != kTrit && (jb % kBlkPerW) == kBlkPerW - 1) {
                                    const int wb = jb / kBlkPerW;  // weight block within the step
                                    const uint32_t dwb = F == kQ2 ? (wb < 2 ? dwp[0] : dwp[1]) : dwp[0];
                                    const uint32_t dwf = __float_as_uint(
                                        f16_bits_to_float((uint16_t)((wb & 1) ? (dwb >> 16) : dwb)));
                                    const uint64_t dw2 = ((uint64_t)dwf << 32) | dwf;
#pragma unroll
                                    for (int k = 0; k < NP; k++) {
                                        ffma2p(acc2[k], tq2[k], dw2);   // acc += d_w * t
                                        tq2[k] = 0;
                                    }
                                }
                            }
                        }
                    }
                    dslot[hs] = dload(s + 2);
                    if (++tb == kTgAccBufs) {
                        tb = 0;
                        tph ^= 1;
                    }
                }
            }
            if (!ok) break;
            if constexpr (kPairs) {
#pragma unroll
                for (int b = 0; b < B; b++)
                    acc[b] = __uint_as_float((uint32_t)(acc2[b >> 1] >> (32 * (b & 1))));
            }
            if (rv) {
#pragma unroll
                for (int b = 0; b < B; b++) {
                    const int64_t o = (int64_t)b * M.N + row;
                    if (F == kTrit) {
                        const float t = __fmul_rn((float)acc[b], p.x_scale[b]);
                        M.y[o] = __fmul_rn(t, M.w_scale);
                        if (M.aux) M.aux[o] = (int)acc[b];
                    } else {
                        M.y[o] = (float)acc[b];
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, kTgAccBufs * 128);
    }
}

template <int F, int B>
inline int launch_tc_gemv(StreamParams &p, int sms, cudaStream_t st) {
    auto kern = tc_gemv_kernel<F, B>;
    constexpr int smem = tg_smem_bytes<F>();
    int bps = 0;
    if (int e = prepare_kernel(reinterpret_cast<const void *>(kern), kTgThreads, (size_t)smem, &bps))
        return e;
    static_assert(sizeof(TgMaps) + sizeof(StreamParams) < 30000, "kernel parameters too large");
    TgMaps maps;
    int units = 0;
    for (int i = 0; i < p.G; i++) {
        p.m[i].unit0 = units;
        units += (p.m[i].N + kTgRows - 1) / kTgRows;
        const uint64_t row_bytes = (uint64_t)p.nchunk * 16;
        if (int e = encode_rows_map(&maps.m[i], p.m[i].w, row_bytes, (uint64_t)p.m[i].N,
                                    (uint32_t)TgFmt<F>::kBytes, (uint32_t)kTgRows,
                                    TgFmt<F>::kBytes))
            return e;

    }
    p.nunits = units;
    int64_t grid = (int64_t)sms * bps;
    if (grid > units) grid = units;
    if (grid < 1) grid = 1;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(kTgThreads), (size_t)smem, st, p, maps);
}

}  // namespace lb
