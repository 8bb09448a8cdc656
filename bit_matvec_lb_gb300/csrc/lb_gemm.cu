// lb_gemm.cu -- prefill GEMM: Q1_0 / Q2_0_g64 weights x q8_0 activations of M tokens, on the
// 5th-generation tensor cores.
//
// Arithmetic, for token m, weight row n, weight block b and its q8_0 blocks j
// ("bankml: verified low-bit inference on commodity CPUs -- a technical report", III.2-III.3 for
// Q1_0 and the 1x4 prefill tile that reuses one weight block across several activation
// columns, III.5 for Q2_0_g64):
//     y[m][n] = sum_j d_x[m][j] * (d_w[n][b(j)] * isum[m][n][j])
// where isum is the integer dot product of the 32 weights of block j with the 32 int8 codes.
//
// GPU design: exact integers on the f16 tensor-core path (tcgen05.mma kind::f16; the int8 kind
// does not exist on this architecture).
//   * Activations: every q8_0 code is an integer in [-128, 127], exact in f16.  A prologue kernel
//     converts q once into f16 tiles already laid out as the tensor core reads them from shared
//     memory (K-major core matrices, lb_tc.cuh), so the main kernel moves them with one bulk
//     copy per 128x32 tile.  The tiles live in a caller-provided workspace.
//   * Weights: expanded in shared memory to W' = w * d_w (w in {-1, +1} or {-1, 0, +1, +2}),
//     which is exact in f16.  The K order inside each 32-wide block is permuted (identically in
//     the activation tiles) so that one f16x2 pair comes from one shift and one mask of a packed
//     weight word.
//   * One 128x128x32 step is two 16-deep MMAs into a tensor-memory accumulator: its value
//     d_w * isum has at most 24 significant bits (|isum| <= 8192, d_w has 11), so it is exact in
//     fp32.  Each 32-wide block is drained separately (d_x changes every 32 columns of K): the
//     drain warps read the accumulator with tcgen05.ld and add d_x * (d_w * isum) with one FFMA
//     per element into registers, flushing to y every 32 blocks, so the fp32 accumulation depth
//     stays below 32 + K/1024.  Four 128-column accumulators (a stage's two K32 steps use two)
//     let the MMAs of the next stage run while the drain reads the previous one.
//   * Warp roles in a 512-thread CTA: warps 0-3 expand weights (one row each), warp 4 copies
//     activation tiles, warps 5 and 6 issue the MMAs (one thread each, alternate stages; warp 5
//     owns tensor memory), warps 8-15 (two warpgroups) drain.  A 4-stage shared-memory ring of
//     {two A tiles, two B tiles} decouples them; every wait is bounded and reports through the
//     device error word.
#include <algorithm>

#include "lb_tc.cuh"

namespace lb {

constexpr int kGemmThreads = 512;
constexpr int kTileM = 128;
constexpr int kTileN = 128;
constexpr int kTileBytes = 8192;                 // one 128 x 32 f16 operand tile
constexpr int kStages = 4;                       // stages of two K32 steps: {A, A, B, B}
constexpr int kStageBytes = 4 * kTileBytes;
constexpr int kIssuers = 2;                      // MMA-issuing warps, alternating stages
constexpr int kAccBufs = 4;                      // tensor-memory accumulators (128 columns each)
constexpr int kSeg = 32;                         // K32 blocks per drain segment
constexpr int kTotPitch = kTileM + 1;            // totals [n][m] pitch (conflict-free both ways)
constexpr int kTotBytes = kTileN * kTotPitch * 4;
constexpr int kTotOffset = kStages * kStageBytes;
constexpr int kGemmSmem = kTotOffset + kTotBytes + 1024;

enum GFmt { kG1 = 0, kG2 = 1 };

// One weight matrix of a (possibly grouped) call: the call's tiles are those of matrix 0, then
// of matrix 1, ...; tile0 is the index of the matrix's first tile.
struct GemmMat {
    const uint8_t *bits;     // [N][K/8] (Q1_0) or [N][K/4] (Q2_0_g64)
    const uint16_t *scales;  // [N][S]
    float *y;                // [M][N]
    int N, tile0;
};

struct GemmParams {
    GemmMat mat[LB_GEMM_MAX_GROUP];
    const uint8_t *ws;       // activation tiles [mtiles][K/32][8192 B]
    const uint16_t *d;       // [M][K/32] q8_0 scales
    int *err;
    int G, M, K, S, nK32, mtiles;
};

// ------------------------------------------------------------------------------------------
// Prologue: q8_0 codes -> f16 activation tiles in the K-major core-matrix layout, with the
// format's K permutation.  Chunk kc (8 positions) of a 32-wide block holds the byte
// interleave of two source words:  Q2_0_g64 words (4(kc/2) + kc%2, +2), Q1_0 words (kc, kc+4).
// Rows past M are zero.  One thread per (tile row, K32 block), rows fastest.
// ------------------------------------------------------------------------------------------
// `zero` (nzero ints, may be NULL) is cleared as well: the planar GEMM's split counters.
template <int F>
__global__ void __launch_bounds__(256) gemm_prep_act_kernel(const int8_t *__restrict__ q,
                                                            uint8_t *__restrict__ ws, int M,
                                                            int K, int mtiles, int *zero,
                                                            int nzero) {
    pdl_launch_dependents();
    pdl_wait();
    const int nK32 = K / 32;
    const int64_t total = (int64_t)mtiles * nK32 * kTileM;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nzero; i += stride)
        zero[i] = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int r = (int)(i % kTileM);
        const int64_t tj = i / kTileM;
        const int j = (int)(tj % nK32);
        const int t = (int)(tj / nK32);
        const int64_t row = (int64_t)t * kTileM + r;
        uint32_t a[8];
        if (row < M) {
            const uint4 *src = reinterpret_cast<const uint4 *>(q + row * K + (int64_t)j * 32);
            const uint4 lo = src[0], hi = src[1];
            a[0] = lo.x; a[1] = lo.y; a[2] = lo.z; a[3] = lo.w;
            a[4] = hi.x; a[5] = hi.y; a[6] = hi.z; a[7] = hi.w;
        } else {
#pragma unroll
            for (int w = 0; w < 8; w++) a[w] = 0;
        }
        uint8_t *tile = ws + ((int64_t)t * nK32 + j) * kTileBytes;
#pragma unroll
        for (int kc = 0; kc < 4; kc++) {
            const uint32_t x = F == kG2 ? a[4 * (kc >> 1) + (kc & 1)] : a[kc];
            const uint32_t y = F == kG2 ? a[4 * (kc >> 1) + (kc & 1) + 2] : a[kc + 4];
            *reinterpret_cast<uint4 *>(tile + canon_offset(r, kc * 8)) = int8_pair_f16(x, y);
        }
    }
}

// ------------------------------------------------------------------------------------------
// Weight expansion of one 32-wide block of one row into its four 16-byte chunks.
//   Q2_0_g64: code words w0 (codes 0..15) and w1 (16..31); f16x2 number s of word u holds codes
//             (16u + s, 16u + s + 8): (w >> 2s) & 0x00030003 are the two codes in separate
//             halves; (1024 + c) - 1025 = c - 1, times d_w.  f16x2 number i = 8u + s goes to
//             chunk i / 4, slot i % 4.
//   Q1_0:     sign word w; f16x2 number i (0..15) holds weights (i, i + 16): bits i and i + 16
//             shifted to bits 15 and 31 select the sign of d_w.  Chunk i / 4, slot i % 4.
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void expand_q2(uint32_t w0, uint32_t w1, __half d, uint4 (&c)[4]) {
    const __half2 d2 = __halves2half2(d, d);
    const __half2 k1025 = __halves2half2(__ushort_as_half(0x6401), __ushort_as_half(0x6401));
    uint32_t o[16];
#pragma unroll
    for (int u = 0; u < 2; u++) {
        const uint32_t w = u ? w1 : w0;
#pragma unroll
        for (int s = 0; s < 8; s++) {
            uint32_t x = ((w >> (2 * s)) & 0x00030003u) | 0x64006400u;
            __half2 v = __hmul2(__hsub2(*reinterpret_cast<__half2 *>(&x), k1025), d2);
            o[8 * u + s] = *reinterpret_cast<uint32_t *>(&v);
        }
    }
#pragma unroll
    for (int kc = 0; kc < 4; kc++)
        c[kc] = make_uint4(o[4 * kc], o[4 * kc + 1], o[4 * kc + 2], o[4 * kc + 3]);
}

__device__ __forceinline__ void expand_q1(uint32_t w, uint16_t dbits, uint4 (&c)[4]) {
    const uint32_t dd = (uint32_t)dbits | ((uint32_t)dbits << 16);
    uint32_t o[16];
#pragma unroll
    for (int i = 0; i < 16; i++) {
        const uint32_t x = w << (15 - i);
        o[i] = dd ^ (~x & 0x80008000u);  // set bit: +d_w, clear bit: -d_w
    }
#pragma unroll
    for (int kc = 0; kc < 4; kc++)
        c[kc] = make_uint4(o[4 * kc], o[4 * kc + 1], o[4 * kc + 2], o[4 * kc + 3]);
}

__device__ __forceinline__ bool wait_or_report(uint64_t *bar, uint32_t parity, int *err) {
    if (mbar_wait(bar, parity)) return true;
    if (err) atomicOr(err, 1);
    return false;
}

// Index and phase parity of a ring of N stages, advanced one step at a time.
template <int N>
struct Ring {
    int idx = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void next() {
        if (++idx == N) {
            idx = 0;
            phase ^= 1u;
        }
    }
};

template <int F>
__global__ void __launch_bounds__(kGemmThreads, 1) gemm_q_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t gsm_raw[];
    uint8_t *gsm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(gsm_raw) + 1023) &
                                               ~(uintptr_t)1023);
    // full[s]: the stage's two A tiles have landed and its two B tiles are written.
    // empty[s]: the stage's four MMAs have completed -- the stage may be refilled, and the two
    //           accumulators it wrote may be drained.
    // tempty[b]: accumulator b has been read out by the eight drain warps.
    __shared__ __align__(8) uint64_t full[kStages], empty[kStages], tempty[kAccBufs], mma_done;
    __shared__ uint32_t tmem_slot;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int gi = 0;
    while (gi + 1 < p.G && p.mat[gi + 1].tile0 <= (int)blockIdx.x) gi++;
    const GemmMat &W = p.mat[gi];
    const int m_tile = ((int)blockIdx.x - W.tile0) % p.mtiles;
    const int n_tile = ((int)blockIdx.x - W.tile0) / p.mtiles;
    const int64_t m0 = (int64_t)m_tile * kTileM, n0 = (int64_t)n_tile * kTileN;
    const int nK32 = p.nK32;       // even: K is a multiple of 64
    const int nst = nK32 / 2;      // stages of two K32 steps

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; s++) {
            mbar_init(&full[s], 5);   // four expander warps + the activation copy (and its bytes)
            mbar_init(&empty[s], 1);  // commit after the stage's MMAs
        }
        for (int b = 0; b < kAccBufs; b++) mbar_init(&tempty[b], 8);  // eight drain warps
        mbar_init(&mma_done, kIssuers);
        fence_mbar_init();
    }
    if (warp == 5) tmem_alloc(&tmem_slot, kAccBufs * kTileN);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    pdl_launch_dependents();

    if (warp < 4) {
        // ---------------- weight expanders: thread = weight row ----------------
        // The packed weights and scale of each stage are read from global memory kQ stages
        // ahead into a small register queue.
        constexpr int kQ = 4;
        const int nl = threadIdx.x;
        const int64_t n = n0 + nl;
        const bool valid = n < W.N;
        const int64_t nn = valid ? n : 0;
        constexpr int kStBytes = F == kG2 ? 16 : 8;       // packed bytes per stage and row
        const uint8_t *row = W.bits + nn * (int64_t)nst * kStBytes;
        const uint16_t *srow = W.scales + nn * (int64_t)p.S;
        // Q2_0_g64: a stage is one 64-weight block (16 code bytes, one scale); Q1_0: half of a
        // 128-weight block (8 sign bytes; the scale of block st / 2).
        auto load_stage = [&](int st, uint4 &c, uint32_t &sc) {
            if (!valid || st >= nst) {
                c = make_uint4(0, 0, 0, 0);
                sc = 0;
            } else if (F == kG2) {
                c = *reinterpret_cast<const uint4 *>(row + (int64_t)st * 16);
                sc = srow[st];
            } else {
                const uint2 v = *reinterpret_cast<const uint2 *>(row + (int64_t)st * 8);
                c = make_uint4(v.x, v.y, 0, 0);
                sc = srow[st >> 1];
            }
        };
        // Slot j of the queue holds the stages j, j + kQ, j + 2 kQ, ...: the stage loop is unrolled
        // by kQ so that every slot is a fixed register set, refilled right after its last use.
        // (Shifting the queue by one slot per stage would make each shift wait for the load
        // issued one stage earlier -- a full memory latency per stage.)
        uint4 qc[kQ];
        uint32_t qs[kQ];
#pragma unroll
        for (int i = 0; i < kQ; i++) load_stage(i, qc[i], qs[i]);
        const uint32_t boff = (uint32_t)canon_offset(nl, 0) + 2 * kTileBytes;
        Ring<kStages> rs;
        bool ok = true;
        for (int st0 = 0; st0 < nst && ok; st0 += kQ) {
#pragma unroll
            for (int j = 0; j < kQ; j++) {
                const int st = st0 + j;
                if (st >= nst) break;
                if (!__all_sync(0xffffffffu, mbar_wait(&empty[rs.idx], rs.phase ^ 1u))) {
                    if (lane == 0) atomicOr(p.err, 1);
                    ok = false;
                    break;
                }
                uint8_t *bt = gsm + rs.idx * kStageBytes + boff;
#pragma unroll
                for (int t = 0; t < 2; t++) {
                    uint4 c[4];
                    if (F == kG2)
                        expand_q2(t ? qc[j].z : qc[j].x, t ? qc[j].w : qc[j].y,
                                  __ushort_as_half((uint16_t)qs[j]), c);
                    else
                        expand_q1(t ? qc[j].y : qc[j].x, (uint16_t)qs[j], c);
#pragma unroll
                    for (int kc = 0; kc < 4; kc++)
                        *reinterpret_cast<uint4 *>(bt + t * kTileBytes + kc * kCoreLBO) = c[kc];
                }
                load_stage(st + kQ, qc[j], qs[j]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&full[rs.idx]);
                rs.next();
            }
        }
    } else if (warp == 4) {
        // ---------------- activation tiles: two 8 KB bulk copies per stage ----------------
        // One thread's bulk copies are served one after another (about 370 clk each, whatever
        // their size up to 32 KB), so the stage's two tiles are issued by two lanes.
        pdl_wait();
        const uint8_t *src = p.ws + ((int64_t)m_tile * nK32 + lane) * kTileBytes;
        Ring<kStages> rs;
        int issued = 0;
        for (int st = 0; st < nst; st++) {
            bool ok = true;
            if (lane == 0) {
                ok = wait_or_report(&empty[rs.idx], rs.phase ^ 1u, p.err);
                if (ok) mbar_arrive_expect_tx(&full[rs.idx], 2 * kTileBytes);
            }
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
            if (lane < 2)
                bulk_g2s(gsm + rs.idx * kStageBytes + lane * kTileBytes,
                         src + (int64_t)st * 2 * kTileBytes, kTileBytes, &full[rs.idx]);
            rs.next();
            issued = st + 1;
        }
        // No copy may still be landing in shared memory when the CTA exits: wait for the
        // stages issued last (immediate on the normal path, bounded on an error path).
        if (lane == 0)
            for (int st = max(0, issued - kStages); st < issued; st++)
                mbar_wait(&full[st % kStages], (st / kStages) & 1);
    } else if (warp >= 5 && warp < 5 + kIssuers) {
        // ---------------- MMA issue: warp 5 + i issues the stages st = i (mod 2) ----------------
        // Issuer i owns accumulators 2i and 2i + 1 (steps 2st and 2st + 1).
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(kTileM, kTileN);
            const int i = warp - 5;
            const uint32_t sbase = smem_u32(gsm);
            for (int st = i; st < nst; st += kIssuers) {
                const int s = st & (kStages - 1);
                if (!wait_or_report(&full[s], (uint32_t)(st / kStages) & 1u, p.err)) break;
                const uint32_t tph = ((uint32_t)(st / kIssuers) & 1u) ^ 1u;
                const uint32_t sa = sbase + (uint32_t)(s * kStageBytes);
                bool ok = true;
#pragma unroll
                for (int t = 0; t < 2; t++) {
                    const int b = 2 * i + t;
                    if (!wait_or_report(&tempty[b], tph, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = smem_desc(sa + t * kTileBytes);
                    const uint64_t bd = smem_desc(sa + (2 + t) * kTileBytes);
                    const uint32_t d = tmem + (uint32_t)(b * kTileN);
                    mma_f16(d, ad, bd, idesc, 0u);
                    mma_f16(d, ad + (256 >> 4), bd + (256 >> 4), idesc, 1u);
                }
                if (!ok) break;
                mma_commit(&empty[s]);
            }
            // Every MMA issued has completed before tensor memory is released.
            mma_commit(&mma_done);
            wait_or_report(&mma_done, 0, p.err);
        }
    } else if (warp >= 8) {
        // ---------------- drain: d_x * (d_w * isum) into registers ----------------
        // Thread = token row (the lane quarter of its warp), 64 weight columns per warpgroup.
        // Each 32-block segment is added into per-CTA totals in shared memory, laid out [n][m]
        // with pitch 129 (conflict-free for this column-wise access and for the row-wise store).
        pdl_wait();
        float *tot = reinterpret_cast<float *>(gsm + kTotOffset);
        const int g = (warp - 8) >> 2, lq = warp & 3;
        const int mrow = lq * 32 + lane;
        const int64_t m = m0 + mrow;
        const bool mvalid = m < p.M;
        const int col0 = g * 64;
        const uint16_t *drow = p.d + (mvalid ? m : 0) * (int64_t)nK32;
        uint64_t acc[32];
#pragma unroll
        for (int c = 0; c < 32; c++) acc[c] = 0;
        bool first = true;
        const uint32_t tlane = tmem + ((uint32_t)(lq * 32) << 16) + (uint32_t)col0;
        // Activation scales of one stage (two fp16 in a word), loaded three stages ahead.
        auto load_dx2 = [&](int st) -> uint32_t {
            return (mvalid && st < nst) ? *reinterpret_cast<const uint32_t *>(drow + 2 * st) : 0u;
        };
        uint32_t dq0 = load_dx2(0), dq1 = load_dx2(1), dq2 = load_dx2(2);
        Ring<kStages> rs;
        for (int st = 0; st < nst; st++) {
            const uint32_t dw = dq0;
            dq0 = dq1;
            dq1 = dq2;
            dq2 = load_dx2(st + 3);
            if (!__all_sync(0xffffffffu, mbar_wait(&empty[rs.idx], rs.phase))) {
                if (lane == 0) atomicOr(p.err, 1);
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int t = 0; t < 2; t++) {
                const int b = (2 * st + t) & (kAccBufs - 1);
                const uint32_t dxb =
                    __float_as_uint(f16_bits_to_float((uint16_t)(t ? (dw >> 16) : dw)));
                const uint64_t dx2 = ((uint64_t)dxb << 32) | dxb;
                const uint32_t taddr = tlane + (uint32_t)(b * kTileN);
                uint64_t r[16];
                tmem_ld32_pairs(taddr, r);
#pragma unroll
                for (int c = 0; c < 16; c++) ffma2p(acc[c], r[c], dx2);
                tmem_ld32_pairs(taddr + 32, r);
                // The accumulator is free once both halves are in registers.
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[b]);
#pragma unroll
                for (int c = 0; c < 16; c++) ffma2p(acc[16 + c], r[c], dx2);
            }
            rs.next();
            if ((2 * st + 2) % kSeg == 0 || st + 1 == nst) {
                float *t = tot + col0 * kTotPitch + mrow;
#pragma unroll
                for (int c = 0; c < 32; c++) {
                    const float lo = __uint_as_float((uint32_t)acc[c]);
                    const float hi = __uint_as_float((uint32_t)(acc[c] >> 32));
                    float *t0 = t + (2 * c) * kTotPitch, *t1 = t0 + kTotPitch;
                    *t0 = first ? lo : *t0 + lo;
                    *t1 = first ? hi : *t1 + hi;
                    acc[c] = 0;
                }
                first = false;
            }
        }
        // All eight drain warps are done with the totals: store the tile, one 128-byte row
        // segment per warp instruction.
        named_sync(1, 256);
        const int wd = warp - 8;
        for (int rr = 0; rr < kTileM / 8; rr++) {
            const int ml = wd * (kTileM / 8) + rr;
            const int64_t mm = m0 + ml;
            if (mm >= p.M) break;
            float *yrow = W.y + mm * (int64_t)W.N;
#pragma unroll
            for (int i = 0; i < kTileN / 32; i++) {
                const int nl = i * 32 + lane;
                if (n0 + nl < W.N) yrow[n0 + nl] = tot[nl * kTotPitch + ml];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, kAccBufs * kTileN);
    }
}

// Checks and launches of a call over G weight matrices sharing one activation (G = 1 for the
// single-matrix entry points): one prologue for the activation, one launch for every tile of
// every matrix.
static int gemm_q_group(int F, const lb_gemm_matrix *mats, int G, const int8_t *q,
                        const uint16_t *d, int64_t M, int64_t K, void *workspace,
                        size_t workspace_bytes, void *stream) {
    const int qk = F == kG1 ? 128 : 64;
    if (!mats || !q || !d || !workspace) return LB_ERR_NULL;
    if (G < 1 || G > LB_GEMM_MAX_GROUP) return LB_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(d) || !aligned16(workspace)) return LB_ERR_ALIGN;
    if (M < 1 || K < qk || K % qk != 0 || M > (1 << 30) || K > (1 << 24)) return LB_ERR_SHAPE;
    const int64_t mtiles = (M + kTileM - 1) / kTileM;
    if (workspace_bytes < (size_t)(mtiles * kTileM * K * 2)) return LB_ERR_SHAPE;
    GemmParams p{};
    int64_t tiles = 0;
    for (int i = 0; i < G; i++) {
        const lb_gemm_matrix &m = mats[i];
        if (!m.bits || !m.scales || !m.y) return LB_ERR_NULL;
        if (!aligned16(m.bits) || !aligned16(m.scales) || !aligned16(m.y)) return LB_ERR_ALIGN;
        if (m.N < 1 || m.N > (1 << 30)) return LB_ERR_SHAPE;
        p.mat[i].bits = m.bits;
        p.mat[i].scales = m.scales;
        p.mat[i].y = m.y;
        p.mat[i].N = (int)m.N;
        p.mat[i].tile0 = (int)tiles;
        tiles += mtiles * ((m.N + kTileN - 1) / kTileN);
        if (tiles > 0x7fffffff) return LB_ERR_SHAPE;
    }
    DeviceInfo di;
    if (int st = current_device_info(&di)) return st;
    p.err = device_error_word();
    if (!p.err) return LB_ERR_LAUNCH;
    auto kern = F == kG1 ? gemm_q_kernel<kG1> : gemm_q_kernel<kG2>;
    int bps = 0;
    if (int e2 = prepare_kernel(reinterpret_cast<const void *>(kern), kGemmThreads, kGemmSmem,
                                &bps))
        return e2;
    cudaStream_t st = as_stream(stream);
    // prologue: activation tiles
    const int64_t work = mtiles * kTileM * (K / 32);
    int64_t pgrid = (work + 255) / 256;
    if (pgrid > (int64_t)di.sms * 16) pgrid = (int64_t)di.sms * 16;
    int e = F == kG1 ? launch_pdl(gemm_prep_act_kernel<kG1>, dim3((unsigned)pgrid), dim3(256), 0,
                                  st, q, (uint8_t *)workspace, (int)M, (int)K, (int)mtiles,
                                  (int *)nullptr, 0)
                     : launch_pdl(gemm_prep_act_kernel<kG2>, dim3((unsigned)pgrid), dim3(256), 0,
                                  st, q, (uint8_t *)workspace, (int)M, (int)K, (int)mtiles,
                                  (int *)nullptr, 0);
    if (e) return e;
    p.ws = (const uint8_t *)workspace;
    p.d = d;
    p.G = G;
    p.M = (int)M;
    p.K = (int)K;
    p.S = (int)((K / qk + 7) / 8 * 8);
    p.nK32 = (int)(K / 32);
    p.mtiles = (int)mtiles;
    return launch_pdl(kern, dim3((unsigned)tiles), dim3(kGemmThreads), kGemmSmem, st, p);
}

static int gemm_q(int F, const uint8_t *bits, const uint16_t *scales, const int8_t *q,
                  const uint16_t *d, float *y, int64_t M, int64_t N, int64_t K, void *workspace,
                  size_t workspace_bytes, void *stream) {
    const lb_gemm_matrix m = {bits, scales, y, N};
    return gemm_q_group(F, &m, 1, q, d, M, K, workspace, workspace_bytes, stream);
}

}  // namespace lb

using namespace lb;

LB_EXPORT size_t lb_gemm_workspace_bytes(int64_t M, int64_t K) {
    if (M < 1 || K < 1) return 0;
    return (size_t)((M + kTileM - 1) / kTileM) * kTileM * (size_t)K * 2;
}

LB_EXPORT int lb_gemm_q1_0(const uint8_t *bits, const uint16_t *scales, const int8_t *q,
                           const uint16_t *d, float *y, int64_t M, int64_t N, int64_t K,
                           void *workspace, size_t workspace_bytes, void *stream) {
    return gemm_q(kG1, bits, scales, q, d, y, M, N, K, workspace, workspace_bytes, stream);
}

LB_EXPORT int lb_gemm_q2_0_g64(const uint8_t *codes, const uint16_t *scales, const int8_t *q,
                               const uint16_t *d, float *y, int64_t M, int64_t N, int64_t K,
                               void *workspace, size_t workspace_bytes, void *stream) {
    return gemm_q(kG2, codes, scales, q, d, y, M, N, K, workspace, workspace_bytes, stream);
}

LB_EXPORT int lb_gemm_q1_0_grouped(const lb_gemm_matrix *mats, int G, const int8_t *q,
                                   const uint16_t *d, int64_t M, int64_t K, void *workspace,
                                   size_t workspace_bytes, void *stream) {
    return gemm_q_group(kG1, mats, G, q, d, M, K, workspace, workspace_bytes, stream);
}

LB_EXPORT int lb_gemm_q2_0_g64_grouped(const lb_gemm_matrix *mats, int G, const int8_t *q,
                                       const uint16_t *d, int64_t M, int64_t K, void *workspace,
                                       size_t workspace_bytes, void *stream) {
    return gemm_q_group(kG2, mats, G, q, d, M, K, workspace, workspace_bytes, stream);
}

namespace lb {
// Entry for other translation units that bring their own scratch (same checks and launches as
// lb_gemm_q1_0 / lb_gemm_q2_0_g64).
int gemm_q_with_workspace(int q2, const uint8_t *bits, const uint16_t *scales, const int8_t *q,
                          const uint16_t *d, float *y, int64_t M, int64_t N, int64_t K,
                          void *workspace, size_t workspace_bytes, void *stream) {
    return gemm_q(q2 ? kG2 : kG1, bits, scales, q, d, y, M, N, K, workspace, workspace_bytes,
                  stream);
}
}  // namespace lb


// ==========================================================================================
// Planar ternary prefill GEMM (tritium.technology "Architecture", sections 1, 2, 4.1 and 5 for
// the arithmetic; the bankml technical report, III.3, for the prefill tile that reuses one
// weight tile across many tokens).  For token m and weight row n:
//     acc[m][n] = sum_{c: pos} q[m][c] - sum_{c: neg} q[m][c]        (int32, exact)
//     y[m][n]   = (float(acc) * x_scale[m]) * w_scale                  (two roundings)
//
// GPU design.  Activations are the same f16 operand tiles as the Q1_0 GEMM (its prologue and
// K permutation); weights are expanded in shared memory to f16 -1 / 0 / +1.  Every partial sum
// of the tensor core is an integer of magnitude at most 128 K < 2^24, exact in the binary32
// accumulator whatever the order of the additions, so each tensor-memory accumulator runs over
// the whole of K and is read once at the end: no per-block drain.  For the same reason K may
// be split across CTAs with no effect on the result: a call whose tiles would leave SMs idle
// runs the ks splits of each tile as one thread-block cluster; every split parks its integer
// partial tiles in its own shared memory, and after a cluster barrier the CTAs add the partials
// of their share of the rows over the whole cluster (distributed shared memory).
//   Tile: 256 tokens (two 128-token tensor-memory accumulators) x 256 weight rows, one
//   M = 128, N = 256 MMA per token tile and 16-deep step.  Shared memory feeds the tensor core
//   both operands and takes the copies and the weight expansion: N = 256 MMAs read a quarter
//   fewer operand bytes per product than N = 128 ones, and one activation tile feeds 256 weight
//   rows, one expanded weight tile 256 tokens.  Measured: with two token tiles per CTA the main
//   loop runs at the MMA rate; with one (small calls) a stage takes about twice its MMA time.
//   Warp roles in a 320-thread CTA (one per SM): warps 0-7 expand weights (thread = weight row)
//   and then read the accumulators out, warp 8 copies activation tiles (one 8 KB bulk copy per
//   lane: one thread's copies are served one after another), warp 9 owns tensor memory and
//   issues the MMAs.  Three stages of one 64-column beat each; every mbarrier wait is bounded
//   and reports through the device error word.  Every barrier of the output phase is reached
//   by every thread of every CTA the same number of times.
// ==========================================================================================
namespace lb {

constexpr int kTritExpWarps = 8;          // warps 0-7: weight expanders, then the output
constexpr int kTritCopyWarp = 8;           // activation copies
constexpr int kTritMmaWarp = 9;            // MMA issue, tensor memory
constexpr int kTritThreads = 320;
constexpr int kTritTileN = 256;            // weight rows per tile (one N = 256 MMA)
constexpr int kTritStages = 3;
// A stage: the two 32-deep activation tiles of each of the CTA's two token tiles (8 KB each),
// then the two 256-row expanded weight tiles they share (16 KB each).
constexpr int kTritBTileBytes = kTritTileN * 32 * 2;
constexpr int kTritAOffBytes = 4 * kTileBytes;
constexpr int kTritStageBytes = kTritAOffBytes + 2 * kTritBTileBytes;
constexpr int kTritSmem = kTritStages * kTritStageBytes + 1024;
constexpr int kTritSplitCtas = 152;        // split K while fewer CTAs than this would run
constexpr int kTritMaxSplit = 4;           // cluster size (8 measured slower)
constexpr int kTritMinStages = 4;          // beats per split, at least
// the partial tiles of one output pass, [token][column] with a 4-float pad (conflict-free):
// 256 tokens x 128 columns, or 128 tokens x 256 columns (one token tile, or a split-K CTA)
static_assert(2 * kTileM * (kTileN + 4) * 4 <= kTritStages * kTritStageBytes &&
                  kTileM * (2 * kTileN + 4) * 4 <= kTritStages * kTritStageBytes,
              "the partial tiles must fit in the stage ring");

struct TritGemmMat {
    const uint4 *planes;     // [N][K/64] beats {pos lo, pos hi, neg lo, neg hi}
    float *y;                // [M][N]
    int32_t *acc;            // [M][N] or NULL
    float w_scale;
    int N, tile0;
};

struct TritGemmParams {
    TritGemmMat mat[LB_GEMM_MAX_GROUP];
    const uint8_t *ws;       // activation tiles [mtiles][K/32][8192 B]
    const float *x_scale;    // [M]
    int *err;
    int G, M, nst, mtiles, mstep, mpairs, ks, sps;
};

// Half a planar beat -- pos word P and neg word Nn of 32 columns, bit c <-> column c -- as the
// four 16-byte chunks of one weight row of a 32-deep operand tile.  f16x2 number i (0..15) holds
// the weights of columns (i, i + 16), the pairing of the Q1_0 activation tiles.  The 2-bit value
// 1 + p - n (0, 1 or 2) of every column is formed for the even and for the odd columns in one
// addition each; field s of the even word is column 2s (high half: 2s + 16), and
// (1024 + f) - 1025 = p - n in f16.
__device__ __forceinline__ void expand_trit(uint32_t P, uint32_t Nn, uint4 (&c)[4]) {
    constexpr uint32_t kEven = 0x55555555u;
    const uint32_t fe = (P & kEven) + (~Nn & kEven);
    const uint32_t fo = ((P >> 1) & kEven) + ((~Nn >> 1) & kEven);
    const __half2 k1025 = __halves2half2(__ushort_as_half(0x6401), __ushort_as_half(0x6401));
    uint32_t o[16];
#pragma unroll
    for (int s = 0; s < 8; s++) {
        uint32_t xe = ((fe >> (2 * s)) & 0x00030003u) | 0x64006400u;
        uint32_t xo = ((fo >> (2 * s)) & 0x00030003u) | 0x64006400u;
        __half2 ve = __hsub2(*reinterpret_cast<__half2 *>(&xe), k1025);
        __half2 vo = __hsub2(*reinterpret_cast<__half2 *>(&xo), k1025);
        o[2 * s] = *reinterpret_cast<uint32_t *>(&ve);
        o[2 * s + 1] = *reinterpret_cast<uint32_t *>(&vo);
    }
#pragma unroll
    for (int kc = 0; kc < 4; kc++)
        c[kc] = make_uint4(o[4 * kc], o[4 * kc + 1], o[4 * kc + 2], o[4 * kc + 3]);
}

// Cluster barrier over every thread of every CTA of the cluster (release / acquire: shared
// memory written before it is visible to the whole cluster after it).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__global__ void __launch_bounds__(kTritThreads, 1)
    gemm_trit_kernel(const __grid_constant__ TritGemmParams p) {
    extern __shared__ uint8_t gsm_raw[];
    uint8_t *gsm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(gsm_raw) + 1023) &
                                               ~(uintptr_t)1023);
    // full[s]: the stage's activation tiles have landed and its two weight tiles are written.
    // empty[s]: the stage's MMAs have completed (the stage may be refilled).
    // mma_done: every MMA of the CTA has completed (the accumulators may be read).
    __shared__ __align__(8) uint64_t full[kTritStages], empty[kTritStages], mma_done;
    __shared__ uint32_t tmem_slot;
    __shared__ float xs_tile[2 * kTileM];  // activation scales of the tile's tokens
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = (int)blockIdx.x / p.ks, split = (int)blockIdx.x % p.ks;  // split = rank
    int gi = 0;
    while (gi + 1 < p.G && p.mat[gi + 1].tile0 <= tile) gi++;
    const TritGemmMat &W = p.mat[gi];
    // a tile is p.mstep (1 or 2) token tiles from m_tile on x 256 weight rows
    const int m_pair = (tile - W.tile0) % p.mpairs;
    const int n_tile = (tile - W.tile0) / p.mpairs;
    const int m_tile = p.mstep * m_pair;
    const int halves = min(p.mstep, p.mtiles - m_tile);  // the last pair may hold one tile
    const int64_t m0 = (int64_t)m_tile * kTileM, n0 = (int64_t)n_tile * kTritTileN;
    const int sb = split * p.sps;                 // first beat of this split
    const int nloc = min(p.nst, sb + p.sps) - sb;  // beats of this split (>= 1 by construction)
    float *part = reinterpret_cast<float *>(gsm);  // partial tiles, once the ring is idle

    if (threadIdx.x == 0) {
        for (int s = 0; s < kTritStages; s++) {
            mbar_init(&full[s], kTritExpWarps + 1);  // expander warps + the activation copies
            mbar_init(&empty[s], 1);                 // commit after the stage's MMAs
        }
        mbar_init(&mma_done, 1);
        fence_mbar_init();
    }
    if (warp == kTritMmaWarp) tmem_alloc(&tmem_slot, 2 * kTritTileN);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    pdl_launch_dependents();

    if (warp < kTritExpWarps) {
        // ---------------- weight expanders: thread = weight row ----------------
        // Beats are read kQ stages ahead into a register queue with one fixed slot per stage of
        // the unrolled loop.
        constexpr int kQ = 4;
        const int nl = threadIdx.x;
        const int64_t n = n0 + nl;
        const bool valid = n < W.N;
        const uint4 *row = W.planes + (valid ? n : 0) * (int64_t)p.nst + sb;
        auto load_beat = [&](int i) -> uint4 {
            return (valid && i < nloc) ? row[i] : make_uint4(0, 0, 0, 0);
        };
        uint4 qb[kQ];
#pragma unroll
        for (int i = 0; i < kQ; i++) qb[i] = load_beat(i);
        const uint32_t boff = (uint32_t)canon_offset(nl, 0) + kTritAOffBytes;
        Ring<kTritStages> rs;
        bool ok = true;
        for (int i0 = 0; i0 < nloc && ok; i0 += kQ) {
#pragma unroll
            for (int j = 0; j < kQ; j++) {
                const int i = i0 + j;
                if (i >= nloc) break;
                if (!__all_sync(0xffffffffu, mbar_wait(&empty[rs.idx], rs.phase ^ 1u))) {
                    if (lane == 0) atomicOr(p.err, 1);
                    ok = false;
                    break;
                }
                uint8_t *bt = gsm + rs.idx * kTritStageBytes + boff;
#pragma unroll
                for (int t = 0; t < 2; t++) {
                    uint4 c[4];
                    expand_trit(t ? qb[j].y : qb[j].x, t ? qb[j].w : qb[j].z, c);
#pragma unroll
                    for (int kc = 0; kc < 4; kc++)
                        *reinterpret_cast<uint4 *>(bt + t * kTritBTileBytes + kc * kCoreLBO) =
                            c[kc];
                }
                qb[j] = load_beat(i + kQ);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&full[rs.idx]);
                rs.next();
            }
        }
        // activation scales of the tile's tokens, for the output phase
        pdl_wait();
        if (threadIdx.x < 2 * kTileM) {
            const int64_t m = m0 + threadIdx.x;
            xs_tile[threadIdx.x] = (threadIdx.x < halves * kTileM && m < p.M) ? p.x_scale[m] : 0.f;
        }
    } else if (warp == kTritCopyWarp) {
        // ---------------- activation tiles: one 8 KB bulk copy per tile, lanes in parallel ----
        pdl_wait();
        const int nt = 2 * halves;                      // tiles per stage
        const int h = lane >> 1, t = lane & 1;           // this lane's token tile and K32 step
        const uint8_t *src = p.ws + ((int64_t)(m_tile + h) * p.nst + sb) * 2 * kTileBytes +
                             (int64_t)t * kTileBytes;
        Ring<kTritStages> rs;
        int issued = 0;
        for (int i = 0; i < nloc; i++) {
            bool ok = true;
            if (lane == 0) {
                ok = wait_or_report(&empty[rs.idx], rs.phase ^ 1u, p.err);
                if (ok) mbar_arrive_expect_tx(&full[rs.idx], (uint32_t)(nt * kTileBytes));
            }
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
            if (lane < nt)
                bulk_g2s(gsm + rs.idx * kTritStageBytes + (2 * h + t) * kTileBytes,
                         src + (int64_t)i * 2 * kTileBytes, kTileBytes, &full[rs.idx]);
            rs.next();
            issued = i + 1;
        }
        // No copy may still be landing in shared memory when the ring is reused or the CTA
        // exits.
        if (lane == 0)
            for (int i = max(0, issued - kTritStages); i < issued; i++)
                mbar_wait(&full[i % kTritStages], (uint32_t)(i / kTritStages) & 1u);
    } else if (warp == kTritMmaWarp) {
        // ---------------- MMA issue: one thread, one accumulator per token tile ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(kTileM, kTritTileN);
            const uint32_t sbase = smem_u32(gsm);
            Ring<kTritStages> rs;
            for (int i = 0; i < nloc; i++) {
                if (!wait_or_report(&full[rs.idx], rs.phase, p.err)) break;
                tc_fence_after();
                const uint32_t sa = sbase + (uint32_t)(rs.idx * kTritStageBytes);
#pragma unroll
                for (int t = 0; t < 2; t++) {
                    const uint64_t bd = smem_desc(sa + kTritAOffBytes + t * kTritBTileBytes);
#pragma unroll
                    for (int h = 0; h < 2; h++) {
                        if (h >= halves) break;
                        const uint64_t ad = smem_desc(sa + (2 * h + t) * kTileBytes);
                        const uint32_t d = tmem + (uint32_t)(h * kTritTileN);
                        mma_f16(d, ad, bd, idesc, (i | t) ? 1u : 0u);
                        mma_f16(d, ad + (256 >> 4), bd + (256 >> 4), idesc, 1u);
                    }
                }
                mma_commit(&empty[rs.idx]);
                rs.next();
            }
            mma_commit(&mma_done);
            wait_or_report(&mma_done, 0, p.err);
        }
    }

    // Output.  Integer partials: every sum is an integer below 2^24, exact in any order; y takes
    // the two roundings of the planar GEMV.  Rows of y are written by whole warps, lane l taking
    // columns 4l .. 4l + 3 of every 128 (coalesced 512-byte stores).
    if (warp < kTritExpWarps) {
        if (!__all_sync(0xffffffffu, mbar_wait(&mma_done, 0)) && lane == 0) atomicOr(p.err, 1);
        tc_fence_after();
    }
    // Writes y[m0 + rr][nbase + 128 g + 4 lane ..] (and acc) from the integer sums a.
    auto store_row = [&](int rr, int g, int64_t nbase, const float4 &a) {
        const int64_t m = m0 + rr;
        const int64_t nb = nbase + g * kTileN + 4 * lane;
        const float xs = xs_tile[rr];
        const float av[4] = {a.x, a.y, a.z, a.w};
        float o[4];
#pragma unroll
        for (int j = 0; j < 4; j++) o[j] = __fmul_rn(__fmul_rn(av[j], xs), W.w_scale);
        float *yrow = W.y + m * (int64_t)W.N;
        int32_t *arow = W.acc ? W.acc + m * (int64_t)W.N : nullptr;
        if ((W.N & 3) == 0 && nb + 4 <= W.N) {
            *reinterpret_cast<float4 *>(yrow + nb) = make_float4(o[0], o[1], o[2], o[3]);
            if (arow)
                *reinterpret_cast<int4 *>(arow + nb) =
                    make_int4(__float2int_rn(av[0]), __float2int_rn(av[1]),
                              __float2int_rn(av[2]), __float2int_rn(av[3]));
        } else {
#pragma unroll
            for (int j = 0; j < 4; j++) {
                if (nb + j < W.N) {
                    yrow[nb + j] = o[j];
                    if (arow) arow[nb + j] = __float2int_rn(av[j]);
                }
            }
        }
    };
    if (p.ks > 1) {
        // K split over the cluster (one token tile per CTA): every split parks its 128 x 256
        // partial tile in its idle stage ring ([token][column], 4-float pad: conflict-free); after
        // a cluster barrier each CTA adds the ks partials of its share of the token rows through
        // distributed shared memory, two rows per warp at a time with every load in flight
        // together; a last cluster barrier keeps every CTA's partials alive until all are read.
        constexpr int pitch = kTritTileN + 4;
        if (warp < kTritExpWarps) {
            const int q = warp & 3, g = warp >> 2;  // lane quarter, column half
            const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(g * kTileN);
            float *dst = part + (q * 32 + lane) * pitch + g * kTileN;
#pragma unroll 1
            for (int c = 0; c < kTileN / 32; c++) {
                uint32_t r[32];
                __syncwarp();  // the tensor-memory load is warp-collective
                tmem_ld32(tl + 32 * c, r);
#pragma unroll
                for (int v = 0; v < 8; v++)
                    *reinterpret_cast<float4 *>(dst + 32 * c + 4 * v) =
                        make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                    __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
            }
        }
        __syncwarp();
        cluster_sync_all();
        if (warp < kTritExpWarps) {
            const int rstep = kTritExpWarps * p.ks;
            for (int r0 = split * kTritExpWarps + warp; r0 < kTileM; r0 += 2 * rstep) {
                if (m0 + r0 >= p.M) break;  // rows run upward: the rest is past M as well
                float4 a[2][2];
#pragma unroll
                for (int u = 0; u < 2; u++) {
                    const int rr = r0 + u * rstep;
                    const bool live = rr < kTileM && m0 + rr < p.M;
#pragma unroll
                    for (int g = 0; g < 2; g++) {
                        a[u][g] = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (!live) continue;
                        const uint32_t local = smem_u32(part + rr * pitch + g * kTileN + 4 * lane);
#pragma unroll
                        for (int sp = 0; sp < kTritMaxSplit; sp++) {
                            if (sp >= p.ks) break;
                            uint32_t addr;
                            float4 t;
                            asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                                         : "=r"(addr) : "r"(local), "r"((uint32_t)sp));
                            asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                                         : "=f"(t.x), "=f"(t.y), "=f"(t.z), "=f"(t.w)
                                         : "r"(addr));
                            a[u][g].x += t.x;
                            a[u][g].y += t.y;
                            a[u][g].z += t.z;
                            a[u][g].w += t.w;
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < 2; u++) {
                    const int rr = r0 + u * rstep;
                    if (rr >= kTileM || m0 + rr >= p.M) break;
#pragma unroll
                    for (int g = 0; g < 2; g++) store_row(rr, g, n0, a[u][g]);
                }
            }
        }
        __syncwarp();
        cluster_sync_all();
    } else {
        // One CTA per tile: the partials are parked in the idle stage ring as [token][column]
        // tiles -- all 256 weight rows at once for one token tile (128 x 256 fits), in two passes
        // of 128 rows for two -- by warps 0-7 (lane quarter w % 4; token tile, or with one token
        // tile column half, w / 4), then written to y row by row: one bulk copy per token row,
        // or per-thread stores (a warp writes 128 columns per instruction).
        const int npass = halves == 1 ? 1 : 2;
        const int ngrp = halves == 1 ? 2 : 1;    // 128-column groups per pass
        const int pitch = ngrp * kTileN + 4;      // partial row pitch in floats (conflict-free)
        // Rows of y 16-byte aligned (y is, and N a multiple of 4) and no integer output: the
        // partials are scaled as they are parked and every token row leaves in one bulk copy.
        const bool bulk = W.acc == nullptr && (W.N & 3) == 0;
        for (int pass = 0; pass < npass; pass++) {
            const int64_t nbase = n0 + pass * kTileN;
            if (warp < kTritExpWarps) {
                const int hi = warp >> 2, q = warp & 3;
                const int h = halves == 1 ? 0 : hi;  // token tile
                const int g = halves == 1 ? hi : 0;  // column group within the pass
                if (h < halves) {
                    const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16) +
                                        (uint32_t)(h * kTritTileN + pass * kTileN + g * kTileN);
                    const int row = h * kTileM + q * 32 + lane;
                    const float xs = m0 + row < p.M ? p.x_scale[m0 + row] : 0.f;
#pragma unroll 1
                    for (int c = 0; c < kTileN / 32; c++) {
                        uint32_t r[32];
                        __syncwarp();  // the tensor-memory load is warp-collective
                        tmem_ld32(tl + 32 * c, r);
                        float4 *dst =
                            reinterpret_cast<float4 *>(part + row * pitch + g * kTileN + 32 * c);
                        if (bulk) {
#pragma unroll
                            for (int v = 0; v < 32; v++)
                                r[v] = __float_as_uint(__fmul_rn(
                                    __fmul_rn(__uint_as_float(r[v]), xs), W.w_scale));
                        }
#pragma unroll
                        for (int v = 0; v < 8; v++)
                            dst[v] = make_float4(__uint_as_float(r[4 * v]),
                                                 __uint_as_float(r[4 * v + 1]),
                                                 __uint_as_float(r[4 * v + 2]),
                                                 __uint_as_float(r[4 * v + 3]));
                    }
                    if (bulk) fence_proxy_async_smem();  // parked rows -> the bulk copies
                }
            }
            __syncthreads();
            if (bulk) {
                const int rr = threadIdx.x;  // one token row per thread of warps 0-7
                if (rr < halves * kTileM && m0 + rr < p.M && nbase < W.N) {
                    const int cols = (int)min((int64_t)ngrp * kTileN, (int64_t)W.N - nbase);
                    bulk_s2g(W.y + (m0 + rr) * (int64_t)W.N + nbase, part + rr * pitch,
                             (uint32_t)cols * 4u);
                    bulk_commit();
                    if (pass + 1 < npass)
                        bulk_wait_read();
                    else
                        bulk_wait_all();
                }
            } else if (warp < kTritExpWarps && nbase < W.N) {
                const int nrows = halves * kTileM;
                for (int rr = warp; rr < nrows; rr += kTritExpWarps) {
                    if (m0 + rr >= p.M) break;  // rows run upward: the rest is past M as well
#pragma unroll
                    for (int g = 0; g < 2; g++) {
                        if (g >= ngrp) break;
                        store_row(rr, g, nbase,
                                  *reinterpret_cast<const float4 *>(part + rr * pitch +
                                                                    g * kTileN + 4 * lane));
                    }
                }
            }
            // every partial read before the next pass overwrites it
            __syncthreads();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kTritMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 2 * kTritTileN);
    }
}

// Per-token absmax int8 quantization (lb_quantize_i8_absmax: s = 127 / amax, q = rne(x s)
// clamped, x_scale = amax / 127) that also writes the planar GEMM's activation operand tiles
// (the workspace contents its prologue would build from q).  One CTA per token row of the
// 128-row tiles; rows past M write zero operand rows.  Thread t quantizes words t, t + 512, ...
// (4 codes each); a 32-wide block is eight words held by eight consecutive lanes, and the lane
// of word kc < 4 takes word kc + 4 from four lanes up to write chunk kc of the block.
constexpr int kQTHold = 4;
__global__ void __launch_bounds__(512) quantize_i8_tiles_kernel(const float *__restrict__ x,
                                                               int8_t *__restrict__ q,
                                                               float *__restrict__ x_scale,
                                                               uint8_t *__restrict__ ws, int M,
                                                               int K) {
    __shared__ float red[32];
    pdl_launch_dependents();
    pdl_wait();
    const int m = blockIdx.x, lane = threadIdx.x & 31;
    const int nK32 = K / 32, r = m % kTileM;
    const int nq = K / 4;
    uint8_t *tiles = ws + (int64_t)(m / kTileM) * nK32 * kTileBytes;
    auto put = [&](int w, uint32_t a, uint32_t b) {  // word w = a, word w + 4 = b
        if ((w & 7) < 4)
            *reinterpret_cast<uint4 *>(tiles + (int64_t)(w >> 3) * kTileBytes +
                                       canon_offset(r, (w & 7) * 8)) = int8_pair_f16(a, b);
    };
    if (m >= M) {
        for (int w = threadIdx.x; w < nq; w += blockDim.x) put(w, 0u, 0u);
        return;
    }
    const float4 *xb = reinterpret_cast<const float4 *>(x + (int64_t)m * K);
    float a = 0.0f;
    float4 held[kQTHold];
#pragma unroll
    for (int h = 0; h < kQTHold; h++) {
        const int i = threadIdx.x + h * blockDim.x;
        held[h] = i < nq ? xb[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 v = held[h];
        a = fmaxf(a, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    for (int i = threadIdx.x + kQTHold * blockDim.x; i < nq; i += blockDim.x) {
        const float4 v = xb[i];
        a = fmaxf(a, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if (lane == 0) red[threadIdx.x >> 5] = a;
    __syncthreads();
    if (threadIdx.x < 32) {
        a = (threadIdx.x < (blockDim.x >> 5)) ? red[threadIdx.x] : 0.0f;
        for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        if (threadIdx.x == 0) red[0] = a;
    }
    __syncthreads();
    const float amax = red[0];
    const float s = (amax != 0.0f) ? __fdiv_rn(127.0f, amax) : 0.0f;
    if (threadIdx.x == 0) x_scale[m] = __fdiv_rn(amax, 127.0f);
    uint32_t *qb = reinterpret_cast<uint32_t *>(q + (int64_t)m * K);
    // every lane of a warp takes part in each shuffle (nq is a multiple of 16: a warp's words
    // past nq are whole 8-word blocks, their results unused)
#pragma unroll
    for (int h = 0; h < kQTHold; h++) {
        const int i = threadIdx.x + h * blockDim.x;
        if (i - lane >= nq) break;
        const uint32_t w = quantize_i8_word(held[h], s);
        const uint32_t w4 = __shfl_down_sync(0xffffffffu, w, 4);
        if (i < nq) {
            qb[i] = w;
            put(i, w, w4);
        }
    }
    for (int i = threadIdx.x + kQTHold * blockDim.x; i - lane < nq; i += blockDim.x) {
        const uint32_t w = i < nq ? quantize_i8_word(xb[i], s) : 0u;
        const uint32_t w4 = __shfl_down_sync(0xffffffffu, w, 4);
        if (i < nq) {
            qb[i] = w;
            put(i, w, w4);
        }
    }
}

// Checks and launches of a planar call over G matrices sharing one activation.  `q` is the
// int8 activation (its operand tiles are built by the prologue kernel), or NULL when the
// workspace already holds them (written by lb_quantize_i8_absmax_tiles).
static int gemm_trit_group(const lb_trit_matrix *mats, int G, const int8_t *q,
                           const float *x_scale, int64_t M, int64_t K, void *workspace,
                           size_t workspace_bytes, void *stream, bool pretiled = false) {
    if (!mats || (!q && !pretiled) || !x_scale || !workspace) return LB_ERR_NULL;
    if (G < 1 || G > LB_GEMM_MAX_GROUP) return LB_ERR_SHAPE;
    if ((q && !aligned16(q)) || !aligned16(x_scale) || !aligned16(workspace)) return LB_ERR_ALIGN;
    if (M < 1 || M > (1 << 30) || K < 64 || K % 64 != 0 || K > (1 << 24) / 128)
        return LB_ERR_SHAPE;
    if (workspace_bytes < lb_gemm_workspace_bytes(M, K)) return LB_ERR_SHAPE;
    const int64_t mtiles = (M + kTileM - 1) / kTileM;
    // Two token tiles per CTA share each expanded weight tile; a call with few tiles takes one
    // per CTA instead, so that more SMs work on it.
    int64_t ntiles = 0;
    for (int i = 0; i < G; i++) ntiles += (mats[i].N + kTritTileN - 1) / kTritTileN;
    const int mstep = ((mtiles + 1) / 2 * ntiles < kTritSplitCtas / 2) ? 1 : 2;
    const int64_t mpairs = (mtiles + mstep - 1) / mstep;
    TritGemmParams p{};
    int64_t tiles = 0;
    for (int i = 0; i < G; i++) {
        const lb_trit_matrix &m = mats[i];
        if (!m.planes || !m.y) return LB_ERR_NULL;
        if (!aligned16(m.planes) || !aligned16(m.y) || (m.acc_opt && !aligned16(m.acc_opt)))
            return LB_ERR_ALIGN;
        if (m.N < 1 || m.N > (1 << 30)) return LB_ERR_SHAPE;
        p.mat[i].planes = reinterpret_cast<const uint4 *>(m.planes);
        p.mat[i].y = m.y;
        p.mat[i].acc = m.acc_opt;
        p.mat[i].w_scale = m.w_scale;
        p.mat[i].N = (int)m.N;
        p.mat[i].tile0 = (int)tiles;
        tiles += mpairs * ((m.N + kTritTileN - 1) / kTritTileN);
        if (tiles > 0x7fffffff / kTritMaxSplit) return LB_ERR_SHAPE;
    }
    const int nst = (int)(K / 64);
    // Split K when the tiles alone would leave SMs idle (ks * tiles <= kTritSplitCtas), with at
    // least kTritMinStages beats per split and no split empty.
    // Only one-token-tile CTAs split (a 128 x 256 partial tile fits the idle stage ring).
    int ks = (int)std::min<int64_t>(kTritMaxSplit, std::max<int64_t>(1, kTritSplitCtas / tiles));
    ks = std::min(ks, std::max(1, nst / kTritMinStages));
    if (mstep != 1) ks = 1;
    const int sps = (nst + ks - 1) / ks;
    ks = (nst + sps - 1) / sps;
    DeviceInfo di;
    if (int st = current_device_info(&di)) return st;
    p.err = device_error_word();
    if (!p.err) return LB_ERR_LAUNCH;
    int bps = 0;
    if (int e = prepare_kernel(reinterpret_cast<const void *>(gemm_trit_kernel), kTritThreads,
                               kTritSmem, &bps))
        return e;
    cudaStream_t st = as_stream(stream);
    const int64_t work = mtiles * kTileM * (K / 32);
    int64_t pgrid = (work + 255) / 256;
    if (pgrid > (int64_t)di.sms * 16) pgrid = (int64_t)di.sms * 16;
    if (!pretiled)
        if (int e = launch_pdl(gemm_prep_act_kernel<kG1>, dim3((unsigned)pgrid), dim3(256), 0, st,
                               q, (uint8_t *)workspace, (int)M, (int)K, (int)mtiles,
                               (int *)nullptr, 0))
            return e;
    p.ws = static_cast<const uint8_t *>(workspace);
    p.x_scale = x_scale;
    p.G = G;
    p.M = (int)M;
    p.nst = nst;
    p.mtiles = (int)mtiles;
    p.mstep = mstep;
    p.mpairs = (int)mpairs;
    p.ks = ks;
    p.sps = sps;
    // The ks splits of a tile are consecutive blocks and form one cluster.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(tiles * ks));
    cfg.blockDim = dim3(kTritThreads);
    cfg.dynamicSmemBytes = kTritSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)ks;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_trit_kernel, p);
    if (e == cudaSuccess) return LB_OK;
    record_cuda_error(e);
    return LB_ERR_LAUNCH;
}

}  // namespace lb

LB_EXPORT size_t lb_gemm_trit_workspace_bytes(int64_t M, int64_t K) {
    return lb_gemm_workspace_bytes(M, K);
}

LB_EXPORT int lb_gemm_trit_planes_grouped(const lb_trit_matrix *mats, int G, const int8_t *q,
                                          const float *x_scale, int64_t M, int64_t K,
                                          void *workspace, size_t workspace_bytes,
                                          void *stream) {
    return gemm_trit_group(mats, G, q, x_scale, M, K, workspace, workspace_bytes, stream);
}

LB_EXPORT int lb_quantize_i8_absmax_tiles(const float *x, int8_t *q, float *x_scale, int64_t M,
                                          int64_t K, void *workspace, size_t workspace_bytes,
                                          void *stream) {
    if (!x || !q || !x_scale || !workspace) return LB_ERR_NULL;
    if (!aligned16(x) || !aligned16(q) || !aligned16(x_scale) || !aligned16(workspace))
        return LB_ERR_ALIGN;
    if (M < 1 || M > (1 << 30) || K < 64 || K % 64 != 0 || K > (1 << 24) / 128)
        return LB_ERR_SHAPE;
    if (workspace_bytes < lb_gemm_workspace_bytes(M, K)) return LB_ERR_SHAPE;
    DeviceInfo di;
    if (int st = current_device_info(&di)) return st;
    const int64_t rows = (M + kTileM - 1) / kTileM * kTileM;
    return launch_pdl(quantize_i8_tiles_kernel, dim3((unsigned)rows), dim3(512), 0,
                      as_stream(stream), x, q, x_scale, (uint8_t *)workspace, (int)M, (int)K);
}

LB_EXPORT int lb_gemm_trit_planes_grouped_tiles(const lb_trit_matrix *mats, int G,
                                                const float *x_scale, int64_t M, int64_t K,
                                                void *workspace, size_t workspace_bytes,
                                                void *stream) {
    return gemm_trit_group(mats, G, nullptr, x_scale, M, K, workspace, workspace_bytes, stream,
                           true);
}

LB_EXPORT int lb_gemm_trit_planes(const uint64_t *planes, float w_scale, const int8_t *q,
                                  const float *x_scale, float *y, int32_t *acc_opt, int64_t M,
                                  int64_t N, int64_t K, void *workspace, size_t workspace_bytes,
                                  void *stream) {
    const lb_trit_matrix m = {planes, w_scale, y, acc_opt, N};
    return gemm_trit_group(&m, 1, q, x_scale, M, K, workspace, workspace_bytes, stream);
}
