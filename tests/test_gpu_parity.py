"""GPU parity: every CUDA entry point against the CPU oracle, on the same seeded inputs.

Bars: integer results (q8_0 codes and scales, repacked planes, Q1_0/Q2_0_g64 block sums, planar
accumulators and planar outputs) bit-exact; fp32 outputs of the Q1_0 / Q2_0_g64 / bf16 products
within |y - exact| <= 1e-5 * sum|terms| + 1e-6.  Sizes span several tiles and ragged tails, batch
1..8, the degenerate cases (code +2, all -128 activations, zero blocks, unit scales) and the
full workload shapes (full comparison where the oracle is fast enough, sampled rows otherwise).
"""
import numpy as np
import pytest
import torch

import bit_matvec_lb_gb300 as lb
import oracle
import synth
from gpu_util import dev, gemv_bf16, gemv_q, gemv_trit, guarded, host, repack_on_gpu, within

pytestmark = pytest.mark.gpu


def _q8(B, K, seed):
    return oracle.quantize_q8_0(synth.activations(B, K, seed))


# ----------------------------------------------------------------------------------------------
# quantizers and repack
# ----------------------------------------------------------------------------------------------
@pytest.mark.parametrize("B,K", [(1, 32), (3, 96), (1, 512), (8, 4096), (2, 12288), (512, 4096)])
def test_quantize_q8_0(B, K):
    x = synth.activations(B, K, seed=B * 7 + K)
    x[0, :32] = 0.0                                    # an all-zero block
    if K >= 64:
        x[0, 32:64] *= 1e4                              # a large block
    q_ref, d_ref = oracle.quantize_q8_0(x)
    q = guarded((B, K), torch.int8)
    d = guarded((B, K // 32), torch.int16)
    lb.lb_quantize_q8_0(dev(x), q, d, B, K)
    torch.cuda.synchronize()
    assert np.array_equal(host(q), q_ref)
    assert np.array_equal(host(d, np.uint16), d_ref)


def test_quantize_q8_0_ties():
    from golden_io import read
    gd = read("q8_0_ties.txt")
    x = np.array([[float(t) for t in gd["x"].split()]], dtype=np.float32)
    q = guarded((1, 32), torch.int8)
    d = guarded((1, 1), torch.int16)
    lb.lb_quantize_q8_0(dev(x), q, d, 1, 32)
    torch.cuda.synchronize()
    assert host(q)[0].tolist() == [int(t) for t in gd["q"].split()]
    assert int(host(d, np.uint16)[0, 0]) == int(gd["d"], 16)


@pytest.mark.parametrize("B,K", [(1, 16), (1, 2560), (8, 2560), (3, 6912)])
def test_quantize_i8_absmax(B, K):
    x = synth.activations(B, K, seed=K + B)
    if B > 1:
        x[1] = 0.0
    q_ref, s_ref = oracle.quantize_i8_absmax(x)
    q = guarded((B, K), torch.int8)
    s = guarded((B,), torch.float32)
    lb.lb_quantize_i8_absmax(dev(x), q, s, B, K)
    torch.cuda.synchronize()
    assert np.array_equal(host(q), q_ref)
    assert np.array_equal(host(s).view(np.uint32), s_ref.view(np.uint32))


@pytest.mark.parametrize("qk,N,K", [(128, 5, 384), (64, 7, 320), (128, 300, 4096), (64, 129, 4096)])
def test_repack(qk, N, K):
    blocks = synth.q1_0_blocks(N, K, seed=1) if qk == 128 else synth.q2_0_blocks(N, K, seed=2)
    bits, scales = repack_on_gpu(blocks, K, qk)
    torch.cuda.synchronize()
    b_ref, s_ref = oracle.repack(blocks, K, qk)
    assert np.array_equal(host(bits).reshape(N, -1), b_ref)
    assert np.array_equal(host(scales, np.uint16).reshape(N, -1), s_ref)


# ----------------------------------------------------------------------------------------------
# Q1_0 / Q2_0_g64 GEMV
# ----------------------------------------------------------------------------------------------
def _check_q(qk, blocks, q, dx, want_isum=True):
    ref = (oracle.q1_0_product if qk == 128 else oracle.q2_0_g64_product)(blocks, q, dx)
    y, isum = gemv_q(qk, blocks, q, dx, want_isum=want_isum)
    if want_isum:
        assert np.array_equal(isum, ref.isum), "integer block sums differ"
    ok, worst = within(y, ref.y_exact, ref.mag)
    assert ok, f"fp32 output outside the bound (worst err/tol = {worst:.3g})"
    return y, ref


def test_q1_0_tiny_config():
    """Q1_0 GEMV tiny: W 256x512, sign bits p=0.5, fp16 |N(0,0.02)| scales, x N(0,1) -> q8_0,
    batch 1, seed 0."""
    blocks = synth.q1_0_blocks(256, 512, seed=0)
    q, dx = oracle.quantize_q8_0(synth.activations(1, 512, seed=0))
    _check_q(128, blocks, q, dx)


@pytest.mark.parametrize("B", [1, 2, 3, 4, 5, 6, 7, 8])
def test_q1_0_ragged(B):
    N, K = 37, 384 if B % 2 else 4224          # 3 or 33 blocks per row: ragged lane coverage
    blocks = synth.q1_0_blocks(N, K, seed=100 + B)
    q, dx = _q8(B, K, seed=200 + B)
    _check_q(128, blocks, q, dx)


@pytest.mark.parametrize("B", [1, 2, 3, 4, 5, 6, 7, 8])
def test_q2_0_ragged(B):
    N, K = 41, 320 if B % 2 else 4160          # 5 or 65 blocks per row
    blocks = synth.q2_0_blocks(N, K, seed=300 + B, probs=(0.25, 0.25, 0.25, 0.25))
    q, dx = _q8(B, K, seed=400 + B)
    _check_q(64, blocks, q, dx)


@pytest.mark.parametrize("B", [1, 8])
def test_q2_0_config_4096(B):
    """Q2_0_g64 GEMV 4096x4096, codes {-1,0,+1} at 31/38/31 %, batch 1 and 8 (full compare)."""
    blocks = synth.q2_0_blocks(4096, 4096, seed=0)
    q, dx = _q8(B, 4096, seed=1)
    _check_q(64, blocks, q, dx, want_isum=(B == 1))


@pytest.mark.parametrize("qk", [128, 64])
def test_production_path_matches_hooked_path(qk):
    """The production instantiation (no block-sum hook) gives the same outputs."""
    N, K, B = 300, 4096, 2
    blocks = synth.q1_0_blocks(N, K, seed=5) if qk == 128 else synth.q2_0_blocks(N, K, seed=5)
    q, dx = _q8(B, K, seed=6)
    y1, _ = gemv_q(qk, blocks, q, dx, want_isum=True)
    y0, _ = gemv_q(qk, blocks, q, dx, want_isum=False)
    ref = (oracle.q1_0_product if qk == 128 else oracle.q2_0_g64_product)(blocks, q, dx)
    assert within(y0, ref.y_exact, ref.mag)[0]
    assert within(y1, ref.y_exact, ref.mag)[0]


@pytest.mark.parametrize("qk", [128, 64])
def test_minus128_extremes(qk):
    """Hand-built activation blocks of -128/-127/127 codes (never produced by the quantizer,
    accepted by the kernels): the integer sums must stay exact."""
    N, K, B = 33, 1024, 3
    blocks = (synth.q1_0_blocks(N, K, seed=9) if qk == 128
              else synth.q2_0_blocks(N, K, seed=9, probs=(0.3, 0.1, 0.3, 0.3)))
    q = synth.int8_codes(B, K, seed=10, extremes=True)
    q[0] = -128
    dx = synth.q8_scales(B, K, seed=11)
    _check_q(qk, blocks, q, dx)


@pytest.mark.parametrize("qk", [128, 64])
def test_unit_scales_exact(qk):
    """With every scale 1.0 each fp32 partial is an integer below 2^24: y == sum isum exactly."""
    N, K, B = 70, 2048, 2
    one = np.float16(1.0).view(np.uint16)
    nb = K // qk
    sc = np.full((N, nb), one, np.uint16)
    blocks = (synth.q1_0_blocks(N, K, seed=12, scales=sc) if qk == 128
              else synth.q2_0_blocks(N, K, seed=12, scales=sc, probs=(0.25,) * 4))
    q = synth.int8_codes(B, K, seed=13)
    dx = np.full((B, K // 32), one, np.uint16)
    y, isum = gemv_q(qk, blocks, q, dx)
    assert np.array_equal(y.astype(np.int64), isum.astype(np.int64).sum(-1))
    ref = (oracle.q1_0_product if qk == 128 else oracle.q2_0_g64_product)(blocks, q, dx)
    assert np.array_equal(isum, ref.isum)


def test_zero_scales_and_zero_activations():
    N, K, B = 16, 512, 2
    blocks = synth.q2_0_blocks(N, K, seed=14)
    blocks[:, :, :2] = 0                                   # d_w = 0
    q, dx = _q8(B, K, seed=15)
    y, _ = gemv_q(64, blocks, q, dx)
    assert np.all(y == 0.0)
    y2, isum2 = gemv_q(128, synth.q1_0_blocks(N, K, seed=16), np.zeros((B, K), np.int8),
                       np.zeros((B, K // 32), np.uint16))
    assert np.all(y2 == 0.0) and np.all(isum2 == 0)


@pytest.mark.parametrize("qk,name,N,K", [(128, "gate", 12288, 4096), (128, "down", 4096, 12288),
                                         (64, "gate", 12288, 4096), (64, "down", 4096, 12288),
                                         (64, "k", 1024, 4096)])
def test_qwen3_shapes_sampled(qk, name, N, K):
    """Full-size Qwen3-8B projections: the whole GEMV runs on the GPU, sampled rows are compared
    with the oracle."""
    blocks = (synth.q1_0_blocks(N, K, seed=500 + N) if qk == 128
              else synth.q2_0_blocks(N, K, seed=500 + N))
    q, dx = _q8(1, K, seed=501)
    y, isum = gemv_q(qk, blocks, q, dx)
    rows = np.unique(np.concatenate([np.arange(0, N, N // 97), [N - 1]]))
    ref = (oracle.q1_0_product if qk == 128 else oracle.q2_0_g64_product)(blocks[rows], q, dx)
    assert np.array_equal(isum[:, rows], ref.isum)
    assert within(y[:, rows], ref.y_exact, ref.mag)[0]


@pytest.mark.parametrize("G", [1, 16])
def test_q2_4096_batch8_sampled(G):
    """The 4096 x 4096 Q2_0_g64 workload at 8 tokens as the bench runs it: one matrix (32 units:
    the lane-per-row kernel with four row groups) and a group of 16 (512 units: the tensor-core
    kernel); sampled rows of the first and last matrix checked against the oracle."""
    N, K, B = 4096, 4096, 8
    blocks = [synth.q2_0_blocks(N, K, seed=820 + i) for i in (0, G - 1)] if G > 1 else \
        [synth.q2_0_blocks(N, K, seed=820)]
    q, dx = _q8(B, K, seed=821)
    reps = [repack_on_gpu(bl, K, 64) for bl in blocks]
    mats, ys = [], []
    for i in range(G):
        bits, scales = reps[0] if i < G - 1 or G == 1 else reps[-1]
        y = guarded((B, N), torch.float32, float("nan"))
        mats.append((bits, scales, y, None, N))
        ys.append(y)
    lb.lb_gemv_q2_0_g64_grouped(mats, dev(q), dev(dx), K, B)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.arange(0, N, 41), [N - 1]]))
    for bl, y in ((blocks[0], ys[0]), (blocks[-1], ys[-1])):
        ref = oracle.q2_0_g64_product(bl[rows], q, dx, want_isum=False)
        ok, worst = within(host(y)[:, rows], ref.y_exact, ref.mag)
        assert ok, worst


# ----------------------------------------------------------------------------------------------
# planar ternary
# ----------------------------------------------------------------------------------------------
def _check_trit(planes, w_scale, q, xs):
    acc_ref, y_ref = oracle.trit_planes_product(planes, w_scale, q, xs)
    acc, y = gemv_trit(planes, w_scale, q, xs)
    assert np.array_equal(acc, acc_ref)
    assert np.array_equal(y.view(np.uint32), y_ref.view(np.uint32)), "planar y not bit-exact"


@pytest.mark.parametrize("B", [1, 2, 3, 5, 8])
def test_trit_ragged(B):
    N, K = 37, 320 if B % 2 else 4160
    planes, _ = synth.trit_planes(N, K, seed=600 + B)
    q = synth.int8_codes(B, K, seed=601)
    xs = np.abs(synth.activations(1, B, seed=602)[0]) * 0.01 + 1e-3
    _check_trit(planes, synth.w_scale(603), q, xs)


@pytest.mark.parametrize("name,N,K", synth.BITNET_2B4T_PROJ[:2] + synth.BITNET_2B4T_PROJ[4:])
@pytest.mark.parametrize("B", [1, 8])
def test_trit_bitnet_shapes(name, N, K, B):
    """BitNet-2B4T projections, int8 per-token absmax activations (quantized on the GPU)."""
    planes, _ = synth.trit_planes(N, K, seed=700 + N + K)
    x = synth.activations(B, K, seed=701)
    qd = guarded((B, K), torch.int8)
    sd = guarded((B,), torch.float32)
    lb.lb_quantize_i8_absmax(dev(x), qd, sd, B, K)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quantize_i8_absmax(x)
    assert np.array_equal(host(qd), q_ref)
    _check_trit(planes, synth.w_scale(702), q_ref, s_ref)


def test_trit_minus128_extremes():
    K = 2560
    q = np.full((2, K), -128, np.int8)
    q[1] = synth.int8_codes(1, K, seed=9, extremes=True)[0]
    allset = np.uint64(0xFFFFFFFFFFFFFFFF)
    planes = np.zeros((3, K // 64, 2), np.uint64)
    planes[0, :, 0] = allset                      # every column +1
    planes[1, :, 1] = allset                      # every column -1
    planes[2] = synth.trit_planes(1, K, seed=10)[0][0]
    _check_trit(planes, 0.5, q, np.array([1.0, 0.25], np.float32))


# ----------------------------------------------------------------------------------------------
# bf16 head
# ----------------------------------------------------------------------------------------------
@pytest.mark.parametrize("B", [1, 2, 3, 4, 8])
def test_bf16_ragged(B):
    N, K = 37, 328 if B % 2 else 2568
    w = synth.bf16_weights(N, K, seed=800 + B)
    x = synth.activations(B, K, seed=801)
    y_ref, mag = oracle.bf16_product(w, x)
    assert within(gemv_bf16(w, x), y_ref, mag)[0]


@pytest.mark.parametrize("B", [1, 8])
def test_bf16_head_sampled(B):
    """BitNet-2B4T dense head 128256 x 2560 bf16: full GEMV on the GPU, sampled rows checked."""
    N, K = synth.BITNET_HEAD
    w = synth.bf16_weights(N, K, seed=900)
    x = synth.activations(B, K, seed=901)
    y = gemv_bf16(w, x)
    rows = np.unique(np.concatenate([np.arange(0, N, 509), [N - 1]]))
    y_ref, mag = oracle.bf16_product(w[rows], x)
    assert within(y[:, rows], y_ref, mag)[0]


# ----------------------------------------------------------------------------------------------
# grouped GEMVs: several matrices sharing one activation in one launch
# ----------------------------------------------------------------------------------------------
@pytest.mark.parametrize("qk", [128, 64])
@pytest.mark.parametrize("B", [1, 2, 5, 8])
def test_grouped_q(qk, B):
    K = 1280 if qk == 128 else 1088
    Ns = [300, 77, 77, 9, 1, 130]
    make = synth.q1_0_blocks if qk == 128 else synth.q2_0_blocks
    blocks = [make(n, K, seed=1000 + i) for i, n in enumerate(Ns)]
    q, dx = _q8(B, K, seed=1100 + B)
    mats, outs = [], []
    for i, (n, bl) in enumerate(zip(Ns, blocks)):
        bits, scales = repack_on_gpu(bl, K, qk)
        y = guarded((B, n), torch.float32, float("nan"))
        isum = guarded((B, n, K // 32), torch.int32) if i % 2 else None
        mats.append((bits, scales, y, isum, n))
        outs.append((y, isum))
    fn = lb.lb_gemv_q1_0_grouped if qk == 128 else lb.lb_gemv_q2_0_g64_grouped
    fn(mats, dev(q), dev(dx), K, B)
    torch.cuda.synchronize()
    ref_fn = oracle.q1_0_product if qk == 128 else oracle.q2_0_g64_product
    for bl, (y, isum) in zip(blocks, outs):
        ref = ref_fn(bl, q, dx)
        assert within(host(y), ref.y_exact, ref.mag)[0]
        if isum is not None:
            assert np.array_equal(host(isum), ref.isum)
    assert lb.lb_device_status() == 0


def test_grouped_q2_full_group():
    """LB_MAX_GROUP matrices in one launch (tile indexing across the whole group)."""
    K, B = 512, 1
    Ns = [17 + (i * 37) % 90 for i in range(lb.MAX_GROUP)]
    blocks = [synth.q2_0_blocks(n, K, seed=2000 + i) for i, n in enumerate(Ns)]
    q, dx = _q8(B, K, seed=2100)
    mats, ys = [], []
    for n, bl in zip(Ns, blocks):
        bits, scales = repack_on_gpu(bl, K, 64)
        y = guarded((B, n), torch.float32, float("nan"))
        mats.append((bits, scales, y, None, n))
        ys.append(y)
    lb.lb_gemv_q2_0_g64_grouped(mats, dev(q), dev(dx), K, B)
    torch.cuda.synchronize()
    for bl, y in zip(blocks, ys):
        ref = oracle.q2_0_g64_product(bl, q, dx, want_isum=False)
        assert within(host(y), ref.y_exact, ref.mag)[0]


@pytest.mark.parametrize("qk", [128, 64])
def test_long_rows_column_slices(qk):
    """Rows longer than one shared-memory stage are streamed in column slices."""
    K = 65536 if qk == 128 else 32768   # 512 chunks per row: two column slices
    N, B = 45, 1
    blocks = synth.q1_0_blocks(N, K, seed=5) if qk == 128 else synth.q2_0_blocks(N, K, seed=5)
    q, dx = _q8(B, K, seed=6)
    _check_q(qk, blocks, q, dx)


@pytest.mark.parametrize("B", [1, 3, 8])
def test_grouped_trit(B):
    K = 2560
    Ns = [640, 640, 33, 1]
    planes = [synth.trit_planes(n, K, seed=3000 + i)[0] for i, n in enumerate(Ns)]
    q = synth.int8_codes(B, K, seed=3100)
    xs = (np.abs(synth.activations(1, B, seed=3101)[0]) * 0.01 + 1e-3).astype(np.float32)
    mats, outs = [], []
    for i, (n, pl) in enumerate(zip(Ns, planes)):
        y = guarded((B, n), torch.float32, float("nan"))
        acc = guarded((B, n), torch.int32) if i != 1 else None
        mats.append((dev(pl), 0.01 * (i + 1), y, acc, n))
        outs.append((y, acc, 0.01 * (i + 1)))
    lb.lb_gemv_trit_planes_grouped(mats, dev(q), dev(xs), K, B)
    torch.cuda.synchronize()
    for pl, (y, acc, ws) in zip(planes, outs):
        acc_ref, y_ref = oracle.trit_planes_product(pl, ws, q, xs)
        assert np.array_equal(host(y).view(np.uint32), y_ref.view(np.uint32))
        if acc is not None:
            assert np.array_equal(host(acc), acc_ref)


def test_device_status_clean():
    assert lb.lb_device_status() == 0


@pytest.mark.parametrize("qk", [128, 64])
@pytest.mark.parametrize("B", [3, 5, 8])
def test_q_batched_ragged_production(qk, B):
    """Batch 3..8 without the block-sum hook (the lane-per-row kernel): ragged row count (not a
    multiple of 32), long rows sliced into several stages, and short rows."""
    for N, K in ((77, 1024 if qk == 128 else 320), (45, 12288)):
        blocks = synth.q1_0_blocks(N, K, seed=600 + B) if qk == 128 else synth.q2_0_blocks(
            N, K, seed=600 + B, probs=(0.25, 0.25, 0.25, 0.25))
        q, dx = _q8(B, K, seed=610 + B)
        ref = (oracle.q1_0_product if qk == 128 else oracle.q2_0_g64_product)(blocks, q, dx)
        y, _ = gemv_q(qk, blocks, q, dx, want_isum=False)
        assert within(y, ref.y_exact, ref.mag)[0]


@pytest.mark.parametrize("qk", [128, 64])
@pytest.mark.parametrize("N", [2500, 3500, 5000])
def test_q_batched_row_groups(qk, N):
    """Lane-per-row kernel with four row groups per warp (2500 rows: 79 units of 32), two (3500
    rows: 110 units) and one (5000 rows: 157 units); K is not a multiple of 256, so the
    tensor-core kernel is not taken."""
    K, B = (384 if qk == 128 else 320), 5
    blocks = synth.q1_0_blocks(N, K, seed=680) if qk == 128 else synth.q2_0_blocks(
        N, K, seed=680, probs=(0.25, 0.25, 0.25, 0.25))
    q, dx = _q8(B, K, seed=681)
    ref = (oracle.q1_0_product if qk == 128 else oracle.q2_0_g64_product)(blocks, q, dx,
                                                                          want_isum=False)
    y, _ = gemv_q(qk, blocks, q, dx, want_isum=False)
    ok, worst = within(y, ref.y_exact, ref.mag)
    assert ok, worst


@pytest.mark.parametrize("N", [2500, 3500])
def test_trit_batched_row_groups(N):
    """Planar down-projection shape (K = 6912) with four and two row groups per warp: bit-exact."""
    K, B = 6912, 8
    planes, _ = synth.trit_planes(N, K, seed=690)
    x = synth.activations(B, K, seed=691)
    qi, xs = oracle.quantize_i8_absmax(x)
    acc_ref, y_ref = oracle.trit_planes_product(planes, 0.0173, qi, xs)
    acc, y = gemv_trit(planes, 0.0173, qi, xs)
    assert np.array_equal(acc, acc_ref)
    assert np.array_equal(y.view(np.uint32), y_ref.view(np.uint32))


def _tc_group_rows():
    """Rows of a grouped call large enough (>= 64 units of 128 rows) for the tensor-core kernel:
    31 ragged matrices of 130 rows, one of 77 and one of a single row (65 units)."""
    return [130] * 31 + [77, 1]


def _q_group(qk, Ns, K, B, seed):
    blocks = (synth.q1_0_blocks(sum(Ns), K, seed=seed) if qk == 128 else
              synth.q2_0_blocks(sum(Ns), K, seed=seed, probs=(0.25, 0.25, 0.25, 0.25)))
    q, dx = _q8(B, K, seed=seed + 1)
    bits, scales = repack_on_gpu(blocks, K, qk)
    per_bits, per_sc = K // qk * 16, lb.scale_stride(K, qk)
    mats, outs, r0 = [], [], 0
    for n in Ns:
        y = guarded((B, n), torch.float32, float("nan"))
        mats.append((bits[r0 * per_bits:(r0 + n) * per_bits], scales[r0 * per_sc:(r0 + n) * per_sc],
                     y, None, n))
        outs.append((blocks[r0:r0 + n], y))
        r0 += n
    fn = lb.lb_gemv_q1_0_grouped if qk == 128 else lb.lb_gemv_q2_0_g64_grouped
    fn(mats, dev(q), dev(dx), K, B)
    torch.cuda.synchronize()
    return q, dx, outs


@pytest.mark.parametrize("qk", [128, 64])
@pytest.mark.parametrize("B", [3, 4, 5, 8])
@pytest.mark.parametrize("K", [1024, 4096])
def test_q_batched_tensor_core(qk, B, K):
    """A grouped call with >= 64 row units and K a multiple of 256 up to the resident maximum
    4096 at 3..8 tokens: the tensor-core kernel from 4 tokens (Q2_0_g64) or 5 (Q1_0), the
    lane-per-row kernel below; every matrix, ragged ones and a single row included, within the
    GEMV bound of the oracle."""
    q, dx, outs = _q_group(qk, _tc_group_rows(), K, B, seed=640 + B + K)
    prod = oracle.q1_0_product if qk == 128 else oracle.q2_0_g64_product
    for blocks, y in outs:
        ref = prod(blocks, q, dx, want_isum=False)
        ok, worst = within(host(y), ref.y_exact, ref.mag)
        assert ok, worst


@pytest.mark.parametrize("B", [3, 4, 5, 8])
def test_trit_batched_tensor_core(B):
    """Planar at batch 3..8 in a grouped call with >= 64 row units (the tensor-core kernel from 5
    tokens, the lane-per-row kernel below): bit-exact accumulators and outputs for every matrix."""
    Ns, K = _tc_group_rows(), 2560
    planes, _ = synth.trit_planes(sum(Ns), K, seed=660 + B)
    x = synth.activations(B, K, seed=670 + B)
    qi, xs = oracle.quantize_i8_absmax(x)
    mats, outs, r0 = [], [], 0
    for n in Ns:
        y = guarded((B, n), torch.float32, float("nan"))
        acc = guarded((B, n), torch.int32)
        mats.append((dev(planes[r0:r0 + n]), 0.0173, y, acc, n))
        outs.append((planes[r0:r0 + n], y, acc))
        r0 += n
    lb.lb_gemv_trit_planes_grouped(mats, dev(qi), dev(xs), K, B)
    torch.cuda.synchronize()
    for pl, y, acc in outs:
        acc_ref, y_ref = oracle.trit_planes_product(pl, 0.0173, qi, xs)
        assert np.array_equal(host(acc), acc_ref)
        assert np.array_equal(host(y).view(np.uint32), y_ref.view(np.uint32))


@pytest.mark.parametrize("B", [3, 8])
def test_trit_batched_ragged(B):
    """Planar at batch 3..8 (lane-per-row kernel): bit-exact accumulators and outputs, ragged
    rows, a sliced long row."""
    for N, K in ((77, 2560), (33, 6912)):
        planes, _ = synth.trit_planes(N, K, seed=620 + B)
        x = synth.activations(B, K, seed=630 + B)
        qi, xs = oracle.quantize_i8_absmax(x)
        acc_ref, y_ref = oracle.trit_planes_product(planes, 0.0173, qi, xs)
        acc, y = gemv_trit(planes, 0.0173, qi, xs)
        assert np.array_equal(acc, acc_ref)
        assert np.array_equal(y.view(np.uint32), y_ref.view(np.uint32))
