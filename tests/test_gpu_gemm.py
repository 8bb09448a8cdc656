"""GPU parity of the prefill GEMMs (Q1_0 / Q2_0_g64 weights x q8_0 activations of M tokens,
on the tensor cores) against the CPU oracle.

Bar: |y - exact| <= 1e-5 * sum|d_w d_x isum| + 1e-6 for every output, where exact is the
real-number value the oracle computes in fp64.  Where every partial is an integer (unit scales)
or a single exact partial (one activation block), the output must equal it bit for bit.  Sizes
span several 128 x 128 tiles with ragged tails in M and N, K deep enough to need several
accumulation segments, the degenerate cases (code +2 with -128 activations at the largest
integer block sum, subnormal and zero weight scales), and the full prefill shapes (512 tokens,
sampled rows).
"""
import numpy as np
import pytest
import torch

import bit_matvec_lb_gb300 as lb
import oracle
import synth
from gpu_util import dev, gemm_q, guarded, repack_on_gpu, within

pytestmark = pytest.mark.gpu


def _blocks(qk, N, K, seed, **kw):
    return synth.q1_0_blocks(N, K, seed=seed, **kw) if qk == 128 else synth.q2_0_blocks(
        N, K, seed=seed, **kw)


def _ref(qk, blocks, q, dx):
    return (oracle.q1_0_product if qk == 128 else oracle.q2_0_g64_product)(blocks, q, dx)


def _check(qk, blocks, q, dx, **kw):
    y = gemm_q(qk, blocks, q, dx, **kw)
    ref = _ref(qk, blocks, q, dx)
    ok, worst = within(y, ref.y_exact, ref.mag)
    assert ok, f"fp32 output outside the bound (worst err/tol = {worst:.3g})"
    return y, ref


@pytest.mark.parametrize("qk", [128, 64])
@pytest.mark.parametrize("M,N,K", [(1, 1, 128), (5, 7, 384), (128, 128, 1024), (130, 257, 1152),
                                   (300, 200, 2048), (257, 129, 4224)])
def test_gemm_ragged(qk, M, N, K):
    probs = (0.25, 0.25, 0.25, 0.25)
    blocks = _blocks(qk, N, K, seed=M + N + K, **({} if qk == 128 else {"probs": probs}))
    q, dx = oracle.quantize_q8_0(synth.activations(M, K, seed=M * 3 + K))
    _check(qk, blocks, q, dx)


@pytest.mark.parametrize("qk", [128, 64])
def test_gemm_unit_scales_exact(qk):
    """All scales 1.0: every partial is an integer and the sums stay below 2^24, so y equals
    the integer sum exactly."""
    M, N, K = 140, 150, 2048
    one = np.float16(1.0).view(np.uint16)
    sc = np.full((N, K // qk), one, np.uint16)
    blocks = _blocks(qk, N, K, seed=21, scales=sc,
                     **({} if qk == 128 else {"probs": (0.25,) * 4}))
    q = synth.int8_codes(M, K, seed=22)
    dx = np.full((M, K // 32), one, np.uint16)
    y = gemm_q(qk, blocks, q, dx)
    ref = _ref(qk, blocks, q, dx)
    assert np.array_equal(y.astype(np.float64), ref.y_exact)
    assert np.array_equal(y.astype(np.int64), ref.isum.astype(np.int64).sum(-1))


def test_gemm_q2_largest_block_sum_exact():
    """Code 3 (weight +2) against -128 everywhere gives |isum| = 8192, the largest block sum,
    times a scale with a full 11-bit significand: the tensor-core partial d_w * isum needs all
    24 bits of binary32.  With d_x = 1 on the first block and 0 on the second, y is that single
    partial and must be exact."""
    M, N, K = 130, 140, 64
    g = synth.rng(31)
    sc = (0x3800 + g.integers(0, 0x400, size=(N, 1))).astype(np.uint16)  # [0.5, 1) full mantissa
    sc[0, 0] = 0x3BFF
    codes = np.full((N, 1, 64), 3, np.uint8)
    codes[1::2, 0, ::3] = 0                                             # some -1 weights too
    blocks = synth.q2_0_blocks(N, K, seed=31, codes=codes, scales=sc)
    q = np.full((M, K), -128, np.int8)
    q[1::2, ::5] = 127
    dx = np.zeros((M, 2), np.uint16)
    dx[:, 0] = np.float16(1.0).view(np.uint16)
    y = gemm_q(64, blocks, q, dx)
    ref = _ref(64, blocks, q, dx)
    assert np.abs(ref.isum).max() == 8192
    assert np.array_equal(y.astype(np.float64), ref.y_exact)


@pytest.mark.parametrize("qk", [128, 64])
def test_gemm_minus128_extremes(qk):
    M, N, K = 131, 133, 1024
    blocks = _blocks(qk, N, K, seed=41, **({} if qk == 128 else {"probs": (0.3, 0.1, 0.3, 0.3)}))
    q = synth.int8_codes(M, K, seed=42, extremes=True)
    q[0] = -128
    dx = synth.q8_scales(M, K, seed=43)
    _check(qk, blocks, q, dx)


@pytest.mark.parametrize("qk", [128, 64])
def test_gemm_subnormal_weight_scales(qk):
    """fp16 subnormal weight scales (0x0001..0x03FF) are exact tensor-core operands; with unit
    activation scales the outputs are far above the absolute slack, so flushing them to zero
    would fail the relative bound."""
    M, N, K = 129, 130, 1024
    g = synth.rng(51)
    sc = g.integers(1, 0x400, size=(N, K // qk)).astype(np.uint16)
    blocks = _blocks(qk, N, K, seed=51, scales=sc)
    q = synth.int8_codes(M, K, seed=52)
    dx = np.full((M, K // 32), np.float16(1.0).view(np.uint16), np.uint16)
    y = gemm_q(qk, blocks, q, dx)
    ref = _ref(qk, blocks, q, dx)
    assert np.abs(ref.y_exact).max() > 1e-3
    assert within(y, ref.y_exact, ref.mag, abs_=0.0)[0]


def test_gemm_zero_scales_and_zero_activations():
    M, N, K = 140, 70, 512
    blocks = synth.q2_0_blocks(N, K, seed=61)
    blocks[:, :, :2] = 0
    q, dx = oracle.quantize_q8_0(synth.activations(M, K, seed=62))
    assert np.all(gemm_q(64, blocks, q, dx) == 0.0)
    y = gemm_q(128, synth.q1_0_blocks(N, K, seed=63), np.zeros((M, K), np.int8),
               np.zeros((M, K // 32), np.uint16))
    assert np.all(y == 0.0)


@pytest.mark.parametrize("qk", [128, 64])
def test_gemm_workspace_reused(qk):
    """Two calls in a row share one workspace (different M, same K): both are right."""
    N, K = 200, 2048
    blocks = _blocks(qk, N, K, seed=71)
    rep = repack_on_gpu(blocks, K, qk)
    ws = guarded(lb.lb_gemm_workspace_bytes(300, K), torch.uint8)
    for M, seed in ((300, 72), (77, 73)):
        q, dx = oracle.quantize_q8_0(synth.activations(M, K, seed=seed))
        y = gemm_q(qk, blocks, q, dx, workspace=ws, repacked=rep)
        ref = _ref(qk, blocks, q, dx)
        assert within(y, ref.y_exact, ref.mag)[0]


@pytest.mark.parametrize("qk,name,N,K", [(128, "q", 4096, 4096), (128, "down", 4096, 12288),
                                         (64, "gate", 12288, 4096), (64, "down", 4096, 12288),
                                         (64, "k", 1024, 4096)])
def test_gemm_prefill_shapes_sampled(qk, name, N, K):
    """512-token prefill through the full-size Qwen3-8B projections: the whole GEMM runs on
    the GPU; every token is compared with the oracle on rows sampled from every 128-row tile."""
    M = synth.PREFILL_M
    blocks = _blocks(qk, N, K, seed=800 + N + K)
    q, dx = oracle.quantize_q8_0(synth.activations(M, K, seed=801))
    y = gemm_q(qk, blocks, q, dx)
    rows = np.unique(np.concatenate([np.arange(0, N, 127), [127, 128, N - 1]]))
    ref = _ref(qk, blocks[rows], q, dx)
    ok, worst = within(y[:, rows], ref.y_exact, ref.mag)
    assert ok, f"worst err/tol = {worst:.3g}"


@pytest.mark.parametrize("qk", [128, 64])
def test_gemm_grouped(qk):
    """Grouped call: three ragged matrices (130, 1, 257 rows) sharing one activation of 130
    tokens; every output within the bound of the oracle and bit-identical to the single-matrix
    call on the same weights."""
    M, K, Ns = 130, 1152 if qk == 128 else 1216, (130, 1, 257)
    q, dx = oracle.quantize_q8_0(synth.activations(M, K, seed=940))
    ws = guarded(lb.lb_gemm_workspace_bytes(M, K), torch.uint8)
    mats, outs = [], []
    for i, n in enumerate(Ns):
        blocks = _blocks(qk, n, K, seed=950 + i)
        bits, scales = repack_on_gpu(blocks, K, qk)
        y = guarded((M, n), torch.float32, float("nan"))
        mats.append((bits, scales, y, n))
        outs.append((blocks, bits, scales, y))
    fn = lb.lb_gemm_q1_0_grouped if qk == 128 else lb.lb_gemm_q2_0_g64_grouped
    fn(mats, dev(q), dev(dx), M, K, ws)
    torch.cuda.synchronize()
    for blocks, bits, scales, y in outs:
        ref = _ref(qk, blocks, q, dx)
        ok, worst = within(y.cpu().numpy(), ref.y_exact, ref.mag)
        assert ok, worst
        y1 = gemm_q(qk, blocks, q, dx, repacked=(bits, scales))
        assert np.array_equal(y.cpu().numpy().view(np.uint32), y1.view(np.uint32))


def test_gemm_device_status_clean():
    assert lb.lb_device_status() == 0
