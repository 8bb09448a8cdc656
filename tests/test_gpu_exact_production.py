"""Unit scales pin the production GEMV binaries' integer paths bit for bit.

With every fp16 scale equal to 1.0 (d_w = d_x = 1) each fp32 partial the kernels form is an
integer below 2^24, so any exact-rounding order gives y == sum over q8_0 blocks of isum, with
isum the oracle's integer block sums ("bankml: verified low-bit inference on commodity CPUs -- a
technical report", III.2-III.3 and III.5: integer block sums, then the scales).  These calls pass
no block-sum output, so they run the instantiations the bench times (no block-sum hook):

  * 1-2 tokens            -> the streaming kernel,
  * 3-8 tokens, K > 4096  -> the lane-per-row kernel,
  * 4-8 tokens (Q2_0_g64) or 5-8 (Q1_0), K % 256 == 0, K <= 4096, >= 64 row units of 128
    -> the tensor-core kernel (3 tokens, and 4 for Q1_0, -> the lane-per-row kernel).

Planar outputs are bit-exact at every scale (their parity tests already compare bit patterns).
"""
import numpy as np
import pytest
import torch

import bit_matvec_lb_gb300 as lb
import oracle
import synth
from gpu_util import dev, guarded, host, repack_on_gpu

pytestmark = pytest.mark.gpu

ONE = np.float16(1.0).view(np.uint16)


def _unit_blocks(qk, N, K, seed):
    sc = np.full((N, K // qk), ONE, np.uint16)
    if qk == 128:
        return synth.q1_0_blocks(N, K, seed=seed, scales=sc)
    return synth.q2_0_blocks(N, K, seed=seed, scales=sc, probs=(0.25,) * 4)


def _expect(qk, blocks, q):
    dx = np.full((q.shape[0], q.shape[1] // 32), ONE, np.uint16)
    ref = (oracle.q1_0_product if qk == 128 else oracle.q2_0_g64_product)(blocks, q, dx)
    return ref.isum.astype(np.int64).sum(-1), dx


def _run_group(qk, Ns, blocks, q, dx):
    """One grouped call over consecutive row ranges of `blocks` (no block-sum output)."""
    B, K = q.shape
    bits, scales = repack_on_gpu(blocks, K, qk)
    per_bits, per_sc = K // qk * 16, lb.scale_stride(K, qk)
    mats, ys, r0 = [], [], 0
    for n in Ns:
        y = guarded((B, n), torch.float32, float("nan"))
        mats.append((bits[r0 * per_bits:(r0 + n) * per_bits],
                     scales[r0 * per_sc:(r0 + n) * per_sc], y, None, n))
        ys.append(y)
        r0 += n
    fn = lb.lb_gemv_q1_0_grouped if qk == 128 else lb.lb_gemv_q2_0_g64_grouped
    fn(mats, dev(q), dev(dx), K, B)
    torch.cuda.synchronize()
    return np.concatenate([host(y) for y in ys], axis=1)


@pytest.mark.parametrize("qk", [128, 64])
@pytest.mark.parametrize("B", [1, 2])
@pytest.mark.parametrize("K", [4096, 12288])
def test_unit_scales_streaming_kernel(qk, B, K):
    N = 203
    blocks = _unit_blocks(qk, N, K, seed=7000 + K + B)
    q = synth.int8_codes(B, K, seed=7100 + B)
    want, dx = _expect(qk, blocks, q)
    y = _run_group(qk, [N], blocks, q, dx)
    assert np.array_equal(y.astype(np.int64), want)
    assert np.all(y == want.astype(np.float32))


@pytest.mark.parametrize("qk", [128, 64])
@pytest.mark.parametrize("B", [3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("K", [6912, 12288])
def test_unit_scales_lane_per_row_kernel(qk, B, K):
    if qk == 128 and K % 128:
        pytest.skip("Q1_0 needs K % 128 == 0")
    N = 77
    blocks = _unit_blocks(qk, N, K, seed=7200 + K + B)
    q = synth.int8_codes(B, K, seed=7300 + B)
    want, dx = _expect(qk, blocks, q)
    y = _run_group(qk, [N], blocks, q, dx)
    assert np.array_equal(y.astype(np.int64), want)


@pytest.mark.parametrize("qk", [128, 64])
@pytest.mark.parametrize("B", [3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("K", [1024, 4096])
def test_unit_scales_tensor_core_kernel(qk, B, K):
    Ns = [130] * 31 + [77, 1]          # 65 row units of 128: the tensor-core kernel from 4-5 tokens
    blocks = _unit_blocks(qk, sum(Ns), K, seed=7400 + K + B)
    q = synth.int8_codes(B, K, seed=7500 + B)
    want, dx = _expect(qk, blocks, q)
    y = _run_group(qk, Ns, blocks, q, dx)
    assert np.array_equal(y.astype(np.int64), want)
    assert lb.lb_device_status() == 0


def test_unit_scales_streaming_q1_eight_rows_per_warp():
    """A one-token Q1_0 call with enough 64-row tiles (601 of them, against 1201 of 32 rows, for
    304 CTA slots: 2 waves x 7/4 < 4 waves) takes the eight-rows-per-warp streaming kernel; with
    unit scales its outputs equal the integer block sums bit for bit, ragged last tile included."""
    K = 256
    Ns = [3840] * 9 + [3841]
    blocks = _unit_blocks(128, sum(Ns), K, seed=7600)
    q = synth.int8_codes(1, K, seed=7601)
    want, dx = _expect(128, blocks, q)
    y = _run_group(128, Ns, blocks, q, dx)
    assert np.array_equal(y.astype(np.int64), want)
    assert lb.lb_device_status() == 0
