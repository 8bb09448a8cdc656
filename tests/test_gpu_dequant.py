"""GPU parity of the dequantization kernels (Q1_0, Q2_0_g64 from the repacked planes; planar
beats) against the CPU oracle: every weight as the binary32 (float)w * d, bit for bit, and its
bf16 rounding (nearest, ties to even), bit for bit.  Shapes: one block, ragged row counts, the
full 4096 x 4096 matrix; scales: random, negative (signed zeros for w = 0), fp16 subnormals,
zero; codes including +2."""
import numpy as np
import pytest
import torch

import bit_matvec_lb_gb300 as lb
import oracle
import synth
from gpu_util import dev, guarded, host, repack_on_gpu

pytestmark = pytest.mark.gpu


def _run(fn, args, N, K, fmt):
    dtype = torch.float32 if fmt == lb.OUT_F32 else torch.int16
    out = guarded((N, K), dtype, -1)
    fn(*args, N, K, fmt, out)
    torch.cuda.synchronize()
    return host(out, np.uint32 if fmt == lb.OUT_F32 else np.uint16)


def _check_q(qk, blocks, K):
    N = blocks.shape[0]
    bits, scales = repack_on_gpu(blocks, K, qk)
    fn = lb.lb_dequantize_q1_0 if qk == 128 else lb.lb_dequantize_q2_0_g64
    f32 = _run(fn, (bits, scales), N, K, lb.OUT_F32)
    assert np.array_equal(f32, oracle.dequant(blocks, K, qk).view(np.uint32))
    bf = _run(fn, (bits, scales), N, K, lb.OUT_BF16)
    assert np.array_equal(bf, oracle.dequant_bf16(blocks, K, qk))


@pytest.mark.parametrize("qk", [128, 64])
@pytest.mark.parametrize("N,K", [(1, 128), (3, 384), (257, 1152), (130, 4224)])
def test_dequant_q_ragged(qk, N, K):
    kw = {} if qk == 128 else {"probs": (0.25, 0.25, 0.25, 0.25)}
    blocks = (synth.q1_0_blocks if qk == 128 else synth.q2_0_blocks)(N, K, seed=N + K, **kw)
    _check_q(qk, blocks, K)


@pytest.mark.parametrize("qk", [128, 64])
def test_dequant_q_special_scales(qk):
    """Negative scales (w = 0 gives -0), fp16 subnormals, zero and the largest finite scale."""
    N, K = 64, 1024
    g = synth.rng(7)
    sc = g.integers(0, 0x10000, size=(N, K // qk)).astype(np.uint16)
    sc = np.where((sc & 0x7C00) == 0x7C00, sc & 0x83FF, sc).astype(np.uint16)  # finite only
    sc[0, :] = 0x0001           # smallest subnormal
    sc[1, :] = 0x8000           # -0
    sc[2, :] = 0x7BFF           # 65504
    sc[3, :] = 0xFBFF           # -65504 (times +2 still finite in fp32; bf16 rounds it)
    kw = {} if qk == 128 else {"probs": (0.25, 0.25, 0.25, 0.25)}
    blocks = (synth.q1_0_blocks if qk == 128 else synth.q2_0_blocks)(N, K, seed=8, scales=sc, **kw)
    _check_q(qk, blocks, K)


def test_dequant_q2_full_size():
    N = K = 4096
    blocks = synth.q2_0_blocks(N, K, seed=9)
    _check_q(64, blocks, K)


@pytest.mark.parametrize("N,K,w", [(1, 64, 0.02), (7, 192, -0.75), (300, 2560, 0.0173),
                                   (2560, 6912, 3.0e-3)])
def test_dequant_trit(N, K, w):
    planes, _ = synth.trit_planes(N, K, seed=N + K)
    pd = dev(planes)
    ref = oracle.trit_planes_dequant(planes, w, K)
    f32 = _run(lb.lb_dequantize_trit_planes, (pd, w), N, K, lb.OUT_F32)
    assert np.array_equal(f32, ref.view(np.uint32))
    bf = _run(lb.lb_dequantize_trit_planes, (pd, w), N, K, lb.OUT_BF16)
    assert np.array_equal(bf, oracle.f32_to_bf16(ref))


def test_dequant_device_status_clean():
    assert lb.lb_device_status() == 0
