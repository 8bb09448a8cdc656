"""GPU parity of base-3 packing (five trits per byte) and of the decode GEMV on it, against the
CPU oracle: the packed bytes bit for bit, the integer accumulators and the fp32 outputs bit for
bit (planar arithmetic: exact integers, two fixed roundings), and equal to the planar GEMV on
the same trits.  Shapes: one beat, groups that straddle planar beats, K not a multiple of 80
(a padded last group), BitNet-2B4T projections, every batch size 1..8, -128 activations."""
import numpy as np
import pytest
import torch

import bit_matvec_lb_gb300 as lb
import oracle
import synth
from gpu_util import dev, guarded, host

pytestmark = pytest.mark.gpu


def pack_gpu(planes, K):
    N = planes.shape[0]
    packed = guarded((N, lb.base3_row_bytes(K)), torch.uint8, 255)
    lb.lb_pack_base3(dev(planes), N, K, packed)
    torch.cuda.synchronize()
    return packed


def gemv_b3(packed, w_scale, q, xs, N, K):
    B = q.shape[0]
    y = guarded((B, N), torch.float32, float("nan"))
    acc = guarded((B, N), torch.int32, -7)
    lb.lb_gemv_base3(packed, w_scale, dev(q), dev(np.asarray(xs, np.float32)), y, acc, N, K, B)
    torch.cuda.synchronize()
    return host(acc), host(y)


@pytest.mark.parametrize("N,K", [(1, 64), (3, 320), (33, 1152), (257, 2560), (130, 6912)])
def test_pack_base3(N, K):
    planes, _ = synth.trit_planes(N, K, seed=N + K)
    assert np.array_equal(host(pack_gpu(planes, K)), oracle.base3_pack(planes, K))


@pytest.mark.parametrize("B", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("N,K", [(1, 64), (37, 1216), (300, 2560), (129, 6912)])
def test_gemv_base3(B, N, K):
    planes, _ = synth.trit_planes(N, K, seed=3 * N + K + B)
    q, xs = oracle.quantize_i8_absmax(synth.activations(B, K, seed=B + K))
    packed = pack_gpu(planes, K)
    acc, y = gemv_b3(packed, 0.0173, q, xs, N, K)
    acc_ref, y_ref = oracle.base3_product(oracle.base3_pack(planes, K), 0.0173, q, xs)
    assert np.array_equal(acc, acc_ref)
    assert np.array_equal(y.view(np.uint32), y_ref.view(np.uint32))


def test_gemv_base3_extremes_and_planar_equality():
    """Activations from {-128, -127, 127} (and a row of -128) against mostly nonzero trits: the
    base-3 GEMV equals the oracle and the planar GEMV on the same trits, bit for bit."""
    N, K, B = 200, 2560 + 64, 8
    planes, _ = synth.trit_planes(N, K, seed=77, probs=(0.45, 0.1, 0.45))
    q = synth.int8_codes(B, K, seed=78, extremes=True)
    q[0] = -128
    xs = np.linspace(0.001, 2.0, B).astype(np.float32)
    acc, y = gemv_b3(pack_gpu(planes, K), 1.0, q, xs, N, K)
    acc_ref, y_ref = oracle.base3_product(oracle.base3_pack(planes, K), 1.0, q, xs)
    assert np.array_equal(acc, acc_ref) and np.array_equal(y.view(np.uint32), y_ref.view(np.uint32))
    yp = guarded((B, N), torch.float32)
    ap = guarded((B, N), torch.int32)
    lb.lb_gemv_trit_planes(dev(planes), 1.0, dev(q), dev(xs), yp, ap, N, K, B)
    torch.cuda.synchronize()
    assert np.array_equal(acc, host(ap)) and np.array_equal(y.view(np.uint32),
                                                            host(yp).view(np.uint32))


def test_gemv_base3_large_rows_sampled():
    """A 4096 x 16384 matrix (many rows per warp, many groups per lane), sampled rows."""
    N, K, B = 4096, 16384, 2
    planes, _ = synth.trit_planes(N, K, seed=81)
    q, xs = oracle.quantize_i8_absmax(synth.activations(B, K, seed=82))
    acc, y = gemv_b3(pack_gpu(planes, K), 0.02, q, xs, N, K)
    rows = np.unique(np.concatenate([np.arange(0, N, 61), [N - 1]]))
    acc_ref, y_ref = oracle.base3_product(oracle.base3_pack(planes[rows], K), 0.02, q, xs)
    assert np.array_equal(acc[:, rows], acc_ref)
    assert np.array_equal(y[:, rows].view(np.uint32), y_ref.view(np.uint32))


def test_base3_device_status_clean():
    assert lb.lb_device_status() == 0
