"""lb_gemm_q2_0_g64_noalloc: the Q2_0_g64 prefill GEMM with the library's fixed scratch instead
of a caller workspace.  Its results must equal lb_gemm_q2_0_g64's bit for bit (same kernels on
the same inputs), on two calls in a row of different shapes, whether this file runs alone or
after the rest of the suite."""
import ctypes

import numpy as np
import pytest

import bit_matvec_lb_gb300 as lb
import oracle
import synth

A = 0x10000  # 16-byte aligned fake device address (never dereferenced)


def test_noalloc_refuses_oversize_and_null_on_host():
    f = lb.load().lb_gemm_q2_0_g64_noalloc
    assert f(None, A, A, A, A, 128, 64, 4096, None) == -1
    # 512 tokens x 12288 columns need 12 MiB of converted activations: above the 8 MiB scratch
    assert f(A, A, A, A, A, 512, 64, 12288, None) == -3
    # 257 tokens round up to 384 rows: 384 x 11008 x 2 B > 8 MiB, while 384 x 10880 x 2 B fits
    assert f(A, A, A, A, A, 257, 64, 11008, None) == -3
    assert f(A, A, A, A, A, 0, 64, 4096, None) == -3


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_two_calls():
    import torch
    from gpu_util import dev, guarded, repack_on_gpu, within

    results = []
    # the last shape fills the scratch exactly: round_up(512, 128) * 8192 * 2 B = 8 MiB
    for (M, N, K, seed) in ((130, 300, 2048, 1), (512, 4096, 4096, 2), (512, 640, 8192, 3)):
        blocks = synth.q2_0_blocks(N, K, seed=900 + seed)
        bits, scales = repack_on_gpu(blocks, K, 64)
        q, dx = oracle.quantize_q8_0(synth.activations(M, K, seed=910 + seed))
        qd, dd = dev(q), dev(dx)
        y0 = guarded((M, N), torch.float32, float("nan"))
        y1 = guarded((M, N), torch.float32, float("nan"))
        ws = guarded(lb.lb_gemm_workspace_bytes(M, K), torch.uint8)
        lb.lb_gemm_q2_0_g64(bits, scales, qd, dd, y0, M, N, K, ws)
        lb.lb_gemm_q2_0_g64_noalloc(bits, scales, qd, dd, y1, M, N, K)
        torch.cuda.synchronize()
        results.append((blocks, q, dx, y0.cpu().numpy(), y1.cpu().numpy()))
    for blocks, q, dx, y0, y1 in results:
        assert np.array_equal(y0.view(np.uint32), y1.view(np.uint32))
    blocks, q, dx, _, y1 = results[0]
    ref = oracle.q2_0_g64_product(blocks, q, dx, want_isum=False)
    assert within(y1, ref.y_exact, ref.mag)[0]
    assert lb.lb_device_status() == 0
