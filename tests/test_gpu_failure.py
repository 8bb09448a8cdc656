"""Failure detection without a GPU fault: a bounded wait that runs out is reported, not hung.

Every wait in the library's kernels gives up after a limit and sets the per-device error word
that lb_device_status() reads (refuse with the reason, never fall back silently: "bankml:
verified low-bit inference on commodity CPUs -- a technical report", III.1; tritium.technology
"Architecture", 4.2).  lb_test_inject_wait_timeout makes the next streaming GEMV starve its first
CTA of weights, so that CTA's consumers give up after a few milliseconds.  Nothing faults, traps
or hangs; the context stays usable and the next call is correct with a clean status.
"""
import numpy as np
import pytest
import torch

import bit_matvec_lb_gb300 as lb
import oracle
import synth
from gpu_util import dev, guarded, host, repack_on_gpu, within

pytestmark = pytest.mark.gpu

LB_ERR_DEVICE = -7


def _call(bits, scales, q, dx, N, K, B):
    y = guarded((B, N), torch.float32, float("nan"))
    lb.lb_gemv_q2_0_g64(bits, scales, dev(q), dev(dx), y, None, N, K, B)
    return y


@pytest.mark.parametrize("B,N,K", [(1, 300, 1024),    # streaming kernel
                                   (5, 77, 1024)])    # lane-per-row kernel
def test_bounded_wait_runs_out_and_is_reported(B, N, K):
    assert lb.lb_device_status() == 0
    blocks = synth.q2_0_blocks(N, K, seed=8800 + B)
    q, dx = oracle.quantize_q8_0(synth.activations(B, K, seed=8810 + B))
    bits, scales = repack_on_gpu(blocks, K, 64)
    ref = oracle.q2_0_g64_product(blocks, q, dx, want_isum=False)

    lb.lb_test_inject_wait_timeout(3000)              # 3 ms instead of about 2 s
    y = _call(bits, scales, q, dx, N, K, B)           # enqueues normally: the error is on device
    assert lb.lb_device_status() == LB_ERR_DEVICE     # reported ...
    assert lb.lb_device_status() == 0                 # ... and cleared by the read
    yh = host(y)
    starved = np.isnan(yh)
    assert starved.any() and not starved.all()        # the first CTA's rows stay unwritten
    assert within(np.where(starved, 0.0, yh), np.where(starved, 0.0, ref.y_exact), ref.mag)[0]

    # the hook is one-shot: the same call again is complete and correct, with a clean status
    y2 = _call(bits, scales, q, dx, N, K, B)
    torch.cuda.synchronize()
    assert lb.lb_device_status() == 0
    ok, worst = within(host(y2), ref.y_exact, ref.mag)
    assert ok, worst
