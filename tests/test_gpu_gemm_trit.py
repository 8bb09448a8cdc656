"""GPU parity of the planar ternary prefill GEMM (lb_gemm_trit_planes, tensor cores) against the
CPU oracle.

Bar: bit-exact.  The integer accumulators are exact by construction (every partial sum is an
integer below 2^24 in magnitude), and y = (float(acc) * x_scale) * w_scale is two fixed binary32
roundings, so acc and y must equal the oracle's bit for bit -- and equal the decode GEMV's for the
same tokens.  Sizes span several 128 x 128 tiles with ragged tails in M and N; small calls split K
across CTAs (the last split of each tile adds the others), large calls do not; the degenerate
cases are the largest accumulator (|acc| = 128 K at K = 2^24 / 128), -128 activations, empty
rows and columns set in neither plane; the BitNet-2B4T prefill shapes run at 512 tokens with
sampled rows compared.
"""
import numpy as np
import pytest
import torch

import bit_matvec_lb_gb300 as lb
import oracle
import synth
from gpu_util import dev, guarded, host

pytestmark = pytest.mark.gpu


def _acts(M, K, seed):
    """Per-token absmax int8 activations of N(0, 1) values, as the planar path quantizes them."""
    return oracle.quantize_i8_absmax(synth.activations(M, K, seed=seed))


def gemm_trit(planes, w_scale, q, xs, workspace=None, planes_dev=None):
    N = planes.shape[0]
    M, K = q.shape
    if workspace is None:
        workspace = guarded(lb.lb_gemm_trit_workspace_bytes(M, K), torch.uint8)
    y = guarded((M, N), torch.float32, float("nan"))
    acc = guarded((M, N), torch.int32, -7)
    lb.lb_gemm_trit_planes(dev(planes) if planes_dev is None else planes_dev, w_scale, dev(q),
                           dev(np.asarray(xs, np.float32)), y, acc, M, N, K, workspace)
    torch.cuda.synchronize()
    return host(acc), host(y)


def _check_exact(planes, w_scale, q, xs, **kw):
    acc, y = gemm_trit(planes, w_scale, q, xs, **kw)
    acc_ref, y_ref = oracle.trit_planes_product(planes, w_scale, q, xs)
    assert np.array_equal(acc, acc_ref), "integer accumulators differ from the oracle"
    assert np.array_equal(y.view(np.uint32), y_ref.view(np.uint32)), "outputs differ"
    return acc, y


@pytest.mark.parametrize("M,N,K", [(1, 1, 64), (5, 7, 192), (128, 128, 1024), (130, 257, 1152),
                                   (300, 200, 2048), (257, 129, 4224)])
def test_gemm_trit_ragged(M, N, K):
    """Several tiles with ragged tails; from K = 512 up these small calls split K."""
    planes, _ = synth.trit_planes(N, K, seed=M + N + K)
    q, xs = _acts(M, K, seed=3 * M + K)
    _check_exact(planes, synth.w_scale(M + 1), q, xs)


def test_gemm_trit_unsplit_many_tiles():
    """Enough tiles (4 x 39 = 156) that K is not split: the direct epilogue."""
    M, N, K = 512, 4992, 512
    planes, _ = synth.trit_planes(N, K, seed=11)
    q, xs = _acts(M, K, seed=12)
    _check_exact(planes, 0.0173, q, xs)


def test_gemm_trit_largest_accumulator():
    """K = 2^24 / 128 (the limit) with -128 everywhere: an all-(+1) row gives acc = -2^24, an
    all-(-1) row +2^24, the largest magnitudes; a random row and an all-zero row beside them.
    K is split four ways here, so the split partials are added at full magnitude too."""
    M, K = 3, (1 << 24) // 128
    trits = np.zeros((4, K), np.int8)
    trits[0] = 1
    trits[1] = -1
    trits[2] = synth.rng(21).integers(-1, 2, size=K)
    planes = synth.trits_to_planes(trits)
    q = np.full((M, K), -128, np.int8)
    q[2, ::3] = 127
    xs = np.array([1.0, 0.5, 3.0e-3], np.float32)
    acc, _ = _check_exact(planes, 1.0, q, xs)
    assert acc[0, 0] == -(1 << 24) and acc[0, 1] == (1 << 24) and np.all(acc[:, 3] == 0)


def test_gemm_trit_extreme_codes():
    """Activations drawn from {-128, -127, 127} against random trits (unit scales: y = acc)."""
    M, N, K = 140, 150, 2560
    planes, _ = synth.trit_planes(N, K, seed=31, probs=(0.45, 0.1, 0.45))
    q = synth.int8_codes(M, K, seed=32, extremes=True)
    _check_exact(planes, 1.0, q, np.ones(M, np.float32))


def test_gemm_trit_matches_gemv():
    """The GEMM over 8 tokens equals the 8-token decode GEMV bit for bit (same definition,
    exact integers, same two roundings)."""
    N, K, B = 300, 2560, 8
    planes, _ = synth.trit_planes(N, K, seed=41)
    q, xs = _acts(B, K, seed=42)
    acc, y = gemm_trit(planes, 0.02, q, xs)
    yv = guarded((B, N), torch.float32, float("nan"))
    av = guarded((B, N), torch.int32)
    lb.lb_gemv_trit_planes(dev(planes), 0.02, dev(q), dev(xs), yv, av, N, K, B)
    torch.cuda.synchronize()
    assert np.array_equal(acc, host(av))
    assert np.array_equal(y.view(np.uint32), host(yv).view(np.uint32))


def test_gemm_trit_workspace_reused():
    """Two calls in a row share one workspace (the second with fewer tokens and another split):
    both exact."""
    N, K = 200, 2048
    planes, _ = synth.trit_planes(N, K, seed=51)
    pd = dev(planes)
    ws = guarded(lb.lb_gemm_trit_workspace_bytes(300, K), torch.uint8)
    for M, seed in ((300, 52), (77, 53), (300, 54)):
        q, xs = _acts(M, K, seed=seed)
        _check_exact(planes, 0.011, q, xs, workspace=ws, planes_dev=pd)


def test_gemm_trit_grouped():
    """Grouped call: three ragged matrices (130, 1, 257 rows) with their own w_scale sharing
    one activation of 130 tokens; every output bit-exact against the oracle and equal to the
    single-matrix call."""
    M, K, Ns = 130, 1216, (130, 1, 257)
    q, xs = _acts(M, K, seed=60)
    ws = guarded(lb.lb_gemm_trit_workspace_bytes(M, K), torch.uint8)
    mats, outs = [], []
    for i, n in enumerate(Ns):
        planes, _ = synth.trit_planes(n, K, seed=61 + i)
        w = synth.w_scale(70 + i)
        y = guarded((M, n), torch.float32, float("nan"))
        acc = guarded((M, n), torch.int32) if i != 1 else None
        mats.append((dev(planes), w, y, acc, n))
        outs.append((planes, w, y, acc))
    lb.lb_gemm_trit_planes_grouped(mats, dev(q), dev(xs), M, K, ws)
    torch.cuda.synchronize()
    for planes, w, y, acc in outs:
        acc_ref, y_ref = oracle.trit_planes_product(planes, w, q, xs)
        assert np.array_equal(host(y).view(np.uint32), y_ref.view(np.uint32))
        if acc is not None:
            assert np.array_equal(host(acc), acc_ref)
        acc1, y1 = gemm_trit(planes, w, q, xs)
        assert np.array_equal(host(y).view(np.uint32), y1.view(np.uint32))


def test_gemm_trit_y_only_outputs():
    """Grouped calls with no integer output, the form in which each token row of y leaves its CTA
    as one bulk copy (N a multiple of 4), beside matrices whose rows take per-thread stores (N
    not a multiple of 4; an integer output).  M = 300 over 44 weight tiles: two-token-tile CTAs
    parking 128 columns per pass and a last pair holding one token tile; M = 100 with K too
    short to split: one-token-tile CTAs parking 256 columns.  Column tails of 4 and 4 + 256;
    every output bit-exact against the oracle, every guard band untouched."""
    K = 128
    for M, Ns in ((300, (9732, 4, 260, 130, 132)), (100, (260, 4, 130, 516, 132))):
        q, xs = _acts(M, K, seed=M + 5)
        ws = guarded(lb.lb_gemm_trit_workspace_bytes(M, K), torch.uint8)
        mats, outs = [], []
        for i, n in enumerate(Ns):
            planes, _ = synth.trit_planes(n, K, seed=300 + 10 * M + i)
            w = synth.w_scale(310 + i)
            y = guarded((M, n), torch.float32, float("nan"))
            acc = guarded((M, n), torch.int32, -7) if i == len(Ns) - 1 else None
            mats.append((dev(planes), w, y, acc, n))
            outs.append((planes, w, y, acc))
        lb.lb_gemm_trit_planes_grouped(mats, dev(q), dev(xs), M, K, ws)
        torch.cuda.synchronize()
        for planes, w, y, acc in outs:
            acc_ref, y_ref = oracle.trit_planes_product(planes, w, q, xs)
            assert np.array_equal(host(y).view(np.uint32), y_ref.view(np.uint32)), planes.shape
            if acc is not None:
                assert np.array_equal(host(acc), acc_ref)


@pytest.mark.parametrize("name,N,K", [("q", 2560, 2560), ("gate", 6912, 2560),
                                      ("down", 2560, 6912), ("k", 640, 2560)])
def test_gemm_trit_prefill_shapes_sampled(name, N, K):
    """512-token prefill through the full-size BitNet-2B4T projections: the whole GEMM runs on
    the GPU; every token is compared with the oracle on rows sampled from every 128-row tile."""
    M = synth.PREFILL_M
    planes, _ = synth.trit_planes(N, K, seed=900 + N + K)
    q, xs = _acts(M, K, seed=901)
    acc, y = gemm_trit(planes, 0.02, q, xs)
    rows = np.unique(np.concatenate([np.arange(0, N, 127), [127, 128, N - 1]]))
    acc_ref, y_ref = oracle.trit_planes_product(planes[rows], 0.02, q, xs)
    assert np.array_equal(acc[:, rows], acc_ref)
    assert np.array_equal(y[:, rows].view(np.uint32), y_ref.view(np.uint32))


def test_gemm_trit_device_status_clean():
    assert lb.lb_device_status() == 0


@pytest.mark.parametrize("M,K,Ns", [(1, 64, (3,)), (130, 1216, (130, 1, 257)),
                                    (300, 2560, (640, 2560)), (512, 6912, (2560,))])
def test_quantize_tiles_then_gemm(M, K, Ns):
    """lb_quantize_i8_absmax_tiles writes q and x_scale bit-identical to lb_quantize_i8_absmax
    (and to the oracle's quantizer) plus the GEMM's operand tiles, from which
    lb_gemm_trit_planes_grouped_tiles gives acc and y bit-identical to the oracle; rows of the
    last 128-token tile past M are written too (as zeros) and a second group reads the same
    tiles."""
    x = synth.activations(M, K, seed=40 + M)
    q_ref, xs_ref = oracle.quantize_i8_absmax(x)
    xd = dev(x)
    q = guarded((M, K), torch.int8)
    xs = guarded((M,), torch.float32, float("nan"))
    ws = guarded(lb.lb_gemm_trit_workspace_bytes(M, K), torch.uint8, 0xFF)
    lb.lb_quantize_i8_absmax_tiles(xd, q, xs, M, K, ws)
    q2 = guarded((M, K), torch.int8)
    xs2 = guarded((M,), torch.float32, float("nan"))
    lb.lb_quantize_i8_absmax(xd, q2, xs2, M, K)
    torch.cuda.synchronize()
    assert np.array_equal(host(q), q_ref) and np.array_equal(host(q2), q_ref)
    assert np.array_equal(host(xs).view(np.uint32), np.asarray(xs_ref, np.float32).view(np.uint32))
    assert np.array_equal(host(xs).view(np.uint32), host(xs2).view(np.uint32))
    for rep in range(2):
        mats, outs = [], []
        for i, n in enumerate(Ns):
            planes, _ = synth.trit_planes(n, K, seed=80 + 7 * i + rep)
            w = synth.w_scale(90 + i + rep)
            y = guarded((M, n), torch.float32, float("nan"))
            acc = guarded((M, n), torch.int32)
            mats.append((dev(planes), w, y, acc, n))
            outs.append((planes, w, y, acc))
        lb.lb_gemm_trit_planes_grouped_tiles(mats, xs, M, K, ws)
        torch.cuda.synchronize()
        for planes, w, y, acc in outs:
            acc_ref, y_ref = oracle.trit_planes_product(planes, w, q_ref, xs_ref)
            assert np.array_equal(host(acc), acc_ref)
            assert np.array_equal(host(y).view(np.uint32), y_ref.view(np.uint32))
    assert lb.lb_device_status() == 0


def test_quantize_tiles_degenerate_rows():
    """The operand-writing quantizer on degenerate tokens: an all-zero row (x_scale 0, every code
    0), a row whose extremes quantize to -127 and +127, a row of one nonzero value, and M = 1
    past which the whole 128-row tile is zero; q, x_scale, acc and y bit-identical to the
    oracle."""
    for M, K in ((130, 128), (1, 256)):
        x = synth.activations(M, K, seed=9300 + M)
        x[0] = 0.0
        if M > 2:
            x[1] *= 1e30
            x[2] = 0.0
            x[2, K // 3] = -3.5
        q_ref, xs_ref = oracle.quantize_i8_absmax(x)
        q = guarded((M, K), torch.int8)
        xs = guarded((M,), torch.float32, float("nan"))
        ws = guarded(lb.lb_gemm_trit_workspace_bytes(M, K), torch.uint8, 0xFF)
        lb.lb_quantize_i8_absmax_tiles(dev(x), q, xs, M, K, ws)
        planes, _ = synth.trit_planes(200, K, seed=9310 + M)
        y = guarded((M, 200), torch.float32, float("nan"))
        acc = guarded((M, 200), torch.int32)
        lb.lb_gemm_trit_planes_grouped_tiles([(dev(planes), 0.03, y, acc, 200)], xs, M, K, ws)
        torch.cuda.synchronize()
        assert np.array_equal(host(q), q_ref)
        assert np.array_equal(host(xs).view(np.uint32),
                              np.asarray(xs_ref, np.float32).view(np.uint32))
        acc_ref, y_ref = oracle.trit_planes_product(planes, 0.03, q_ref, xs_ref)
        assert np.array_equal(host(acc), acc_ref)
        assert np.array_equal(host(y).view(np.uint32), y_ref.view(np.uint32))
    assert lb.lb_device_status() == 0
