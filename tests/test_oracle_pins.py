"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test checks the oracle against one of: a value printed by hand from the pages' format
definitions (tests/golden/), a closed form, an invariant, an exhaustive or brute-force
computation with independent library primitives (numpy bit unpacking, int64 matmul, numpy's own
IEEE binary16 conversion, exact rational arithmetic), chosen so that a plausible slip -- a
dropped term, a flipped sign or polarity, a wrong bit index, a transposed operand, a missing
rounding step -- fails at least one of them.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from golden_io import read


def _hexbytes(s):
    return np.array([int(t, 16) for t in s.split()], dtype=np.uint8)


def _f16(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


# ----------------------------------------------------------------------------------------------
# IEEE binary16 / bfloat16 conversions (pinned against numpy's independent implementation)
# ----------------------------------------------------------------------------------------------
def test_f16_decode_exhaustive():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f16_bits_to_f32_array(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _f32_samples():
    g = np.random.Generator(np.random.PCG64(1234))
    rnd = g.integers(0, 2**32, size=200_000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    # every binary16 value and the float32 neighbours of every midpoint between two of them
    h = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = ((h[:-1] + h[1:]) / 2).astype(np.float32)
    near = np.concatenate([mids, np.nextafter(mids, np.float32(np.inf)),
                           np.nextafter(mids, np.float32(0))])
    edge = np.array([65504, 65519.99, 65520, 65536, 1e9, 2.0**-24, 2.0**-25, 2.0**-26,
                     3 * 2.0**-26, 2.0**-14, 6e-8, 5.96e-8], dtype=np.float32)
    allv = np.concatenate([rnd, near, edge])
    return np.concatenate([allv, -allv])


def test_f16_encode_against_numpy():
    xs = _f32_samples()
    xs = xs[np.isfinite(xs)]
    with np.errstate(over="ignore"):
        ref = xs.astype(np.float16).view(np.uint16)
    lib = oracle._load()
    ours = np.fromiter((lib.oracle_f32_to_f16(float(v)) for v in xs), dtype=np.uint16,
                       count=xs.size)
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first x={xs[bad[0]]!r}"


def test_f16_encode_nan_inf():
    assert oracle.f32_to_f16(float("inf")) == 0x7C00
    assert oracle.f32_to_f16(float("-inf")) == 0xFC00
    assert (oracle.f32_to_f16(float("nan")) & 0x7C00) == 0x7C00
    assert (oracle.f32_to_f16(float("nan")) & 0x3FF) != 0


def test_bf16_widening():
    g = np.random.Generator(np.random.PCG64(5))
    b = g.integers(0, 65536, size=4096, dtype=np.uint32).astype(np.uint16)
    ref = (b.astype(np.uint32) << 16).view(np.float32)
    ours = np.array([oracle.bf16_to_f32(int(v)) for v in b], dtype=np.float32)
    fin = np.isfinite(ref)
    assert np.array_equal(ours[fin].view(np.uint32), ref[fin].view(np.uint32))


# ----------------------------------------------------------------------------------------------
# q8_0 quantizer
# ----------------------------------------------------------------------------------------------
def test_q8_0_golden_ties():
    gd = read("q8_0_ties.txt")
    x = np.array([float(t) for t in gd["x"].split()], dtype=np.float32)
    q, d = oracle.quantize_q8_0(x[None, :])
    assert q[0].tolist() == [int(t) for t in gd["q"].split()]
    assert int(d[0, 0]) == int(gd["d"], 16)


def test_q8_0_zero_block():
    q, d = oracle.quantize_q8_0(np.zeros((2, 64), np.float32))
    assert not q.any() and not d.any()


def test_q8_0_properties():
    x = synth.activations(4, 4096, seed=11)
    q, d = oracle.quantize_q8_0(x)
    xb = x.reshape(4, -1, 32).astype(np.float64)
    qb = q.reshape(4, -1, 32).astype(np.int64)
    amax = np.abs(xb).max(-1)
    # scale: binary16 of amax/127 (amax/127 rounded to binary32 first), numpy's own conversion
    ref_d = (amax.astype(np.float32) / np.float32(127)).astype(np.float16).view(np.uint16)
    assert np.array_equal(d, ref_d)
    assert np.abs(qb).max() <= 127
    # the largest element of every block maps to +-127 with its own sign
    idx = np.abs(xb).argmax(-1)
    top = np.take_along_axis(qb, idx[..., None], -1)[..., 0]
    topx = np.take_along_axis(xb, idx[..., None], -1)[..., 0]
    assert np.array_equal(top, np.where(topx > 0, 127, -127))
    # reconstruction: |x - q*amax/127| <= amax/254 (half a step), up to binary32 rounding
    err = np.abs(xb - qb * (amax[..., None] / 127.0))
    assert np.all(err <= amax[..., None] / 254.0 * (1 + 1e-5))
    # sign symmetry
    qn, dn = oracle.quantize_q8_0(-x)
    assert np.array_equal(qn, -q) and np.array_equal(dn, d)


def test_q8_0_scaled_grid():
    # amax = 254 makes the multiplier 127/254 = 0.5 exactly, so q = rne(k/2) for integer k:
    # even k give k/2; odd k are exact ties and go to the even one of (k-1)/2, (k+1)/2.
    k = np.arange(-30, 1, dtype=np.int64)                      # 31 integers, odd and even
    x = np.concatenate([k, [254]]).astype(np.float32)
    q, d = oracle.quantize_q8_0(x[None, :])
    expect = [kk // 2 if kk % 2 == 0 else ((kk - 1) // 2 if ((kk - 1) // 2) % 2 == 0
                                           else (kk + 1) // 2) for kk in k.tolist()]
    assert q[0, :-1].tolist() == expect
    assert q[0, -1] == 127
    assert int(d[0, 0]) == np.float16(2.0).view(np.uint16)


def test_i8_absmax_quantizer():
    x = np.array([[-2.0, 1.0, 0.5, 0.0, 2.0, -1.0, 0.25, 0.75],
                  [-127.0, 2.5, 0.5, -3.5, 1.5, 126.5, -0.5, 3.0],
                  [1.375, -0.6875, 0.6875, 0.0, 0.0, 0.0, 0.0, -1.375]], dtype=np.float32)
    q, s = oracle.quantize_i8_absmax(x)
    # token 0: multiplier 127/2 = 63.5 exactly: 1 -> 63.5 -> 64 (tie to even), 0.5 -> 31.75 ->
    # 32, 0.25 -> 15.875 -> 16, 0.75 -> 47.625 -> 48, -1 -> -63.5 -> -64
    assert q[0].tolist() == [-127, 64, 32, 0, 127, -64, 16, 48]
    assert s[0] == np.float32(2.0) / np.float32(127.0)
    # token 1 has its own absmax (127, taken by a negative value: the multiplier is exactly 1),
    # and its ties go to the even neighbour: 2.5 -> 2, 0.5 -> 0, -3.5 -> -4, 1.5 -> 2,
    # 126.5 -> 126, -0.5 -> 0
    assert q[1].tolist() == [-127, 2, 0, -4, 2, 126, 0, 3]
    assert s[1] == np.float32(1.0)
    # token 2: the multiplier is 127 / 1.375 = 92.3636... rounded once, to 92.363640 in binary32
    # (1 / (1.375 / 127) would give 92.363632); 0.6875 times it is 63.500004, just above the
    # tie, so +-0.6875 -> +-64 (the other multiplier gives 63.499996 -> +-63)
    assert q[2].tolist() == [127, -64, 64, 0, 0, 0, 0, -127]
    assert s[2] == np.float32(1.375) / np.float32(127.0)
    q0, s0 = oracle.quantize_i8_absmax(np.zeros((1, 16), np.float32))
    assert not q0.any() and s0[0] == 0.0


# ----------------------------------------------------------------------------------------------
# Q1_0
# ----------------------------------------------------------------------------------------------
def test_q1_0_golden_block():
    gd = read("q1_0_block.txt")
    blk = _hexbytes(gd["block"]).reshape(1, 1, 18)
    q = np.ones((1, 128), np.int8)
    dx = np.full((1, 4), int(gd["dx"], 16), np.uint16)
    r = oracle.q1_0_product(blk, q, dx)
    assert r.isum[0, 0].tolist() == [int(t) for t in gd["isum"].split()]
    assert r.y_exact[0, 0] == float(gd["y"]) and r.y_chain[0, 0] == float(gd["y"])


def _q1_dense(blocks, K):
    """Independent decode: numpy little-endian bit unpacking -> +-1 int matrix [N][K]."""
    N = blocks.shape[0]
    bits = np.unpackbits(blocks[:, :, 2:].reshape(N, -1), axis=1, bitorder="little")
    return (bits.astype(np.int64) * 2 - 1).reshape(N, K)


def _scales(blocks):
    return blocks[:, :, 0].astype(np.uint16) | (blocks[:, :, 1].astype(np.uint16) << 8)


@pytest.mark.parametrize("N,K,B", [(3, 128, 1), (5, 384, 3), (2, 1024, 2)])
def test_q1_0_brute_force(N, K, B):
    blocks = synth.q1_0_blocks(N, K, seed=N * 100 + K)
    q = synth.int8_codes(B, K, seed=7)
    dx = synth.q8_scales(B, K, seed=8)
    r = oracle.q1_0_product(blocks, q, dx)
    W = _q1_dense(blocks, K)
    qs = q.astype(np.int64).reshape(B, K // 32, 32)
    Ws = W.reshape(N, K // 32, 32)
    isum = np.einsum("njk,bjk->bnj", Ws, qs)
    assert np.array_equal(r.isum, isum)
    # exact value by rational arithmetic
    dw = _f16(_scales(blocks))            # [N][K/128]
    dxf = _f16(dx)                        # [B][K/32]
    for b in range(B):
        for n in range(N):
            e = sum(Fraction(dw[n, j // 4]) * Fraction(dxf[b, j]) * int(isum[b, n, j])
                    for j in range(K // 32))
            assert Fraction(r.y_exact[b, n]) == e or abs(float(e) - r.y_exact[b, n]) <= 1e-15 * max(1.0, abs(float(e)))
    # the tolerance magnitude: sum over q8_0 blocks of |d_w * d_x * isum|, from the dense decode
    mag = np.abs(np.repeat(dw, 4, axis=1)[None, :, :] * dxf[:, None, :] * isum).sum(-1)
    assert np.allclose(r.mag, mag, rtol=1e-13, atol=0)


def test_q1_0_all_ones_identity():
    N, K, B = 4, 512, 2
    blocks = synth.q1_0_blocks(N, K, seed=3)
    q = synth.int8_codes(B, K, seed=4)
    dx = synth.q8_scales(B, K, seed=5)
    ones = blocks.copy()
    ones[:, :, 2:] = 0xFF
    zeros = blocks.copy()
    zeros[:, :, 2:] = 0x00
    r1 = oracle.q1_0_product(ones, q, dx)
    r0 = oracle.q1_0_product(zeros, q, dx)
    sq = q.astype(np.int64).reshape(B, K // 32, 32).sum(-1)          # sum of q per q8 block
    dw = _f16(_scales(blocks))
    dxf = _f16(dx)
    expect = np.einsum("nj,bj->bn", np.repeat(dw, 4, axis=1), dxf * sq)
    assert np.allclose(r1.y_exact, expect, rtol=1e-13, atol=0)
    assert np.allclose(r0.y_exact, -expect, rtol=1e-13, atol=0)
    assert np.array_equal(r1.isum, np.broadcast_to(sq[:, None, :], r1.isum.shape))


# ----------------------------------------------------------------------------------------------
# Q2_0_g64
# ----------------------------------------------------------------------------------------------
def test_q2_0_golden_block():
    gd = read("q2_0_block.txt")
    blk = _hexbytes(gd["block"]).reshape(1, 1, 18)
    q = np.zeros((1, 64), np.int8)
    q[0, :8] = [int(t) for t in gd["q"].split()]
    dx = np.array([[int(t, 16) for t in gd["dx"].split()]], np.uint16)
    r = oracle.q2_0_g64_product(blk, q, dx)
    assert r.isum[0, 0].tolist() == [int(t) for t in gd["isum"].split()]
    assert r.y_exact[0, 0] == float(gd["y"])


def _q2_dense(blocks, K):
    """Independent decode: shift/mask of every byte with numpy -> int weights [N][K]."""
    N = blocks.shape[0]
    by = blocks[:, :, 2:].astype(np.int64)                             # [N][nb][16]
    codes = np.stack([(by >> (2 * r)) & 3 for r in range(4)], axis=-1)  # [N][nb][16][4]
    return (codes - 1).reshape(N, K)


@pytest.mark.parametrize("N,K,B,probs", [(3, 64, 1, synth.TERNARY_PROBS),
                                         (4, 448, 3, (0.25, 0.25, 0.25, 0.25)),
                                         (2, 1024, 2, (0.2, 0.2, 0.2, 0.4))])
def test_q2_0_brute_force(N, K, B, probs):
    blocks = synth.q2_0_blocks(N, K, seed=N + K, probs=probs)
    q = synth.int8_codes(B, K, seed=9)
    dx = synth.q8_scales(B, K, seed=10)
    r = oracle.q2_0_g64_product(blocks, q, dx)
    W = _q2_dense(blocks, K)
    isum = np.einsum("njk,bjk->bnj", W.reshape(N, K // 32, 32),
                     q.astype(np.int64).reshape(B, K // 32, 32))
    assert np.array_equal(r.isum, isum)
    dw = np.repeat(_f16(_scales(blocks)), 2, axis=1)                   # per q8 block
    expect = np.einsum("nj,bnj->bn", dw, _f16(dx)[:, None, :] * isum)
    assert np.allclose(r.y_exact, expect, rtol=1e-12, atol=1e-300)
    # the tolerance magnitude: sum over q8_0 blocks of |d_w * d_x * isum|, from the dense decode
    mag = np.abs(dw[None, :, :] * _f16(dx)[:, None, :] * isum).sum(-1)
    assert np.allclose(r.mag, mag, rtol=1e-13, atol=0)


@pytest.mark.parametrize("code,factor", [(1, 0), (2, 1), (0, -1), (3, 2)])
def test_q2_0_constant_codes(code, factor):
    N, K, B = 3, 256, 2
    codes = np.full((N, K // 64, 64), code, np.uint8)
    blocks = synth.q2_0_blocks(N, K, seed=21, codes=codes)
    q = synth.int8_codes(B, K, seed=22)
    dx = synth.q8_scales(B, K, seed=23)
    r = oracle.q2_0_g64_product(blocks, q, dx)
    sq = q.astype(np.int64).reshape(B, K // 32, 32).sum(-1)
    dw = np.repeat(_f16(_scales(blocks)), 2, axis=1)
    expect = factor * np.einsum("nj,bj->bn", dw, _f16(dx) * sq)
    if factor == 0:
        assert np.all(r.y_exact == 0.0) and np.all(r.y_chain == 0.0)
    else:
        assert np.allclose(r.y_exact, expect, rtol=1e-13, atol=0)


# ----------------------------------------------------------------------------------------------
# planar ternary
# ----------------------------------------------------------------------------------------------
def test_trit_planes_golden_beat():
    gd = read("trit_planes_beat.txt")
    planes = np.array([[[int(gd["pos"], 16), int(gd["neg"], 16)]]], np.uint64)
    q = np.full((1, 64), int(gd["qmid"]), np.int8)
    q[0, 0] = int(gd["q0"])
    q[0, 63] = int(gd["q63"])
    acc, y = oracle.trit_planes_product(planes, float(gd["w_scale"]), q,
                                        np.array([float(gd["x_scale"])], np.float32))
    assert acc[0, 0] == int(gd["acc"]) and y[0, 0] == np.float32(gd["y"])


@pytest.mark.parametrize("N,K,B", [(4, 64, 1), (7, 320, 3), (3, 2560, 2)])
def test_trit_planes_brute_force(N, K, B):
    planes, trits = synth.trit_planes(N, K, seed=K + N)
    q = synth.int8_codes(B, K, seed=31)
    xs = np.array([0.013, 0.021, 0.5][:B], np.float32)
    acc, y = oracle.trit_planes_product(planes, 0.037, q, xs)
    ref = q.astype(np.int64) @ trits.astype(np.int64).T                # [B][N]
    assert np.array_equal(acc, ref)
    # two binary32 roundings in the stated order
    assert np.array_equal(y, (ref.astype(np.float32) * xs[:, None]) * np.float32(0.037))


def test_trit_planes_match_q2_codes():
    """The planar layout and the offset-code layout encode the same ternary matrix: with every
    scale 1 the planar accumulator equals the sum of the code layout's block sums."""
    N, K, B = 5, 512, 2
    g = np.random.Generator(np.random.PCG64(41))
    codes = g.integers(0, 3, size=(N, K // 64, 64)).astype(np.uint8)   # no +2 in planar
    one = np.float16(1.0).view(np.uint16)
    blocks = synth.q2_0_blocks(N, K, seed=0, codes=codes,
                               scales=np.full((N, K // 64), one, np.uint16))
    planes = synth.trits_to_planes(codes.reshape(N, K).astype(np.int8) - 1)
    q = synth.int8_codes(B, K, seed=42)
    r = oracle.q2_0_g64_product(blocks, q, np.full((B, K // 32), one, np.uint16))
    acc, _ = oracle.trit_planes_product(planes, 1.0, q, np.ones(B, np.float32))
    assert np.array_equal(acc, r.isum.sum(-1))


def test_trit_planes_minus128_extremes():
    K = 512
    q = np.full((1, K), -128, np.int8)
    allset = np.uint64(0xFFFFFFFFFFFFFFFF)
    pos = np.zeros((1, K // 64, 2), np.uint64)
    pos[..., 0] = allset
    neg = np.zeros((1, K // 64, 2), np.uint64)
    neg[..., 1] = allset
    a_pos, _ = oracle.trit_planes_product(pos, 1.0, q, np.ones(1, np.float32))
    a_neg, _ = oracle.trit_planes_product(neg, 1.0, q, np.ones(1, np.float32))
    assert a_pos[0, 0] == -128 * K and a_neg[0, 0] == 128 * K


def test_trit_planes_overlap_rejected():
    planes = np.zeros((1, 1, 2), np.uint64)
    planes[0, 0] = [1, 1]
    with pytest.raises(ValueError):
        oracle.trit_planes_product(planes, 1.0, np.zeros((1, 64), np.int8),
                                   np.ones(1, np.float32))


# ----------------------------------------------------------------------------------------------
# bf16 head
# ----------------------------------------------------------------------------------------------
def test_bf16_product_against_float64_matmul():
    N, K, B = 9, 320, 3
    w = synth.bf16_weights(N, K, seed=51)
    x = synth.activations(B, K, seed=52)
    y, mag = oracle.bf16_product(w, x)
    W = (w.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = x.astype(np.float64) @ W.T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-14)
    assert np.allclose(mag, np.abs(x.astype(np.float64)) @ np.abs(W).T, rtol=1e-12)


# ----------------------------------------------------------------------------------------------
# float results: exactness of the reference value, unit-scale exactness, fp32 chain
# ----------------------------------------------------------------------------------------------
def test_unit_scale_chain_is_exact():
    """With every scale 1.0 each fp32 partial is an integer below 2^24, so the fp32 chain must
    equal the integer sum of the block sums exactly."""
    N, K, B = 6, 1024, 2
    one = np.float16(1.0).view(np.uint16)
    blocks = synth.q1_0_blocks(N, K, seed=61, scales=np.full((N, K // 128), one, np.uint16))
    q = synth.int8_codes(B, K, seed=62)
    r = oracle.q1_0_product(blocks, q, np.full((B, K // 32), one, np.uint16))
    assert np.array_equal(r.y_chain.astype(np.int64), r.isum.sum(-1))
    assert np.array_equal(r.y_exact.astype(np.int64), r.isum.sum(-1))


def test_chain_within_bound_of_exact():
    N, K, B = 64, 4096, 2
    blocks = synth.q2_0_blocks(N, K, seed=71)
    x = synth.activations(B, K, seed=72)
    q, dx = oracle.quantize_q8_0(x)
    r = oracle.q2_0_g64_product(blocks, q, dx)
    assert np.all(np.abs(r.y_chain - r.y_exact) <= r.tolerance())
    # the bound is not vacuous: magnitudes are far above the absolute floor
    assert np.median(r.mag) > 1e-2


# ----------------------------------------------------------------------------------------------
# load-time split and dequantization
# ----------------------------------------------------------------------------------------------
def test_repack_split():
    # two rows x two Q1_0 blocks, every byte distinct: scale bytes 0..1, data bytes 2..17
    blocks = (np.arange(2 * 2 * 18, dtype=np.uint16) % 251).astype(np.uint8).reshape(2, 2, 18)
    bits, scales = oracle.repack(blocks, K=256, qk=128)
    # scale rows are padded to 8 entries (16 bytes) with zeros
    assert scales.tolist() == [[0x0100, 0x1312, 0, 0, 0, 0, 0, 0],
                               [0x2524, 0x3736, 0, 0, 0, 0, 0, 0]]
    assert bits[0, :16].tolist() == list(range(2, 18))
    assert bits[0, 16:].tolist() == list(range(20, 36))
    assert bits[1, :16].tolist() == list(range(38, 54))


def test_dequant_matches_independent_decode():
    N, K = 3, 256
    b1 = synth.q1_0_blocks(N, K, seed=81)
    b2 = synth.q2_0_blocks(N, K, seed=82, probs=(0.25, 0.25, 0.25, 0.25))
    d1 = oracle.dequant(b1, K, 128)
    d2 = oracle.dequant(b2, K, 64)
    assert np.array_equal(d1, (_q1_dense(b1, K) * np.repeat(_f16(_scales(b1)), 128, 1)).astype(np.float32))
    assert np.array_equal(d2, (_q2_dense(b2, K) * np.repeat(_f16(_scales(b2)), 64, 1)).astype(np.float32))


# ----------------------------------------------------------------------------------------------
# dequantization to bf16 and planar dequantization (reading R10)
# ----------------------------------------------------------------------------------------------
def _torch_bf16_bits(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def test_f32_to_bf16_against_torch():
    """Round to nearest, ties to even, pinned against torch's own float32 -> bfloat16 conversion
    (an independent implementation): every dequantized value a weight can take (every finite
    fp16 scale times -1, +1 and +2), constructed ties with even and odd kept halves, and random
    binary32 bit patterns."""
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = h.view(np.float16).astype(np.float32)
    f = f[np.isfinite(f)]
    vals = [f, -f, 2 * f]
    keep = np.arange(0, 1 << 16, 7, dtype=np.uint32)
    keep = keep[(keep & 0x7F80) != 0x7F80]          # finite kept halves
    for drop in (0x8000, 0x7FFF, 0x8001, 0x0000, 0xFFFF):
        vals.append(((keep << 16) | drop).view(np.float32))
    g = synth.rng(99)
    r = g.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32).view(np.float32)
    vals.append(r[np.isfinite(r)])
    x = np.concatenate(vals)
    assert np.array_equal(oracle.f32_to_bf16(x), _torch_bf16_bits(x))
    # infinities stay infinite, NaN stays NaN
    special = np.array([np.inf, -np.inf, np.nan], np.float32)
    out = oracle.f32_to_bf16(special)
    assert out[0] == 0x7F80 and out[1] == 0xFF80 and (out[2] & 0x7F80) == 0x7F80 and out[2] & 0x7F


def test_f32_to_bf16_ties_by_hand():
    # 1 + 2^-8 is half an ulp above 1.0 (bf16 keeps 7 fraction bits): ties go to the even 1.0;
    # 1 + 3 * 2^-8 is half-way between 1 + 2^-7 (odd) and 1 + 2^-6 (even): rounds up
    assert oracle.f32_to_bf16(np.array([1.00390625, 1.01171875, -1.00390625], np.float32)).tolist() \
        == [0x3F80, 0x3F82, 0xBF80]


def test_dequant_bf16_is_rounded_f32():
    N, K = 4, 512
    b = synth.q2_0_blocks(N, K, seed=83, probs=(0.25, 0.25, 0.25, 0.25))
    f = oracle.dequant(b, K, 64)
    assert np.array_equal(oracle.dequant_bf16(b, K, 64), _torch_bf16_bits(f))


def test_trit_planes_dequant_matches_generator_trits():
    """The oracle's decode of the planes against the dense trits the encoder was given."""
    N, K = 5, 320
    planes, trits = synth.trit_planes(N, K, seed=84)
    w = synth.w_scale(85)
    assert np.array_equal(oracle.trit_planes_dequant(planes, w, K),
                          trits.astype(np.float32) * np.float32(w))
    neg = -0.5
    d = oracle.trit_planes_dequant(planes, neg, K)
    assert np.array_equal(np.signbit(d[trits == 0]), np.ones((trits == 0).sum(), bool))
    bad = planes.copy()
    bad[0, 0, 1] |= bad[0, 0, 0] | np.uint64(1)
    bad[0, 0, 0] |= np.uint64(1)
    with pytest.raises(ValueError):
        oracle.trit_planes_dequant(bad, w, K)


# ----------------------------------------------------------------------------------------------
# base-3 packing (reading R15)
# ----------------------------------------------------------------------------------------------
def test_base3_golden_bytes():
    """Bytes worked by hand from the definition ([TR] III.8), placed as bytes 0..5 of the first
    group of a row whose other columns are zero trits."""
    gd = read("base3_bytes.txt")
    K = 128
    trits = np.zeros((1, K), np.int8)
    for j in range(6):
        trits[0, 5 * j: 5 * j + 5] = [int(t) for t in gd[f"trits{j}"].split()]
    packed = oracle.base3_pack(synth.trits_to_planes(trits), K)
    assert packed.shape == (1, 32)
    assert packed[0, :6].tolist() == [int(gd[f"byte{j}"]) for j in range(6)]
    assert np.all(packed[0, 6:] == 121)       # zero trits, including the padding past K


def test_base3_round_trip_and_padding():
    for K in (64, 320, 2560, 6912):
        planes, trits = synth.trit_planes(4, K, seed=K)
        packed = oracle.base3_pack(planes, K)
        assert packed.shape == (4, (K + 79) // 80 * 16)
        assert packed.max() <= 242
        assert np.array_equal(oracle.base3_unpack(packed, K), trits)
        # the columns past K (to the end of the last 80-column group) hold zero trits
        tail = (K + 79) // 80 * 80 - K
        if tail:
            full = oracle.base3_unpack(packed, (K + 79) // 80 * 80)
            assert np.all(full[:, K:] == 0)


def test_base3_product_equals_planar_and_brute_force():
    """The base-3 product of the same trits equals the planar oracle's bit for bit, and the
    accumulators equal a brute-force int64 matmul of the generator's dense trits."""
    N, K, B = 9, 2560 + 64, 3
    planes, trits = synth.trit_planes(N, K, seed=91)
    q = synth.int8_codes(B, K, seed=92, extremes=False)
    q[0, :] = -128
    xs = np.array([0.5, 0.013, 3.0], np.float32)
    acc3, y3 = oracle.base3_product(oracle.base3_pack(planes, K), 0.02, q, xs)
    accp, yp = oracle.trit_planes_product(planes, 0.02, q, xs)
    assert np.array_equal(acc3, accp)
    assert np.array_equal(y3.view(np.uint32), yp.view(np.uint32))
    assert np.array_equal(acc3.astype(np.int64), q.astype(np.int64) @ trits.astype(np.int64).T)


def test_base3_rejects_non_base3_bytes():
    packed = np.full((1, 16), 121, np.uint8)
    packed[0, 3] = 243
    with pytest.raises(ValueError):
        oracle.base3_product(packed, 1.0, np.zeros((1, 64), np.int8), np.ones(1, np.float32))
