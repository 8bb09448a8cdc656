"""The bench's byte model against the byte figures the pages print.

Every GB/s the bench reports divides bytes computed by `bench.q1_bytes`, `q2_bytes`,
`trit_bytes` and `bf16_bytes` (per-call weight bytes of the four formats) by a device time, so
a slip in one of them would move every figure of its rows.  The pages quote the same totals
for their own models, which pins these functions without a GPU:

* "bankml: verified low-bit inference on commodity CPUs -- a technical report", IV.3 (Where the
  time goes, end to end): one token's 253 ternary matrix products of Ternary-Bonsai-8B, the
  Qwen3-8B shapes in Q2_0_g64, come to 2.13 GB of weights;
* "bankml: Ternary and 1-Bit Models on the CPU You Already Have, Verified in Rust", benchmarks
  of the ternary kernel per matrix: the 253rd of those products is the 151669 x 4096 output
  matrix;
* tritium.technology "Architecture", 3 (the bandwidth math): the bf16 head of a 128256-word
  vocabulary over 2560 columns is 656,670,720 bytes (1,313,341,440 when widened to f32);
* tritium.technology "Architecture", 7 (Threading): a BitNet-2B4T decode step issues 210
  ternary matvecs, the largest of them 4.4 MB.
"""
import pytest

import bench
import synth

QWEN3_OUTPUT = (151669, 4096)  # the output matrix of the per-matrix benchmark table


def test_ternary_token_is_2_13_gb():
    body = synth.QWEN3_8B_LAYERS * sum(bench.q2_bytes(n, k) for _, n, k in synth.QWEN3_8B_PROJ)
    total = body + bench.q2_bytes(*QWEN3_OUTPUT)
    assert synth.QWEN3_8B_LAYERS * len(synth.QWEN3_8B_PROJ) + 1 == 253
    assert round(total / 1e9, 2) == 2.13
    # the decode rows time the 252 layer products; the output matrix is not among them
    assert body == 1_953_497_088


def test_one_bit_token_is_half_the_ternary_bytes():
    # Q1_0 packs 128 weights in the 18 bytes that hold 64 in Q2_0_g64
    body = synth.QWEN3_8B_LAYERS * sum(bench.q1_bytes(n, k) for _, n, k in synth.QWEN3_8B_PROJ)
    assert 2 * body == 1_953_497_088


def test_bf16_head_bytes():
    assert bench.bf16_bytes(*synth.BITNET_HEAD) == 656_670_720
    assert synth.BITNET_HEAD == (128256, 2560)


def test_bitnet_matvecs_210_largest_4_4_mb():
    shapes = [(n, k) for _, n, k in synth.BITNET_2B4T_PROJ] * synth.BITNET_2B4T_LAYERS
    assert len(shapes) == 210
    largest = max(bench.trit_bytes(n, k) for n, k in shapes)
    assert round(largest / 1e6, 1) == 4.4


@pytest.mark.parametrize("fn,N,K,per_row_beat", [(bench.q2_bytes, 3, 64, 18),
                                                  (bench.q1_bytes, 3, 128, 18),
                                                  (bench.trit_bytes, 3, 64, 16)])
def test_one_block_per_row(fn, N, K, per_row_beat):
    # the smallest call: one block (beat) per row
    assert fn(N, K) == N * per_row_beat
