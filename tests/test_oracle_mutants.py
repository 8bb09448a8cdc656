"""The oracle's pins must catch plausible mistakes.

Each case plants one slip in a copy of oracle/lb_oracle.c (on the CPU, in a temporary
directory), builds it, and runs the pin suite against that copy in a subprocess: the suite must
fail.  The cases are the errors a careful reader could make with the pages' definitions -- a bit
or code order read the wrong way round, a flipped polarity, a dropped offset or term, a wrong
index, a rounding rule or a scale taken from the wrong quantity.
"""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "lb_oracle.c")

MUTANTS = [
    ("q1_msb_first", "int bit = (qs[i / 8] >> (i % 8)) & 1;",
     "int bit = (qs[i / 8] >> (7 - i % 8)) & 1;"),
    ("q1_polarity", "return bit ? +1 : -1;", "return bit ? -1 : +1;"),
    ("q2_high_bits_first", "int c = (qs[i / 4] >> (2 * (i % 4))) & 3;",
     "int c = (qs[i / 4] >> (6 - 2 * (i % 4))) & 3;"),
    ("q2_no_offset", "return c - 1;", "return c;"),
    ("q_wrong_act_index", "(int64_t)q[b * K + blk * qk + widx]", "(int64_t)q[b * K + widx]"),
    ("q_wrong_dx_index", "oracle_f16_to_f32(dx[b * nq8 + jj])", "oracle_f16_to_f32(dx[b * nq8 + blk])"),
    ("q_dropped_term", "for (int j = 0; j < per; j++) {", "for (int j = 0; j < per - 1; j++) {"),
    ("q8_round_half_away", "return (float)((fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0);",
     "return (float)(d >= 0 ? fl + 1.0 : fl);"),
    ("q8_scale_from_amax", "d[b * nb + j] = oracle_f32_to_f16(dd);",
     "d[b * nb + j] = oracle_f32_to_f16(amax);"),
    ("f16_subnormal_exp", "mag = ldexp((double)frac, -24);", "mag = ldexp((double)frac, -25);"),
    ("f16_tie_to_odd", "if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0))",
     "if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) == 0.0))"),
    ("planar_swapped_planes", "uint64_t pos = planes[(r * nbeat + g) * 2 + 0];",
     "uint64_t pos = planes[(r * nbeat + g) * 2 + 1];"),
    ("planar_folded_scales", "float t = (float)a * x_scale[b];\n            y[b * N + r] = t * w_scale;",
     "y[b * N + r] = (float)a * (x_scale[b] * w_scale);"),
    ("planar_negated_in_int8", "a -= x;         /* w = -1: subtract */",
     "a += (int8_t)(-x);"),
    ("repack_scale_bytes_swapped",
     "return (uint16_t)(block18[0] | ((uint16_t)block18[1] << 8));",
     "return (uint16_t)(block18[1] | ((uint16_t)block18[0] << 8));"),
    ("bf16_wrong_shift", "return bits_f32((uint32_t)b << 16);", "return bits_f32((uint32_t)b << 15);"),
    ("bf16_round_truncates", "if (drop > 0x8000u || (drop == 0x8000u && (keep & 1u)))",
     "if (0)"),
    ("bf16_ties_away", "(drop == 0x8000u && (keep & 1u))", "(drop == 0x8000u)"),
    ("planar_dequant_swapped_planes", "uint64_t pos = beat[0], neg = beat[1];",
     "uint64_t pos = beat[1], neg = beat[0];"),
    ("base3_digit_without_offset", "value += (t + 1) * place;", "value += t * place;"),
    ("base3_high_digit_first", "int j = (int)((col % 80) / 5), i = (int)(col % 5);",
     "int j = (int)((col % 80) / 5), i = 4 - (int)(col % 5);"),
    ("base3_group_of_64", "int64_t g = col / 80;", "int64_t g = col / 64;"),
    ("i8_amax_signed", "float a = fabsf(xb[k]);", "float a = xb[k];"),
    ("i8_amax_first_token", "float a = fabsf(xb[k]);", "float a = fabsf(x[k]);"),
    ("i8_round_half_away", "float v = round_half_even(xb[k] * s);", "float v = roundf(xb[k] * s);"),
    ("i8_multiplier_from_scale", "float s = (amax != 0.0f) ? 127.0f / amax : 0.0f;",
     "float s = (amax != 0.0f) ? 1.0f / (amax / 127.0f) : 0.0f;"),
    ("bf16_transposed_weight", "oracle_bf16_to_f32(w[n * K + k])", "oracle_bf16_to_f32(w[k * N + n])"),
    ("bf16_mag_signed", "m += fabs(p);", "m += p;"),
    ("repack_padding_one", "scales[n * S + blk] = 0;", "scales[n * S + blk] = 0x3c00;"),
    ("dequant_first_block_scale", "float d = oracle_f16_to_f32(block_scale_bits(block18));",
     "float d = oracle_f16_to_f32(block_scale_bits(blocks + n * nblk * 18));"),
    ("planar_first_token_only", "int64_t x = q[b * K + g * 64 + c];", "int64_t x = q[g * 64 + c];"),
    ("planar_beats_column_major",
     "uint64_t pos = planes[(r * nbeat + g) * 2 + 0];\n                uint64_t neg = planes[(r * nbeat + g) * 2 + 1];",
     "uint64_t pos = planes[(g * N + r) * 2 + 0];\n                uint64_t neg = planes[(g * N + r) * 2 + 1];"),
    ("q_mag_signed", "m += fabs(term);", "m += term;"),
    ("q_mag_without_isum", "m += fabs(term);", "m += fabs((double)dw * (double)dxf) * 32.0 * 128.0;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    msrc = tmp_path / "mutant.c"
    msrc.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", str(so), str(msrc), "-lm"], check=True)
    env = dict(os.environ, LB_ORACLE_SO=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"pins did not catch mutant {name}:\n{r.stdout[-2000:]}"
