"""Each pin set must catch plausible mistakes in the oracle.

Every mutant below is a copy of the oracle's C source with one plausible
mistake planted by text substitution (on the CPU, in a temporary directory;
the oracle itself is untouched).  The test compiles the mutant and runs all
pins against it: at least one pin must fail, or the pins are too weak.
"""
import os
import shutil

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.dirname(os.path.abspath(oracle.__file__))

MUTANTS = {
    "f16_ties_away": ("if (rem > half || (rem == half && (q & 1)))", "if (rem >= half)"),
    "f16_truncate": ("if (rem > half || (rem == half && (q & 1)))", "if (0)"),
    "f16_subnormal_scale": ("v = ldexp((double)m, -24);", "v = ldexp((double)m, -25);"),
    "f16_no_subnormals": ("uint32_t enc = (e < -14) ? (uint32_t)q", "uint32_t enc = (e < -14) ? 0u"),
    "q8_0_unsigned_quants": ("float q = (float)(int8_t)b[2 + e];", "float q = (float)b[2 + e];"),
    "q4k_nibbles_swapped": ("int q = hi ? (qs[32 * p + i] >> 4) : (qs[32 * p + i] & 15);",
                            "int q = hi ? (qs[32 * p + i] & 15) : (qs[32 * p + i] >> 4);"),
    "q4k_wrong_subblock": ("q4k_scale_min(S, s, &sc, &m);", "q4k_scale_min(S, s ^ 1, &sc, &m);"),
    "q4k_high_scale_bits": ("*sc = (S[s + 4] & 15) | ((S[s - 4] >> 6) << 4);",
                            "*sc = (S[s + 4] & 15) | ((S[s] >> 6) << 4);"),
    "q4k_min_uses_d": ("float c = dmin * (float)m;", "float c = d * (float)m;"),
    "q4k_sign_flipped": ("y[e] = oracle_f32_to_f16(a - c);", "y[e] = oracle_f32_to_f16(c - a);"),
    "q4k_min_dropped": ("y[e] = oracle_f32_to_f16(a - c);", "y[e] = oracle_f32_to_f16(a);"),
    "q4k_group_stride": ("int p = e / 64;", "int p = e / 32 % 4;"),
    "q6k_ql_half_swapped": ("case 2:  lo = L[l] >> 4; ", "case 2:  lo = L[l + 32] >> 4; "),
    "q6k_qh_shift": ("case 1:  lo = L[l + 32] & 15;  hb = (H[l] >> 2) & 3;",
                     "case 1:  lo = L[l + 32] & 15;  hb = (H[l] >> 4) & 3;"),
    "q6k_scale_per_32": ("float s = (float)sc[e / 16];", "float s = (float)sc[e / 32];"),
    "q6k_offset": ("int q6 = (lo | (hb << 4)) - 32;", "int q6 = (lo | (hb << 4)) - 31;"),
    "q6k_unsigned_scale": ("const int8_t *sc = (const int8_t *)(b + 192);",
                           "const uint8_t *sc = (const uint8_t *)(b + 192);"),
    "q4_0_offset": ("y[e] = oracle_f32_to_f16(d * (float)(nib - 8));", "y[e] = oracle_f32_to_f16(d * (float)(nib - 7));"),
    "q4_0_nibble_halves": ("int nib = e < 16 ? (qs[e] & 15) : (qs[e - 16] >> 4);\n        y[e]",
                           "int nib = e < 16 ? (qs[e] >> 4) : (qs[e - 16] & 15);\n        y[e]"),
    "q5_qh_bit_order": ("return nib | (int)(((h >> e) & 1u) << 4);", "return nib | (int)(((h >> (e ^ 16)) & 1u) << 4);"),
    "q5_qh_big_endian": ("uint32_t h = (uint32_t)qh[0] | ((uint32_t)qh[1] << 8) | ((uint32_t)qh[2] << 16) | ((uint32_t)qh[3] << 24);",
                         "uint32_t h = (uint32_t)qh[3] | ((uint32_t)qh[2] << 8) | ((uint32_t)qh[1] << 16) | ((uint32_t)qh[0] << 24);"),
    "q5_0_offset": ("(q5_value(b + 2, b + 6, e) - 16)", "(q5_value(b + 2, b + 6, e) - 15)"),
    "q5_1_min_dropped": ("y[e] = oracle_f32_to_f16(dq + m);", "y[e] = oracle_f32_to_f16(dq);"),
    "q5_1_offset_kept": ("float dq = d * (float)q5_value(b + 4, b + 8, e);", "float dq = d * (float)(q5_value(b + 4, b + 8, e) - 16);"),
    "q5_1_min_scaled_by_d": ("y[e] = oracle_f32_to_f16(dq + m);", "y[e] = oracle_f32_to_f16(dq + d * m);"),
    "q5k_qh_bit": ("int q5 = nib | (((qh[pos] >> sub) & 1) << 4);", "int q5 = nib | (((qh[pos] >> grp) & 1) << 4);"),
    "q5k_qh_offset": ("const uint8_t *qh = b + 16;\n    const uint8_t *qs = b + 48;", "const uint8_t *qh = b + 48;\n    const uint8_t *qs = b + 16;"),
    "q5k_wrong_subblock": ("q4k_scale_min(S, sub, &scale, &mn);", "q4k_scale_min(S, grp, &scale, &mn);"),
    "q5k_min_dropped": ("y[e] = oracle_f32_to_f16(prod - off);", "y[e] = oracle_f32_to_f16(prod);"),
    "f32_big_endian": ("uint32_t x = (uint32_t)b[0] | ((uint32_t)b[1] << 8) | ((uint32_t)b[2] << 16) | ((uint32_t)b[3] << 24);",
                       "uint32_t x = (uint32_t)b[3] | ((uint32_t)b[2] << 8) | ((uint32_t)b[1] << 16) | ((uint32_t)b[0] << 24);"),
    "bf16_low_half": ("uint32_t x = (uint32_t)rd_u16le(b) << 16;", "uint32_t x = (uint32_t)rd_u16le(b);"),
    "bf16_read_as_f16": ("case T_BF16: y[0] = decode_bf16_elem(b); break;", "case T_BF16: y[0] = rd_u16le(b); break;"),
    "f16_bytes_swapped": ("case T_F16:  y[0] = rd_u16le(b); break;",
                          "case T_F16:  y[0] = (uint16_t)((b[0] << 8) | b[1]); break;"),
    "e4m3_ties_away": ("if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0))", "if (frac >= 0.5)"),
    "e4m3_no_clamp": ("if (e > 8 || (e == 8 && q > 14.0))", "if (e > 9)"),
    "e4m3_bias_8": ("return (uint8_t)(sign | (uint8_t)(((e + 7) << 3) | ((int)q - 8)));",
                    "return (uint8_t)(sign | (uint8_t)(((e + 8) << 3) | ((int)q - 8)));"),
    "e4m3_subnormal_unit": ("round_half_even(a * 512.0)", "round_half_even(a * 1024.0)"),
    "e4m3_quant_signed_amax": ("float v = fabsf(oracle_f16_to_f32(row[k]));", "float v = oracle_f16_to_f32(row[k]);"),
    "e4m3_quant_inv_from_scale": ("inv = 448.0f / amax;", "inv = 1.0f / s;"),
    "e4m3_gemm_drops_x_scale": ("* (double)sw[n] * (double)sx[m];", "* (double)sw[n];"),
    "gemm_reversed_operand": ("acc += x[k] * w[k];", "acc += x[k] * w[K - 1 - k];"),
    "gemm_f32_accumulator": ("double acc = 0.0;", "float acc = 0.0f;"),
    "gemm_drops_last_term": ("for (int64_t k = 0; k < K; k++)\n        acc += x[k] * w[k];",
                             "for (int64_t k = 0; k + 1 < K; k++)\n        acc += x[k] * w[k];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    for s in oracle.SOURCES:
        shutil.copy(os.path.join(SRC, s), tmp_path / s)
    src = (tmp_path / "oracle.c").read_text()
    assert src.count(old) == 1, f"mutation site not found exactly once: {old!r}"
    (tmp_path / "oracle.c").write_text(src.replace(old, new))
    lib = oracle.build(out=str(tmp_path / "libmutant.so"), src_dir=str(tmp_path))
    orc = oracle.Oracle(lib)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {name}"
